"""CPU oracle for one training step of a LoRA-adapted linear layer.

TEST INFRASTRUCTURE ONLY: this module is the plain, slow, obviously-correct definition that the
CUDA path is checked against. Only the tests, the package's smoke check and the benchmark's
CPU-baseline leg may import it; the product path never does.

Everything is numpy float64. Each function restates one step of the method as the pages define it:

  * "8. LoRA Fundamentals" (Juno), section "How it works":
      W_eff = W + s * B @ A, A is (rank x in), B is (out x rank), s = alpha/rank or alpha/sqrt(rank);
      canonical DoRA y = (magnitude / ||W + Delta||) * (W x + Delta x), row norm detached.
  * "4.3. Training Guide" (Juno), sections "Gradient accumulation", "Gradient clipping",
    "Optimizer", "Schedules", "Dropout".
  * "Backward Bug Hunts and Vulkan Tiled GEMM" (CatGame), sections "Bug #1" and "Bug #2":
    the LoRA gradients dA = B^T-side product and dB = out_prod of grad and the shrink activations.
  * "Multi-LoRA Training Example (fully-async)", section "Design (decoupled per-adapter
    optimizers)": per-slot accumulation with weight 1, 1/adapter_global_batch_size at step time,
    per-slot Adam state, step count and clipping; and the retirement of a finished adapter.
  * "4.3. Training Guide", section "Validation early stopping": snapshot and restore of the best
    A/B with an optimizer reset.

Where the pages leave a step open the oracle takes one reading and the CUDA path implements the
same reading independently (no shared code):
  * Adam constants beta1 = 0.9, beta2 = 0.999, eps = 1e-8 outside the square root; bias
    correction with k = completed updates + 1; decay uses the scheduled lr (not bias-corrected)
    and the pre-update value of A.
  * Moments see the clipped, normalised gradient c * g; "raw" means "without decay".
  * Clip iff max_norm > 0 and norm > max_norm (strict), scale max_norm / norm, no epsilon.
  * Non-finite: a non-finite double sum of squares rejects the step; nothing mutates.
  * Dropout mask: a stateless SplitMix64-finaliser hash, spelled out in `dropout_keep`.
  * The dropout scale q = 1/(1-p) is rounded to fp32 and folded into the LoRA scale.
  * DoRA magnitude gets Adam with the base lr (ratio 1) and no decay.

Parity pins live in tests/test_oracle_pins.py; every function here is pinned by at least one
check that does not re-run the function's own formula.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

STATUS_OK = 0
STATUS_NONFINITE = 6

KIND_A, KIND_B, KIND_MAG = 0, 1, 2

_U64 = np.uint64
_MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15


# ----------------------------------------------------------------------------------------------
# scaling and schedule  ("8. LoRA Fundamentals" / How it works; "4.3. Training Guide" / Schedules)
# ----------------------------------------------------------------------------------------------
def lora_scale(alpha: float, rank: int, rslora: bool) -> float:
    """s = alpha / rank (standard) or alpha / sqrt(rank) (rsLoRA), as an fp32 value."""
    s = alpha / math.sqrt(rank) if rslora else alpha / rank
    return float(np.float32(s))


def lr_at(kind: str, base: float, step: int, warmup: int, total: int, min_lr: float) -> float:
    """Scheduled learning rate at optimizer-update index `step` (counts updates, not chunks).

    constant: base.  cosine: linear warmup base*(step+1)/warmup for step < warmup, then
    min_lr + (base - min_lr) * (1 + cos(pi * progress)) / 2 with progress clamped to [0, 1]
    over the remaining total - warmup updates."""
    if kind == "constant":
        return float(base)
    if step < warmup:
        return float(base) * (step + 1) / warmup
    if total <= warmup:
        return float(min_lr)
    progress = min(1.0, (step - warmup) / (total - warmup))
    return float(min_lr) + 0.5 * (float(base) - float(min_lr)) * (1.0 + math.cos(math.pi * progress))


# ----------------------------------------------------------------------------------------------
# stateless dropout mask  ("4.3. Training Guide" / Dropout; "8. LoRA Fundamentals" / training loop)
# ----------------------------------------------------------------------------------------------
def mix64(z):
    """SplitMix64 output finaliser (Steele, Lea & Flood 2014; Stafford's mix variant 13):
    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31,
    all modulo 2^64. Works on Python ints and on uint64 numpy arrays."""
    if isinstance(z, (int, np.integer)):
        z = int(z) & _MASK64
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        return z ^ (z >> 31)
    z = np.asarray(z, dtype=_U64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> _U64(30))) * _U64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> _U64(27))) * _U64(0x94D049BB133111EB)
        z = z ^ (z >> _U64(31))
    return z


def dropout_key(seed: int, opt_step: int, accum_ordinal: int, layer: int, proj: int) -> int:
    """Per-(seed, optimizer step, accumulation ordinal, layer, projection) key, chained:
    k0 = mix(seed ^ golden), k1 = mix(k0 ^ step), k2 = mix(k1 ^ (ordinal<<48 | layer<<16 | proj))."""
    k = mix64((seed ^ GOLDEN_GAMMA) & _MASK64)
    k = mix64(k ^ (opt_step & _MASK64))
    packed = ((accum_ordinal & 0xFFFF) << 48) | ((layer & 0xFFFFFFFF) << 16) | (proj & 0xFFFF)
    return mix64(k ^ packed)


def dropout_threshold(p: float) -> int:
    """tau = floor(p * 2^32) in double, clamped to 2^32 - 1; an element is dropped iff the top
    32 bits of its hash are below tau, so P(drop) = tau / 2^32."""
    if p <= 0.0:
        return 0
    return min(int(math.floor(float(p) * 4294967296.0)), 0xFFFFFFFF)


def dropout_q(p: float) -> float:
    """Inverted-dropout scale 1 / (1 - p), rounded to fp32."""
    return float(np.float32(1.0 / (1.0 - float(p))))


def dropout_keep(p: float, seed: int, opt_step: int, accum_ordinal: int, layer: int, proj: int,
                 T: int, in_dim: int, chunk_tokens: int = 0) -> np.ndarray:
    """Keep mask M [T, in] (1.0 = kept) for the T tokens of one call.

    Token t of the call belongs to accumulation chunk accum_ordinal + t // chunk_tokens at
    position t % chunk_tokens (one chunk when chunk_tokens == 0). Element (t, i) hashes
    mix(key(chunk) ^ (position * in + i)). With p == 0 every element is kept."""
    if p <= 0.0:
        return np.ones((T, in_dim), dtype=np.float64)
    ct = T if chunk_tokens <= 0 else chunk_tokens
    tau = _U64(dropout_threshold(p))
    keep = np.empty((T, in_dim), dtype=bool)
    cols = np.arange(in_dim, dtype=_U64)
    for c0 in range(0, T, ct):
        ordinal = accum_ordinal + c0 // ct
        key = _U64(dropout_key(seed, opt_step, ordinal, layer, proj))
        n = min(ct, T - c0)
        pos = np.arange(n, dtype=_U64)[:, None]
        with np.errstate(over="ignore"):
            idx = pos * _U64(in_dim) + cols[None, :]
        h = mix64(key ^ idx)
        keep[c0:c0 + n] = (h >> _U64(32)) >= tau
    return keep.astype(np.float64)


# ----------------------------------------------------------------------------------------------
# forward / backward  ("8. LoRA Fundamentals" / How it works; "Backward Bug Hunts" / Bug #1, #2)
# ----------------------------------------------------------------------------------------------
def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().float().numpy()
    return np.asarray(a, dtype=np.float64)


def dora_row_norm(W, A, B, s: float) -> np.ndarray:
    """n_o = || W_o + s * (B @ A)_o ||_2, the detached DoRA row norm of the merged weight."""
    W, A, B = _f64(W), _f64(A), _f64(B)
    merged = W + s * (B @ A)
    return np.sqrt(np.sum(merged * merged, axis=1))


@dataclass
class Forward:
    Y: np.ndarray   # [T, out]
    H: np.ndarray   # [T, r] = Xd @ A^T  (unscaled shrink activations)
    Z: np.ndarray   # [T, out] pre-magnitude output (equals Y without DoRA)


def lora_forward(X, W, A, B, s: float, keep=None, q: float = 1.0, mag=None, rownorm=None) -> Forward:
    """Y = X W^T + s q (Xd A^T) B^T with Xd = M * X; DoRA: Y = (m / n) * (that)."""
    X, W, A, B = _f64(X), _f64(W), _f64(A), _f64(B)
    Xd = X if keep is None else keep * X
    H = Xd @ A.T
    Z = X @ W.T + (s * q) * (H @ B.T)
    if mag is None:
        return Forward(Z, H, Z)
    ratio = _f64(mag) / _f64(rownorm)
    return Forward(Z * ratio[None, :], H, Z)


@dataclass
class Backward:
    dX: np.ndarray   # [T, in]
    dA: np.ndarray   # [r, in]
    dB: np.ndarray   # [out, r]
    dm: Optional[np.ndarray]  # [out] (DoRA only)
    G: np.ndarray    # [T, r] = dY' @ B


def lora_backward(X, W, A, B, dY, s: float, keep=None, q: float = 1.0, mag=None,
                  rownorm=None) -> Backward:
    """Gradients of L = sum(Y * dY) for the forward above, with the DoRA row norm held fixed:
        dY' = dY (plain) or dY * (m / n) per output column (DoRA)
        G   = dY' B
        dX  = dY' W + s q (G A) * M
        dA  = s q G^T Xd
        dB  = s q dY'^T (Xd A^T)
        dm  = sum_t dY * Z / n   (DoRA)"""
    X, W, A, B, dY = _f64(X), _f64(W), _f64(A), _f64(B), _f64(dY)
    M = np.ones_like(X) if keep is None else keep
    Xd = M * X
    sq = s * q
    if mag is None:
        dYp = dY
    else:
        dYp = dY * (_f64(mag) / _f64(rownorm))[None, :]
    G = dYp @ B
    dX = dYp @ W + sq * (G @ A) * M
    dA = sq * (G.T @ Xd)
    H = Xd @ A.T
    dB = sq * (dYp.T @ H)
    dm = None
    if mag is not None:
        Z = X @ W.T + sq * (H @ B.T)
        dm = np.sum(dY * Z, axis=0) / _f64(rownorm)
    return Backward(dX, dA, dB, dm, G)


# ----------------------------------------------------------------------------------------------
# FP8 frozen base ("LoRA Training and Serving" / Quantized rollout: an FP8 base under a bf16-
# trained adapter; "Backward Bug Hunts" and "4.3. Training Guide" / Quick start: quantized frozen
# weights under the LoRA backward)
# ----------------------------------------------------------------------------------------------
# E4M3 (OCP 8-bit float): sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities, NaN =
# S.1111.111, largest finite 448 = 1.75 * 2^8, smallest normal 2^-6, subnormals m * 2^-9.
E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.power(2.0, e - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def e4m3_encode(x) -> np.ndarray:
    """float32 values -> uint8 codes: round to nearest, ties to even, finite values beyond the
    largest code saturate to +-448, NaN -> 0x7F with the sign bit of x.

    Element-wise on the value's binade: below 2^-6 the grid is the subnormal step 2^-9 (q = 8
    steps is 2^-6 itself, the smallest normal); in the binade [2^e, 2^(e+1)) it is 2^(e-3), the
    value is q steps with q in 8..16 (16 carries into the next binade), and the code is
    ((e + 7) << 3) | (q - 8)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.int64)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    sub = a < 2.0 ** -6
    q_sub = np.round(a / 2.0 ** -9)                     # numpy rounds half to even
    _, ex = np.frexp(np.where(sub, 1.0, a))             # a = f * 2^ex, f in [0.5, 1)
    e = ex.astype(np.int64) - 1                          # a in [2^e, 2^(e+1))
    q = np.round(np.where(sub, 0.0, a) / np.power(2.0, (e - 3).astype(np.float64)))
    carry = q >= 16
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8, q).astype(np.int64)
    code = np.where(sub, q_sub.astype(np.int64), ((e + 7) << 3) | (q - 8))
    code = np.where(a >= E4M3_MAX, 0x7E, np.minimum(code, 0x7E))
    code = np.where(nan, 0x7F, code)
    return (sign | code).astype(np.uint8)


def quantize_rows_e4m3(M):
    """Per-row scaled E4M3 codes of an fp32 (or bf16-valued) matrix, all arithmetic in fp32:
    with amax_r = max |M[r, :]|, the row is multiplied by r_r = 448 / amax_r and encoded
    (codes = e4m3(M[r, :] * r_r)), and s_r = amax_r / 448 is the scale that multiplies the
    decoded codes back; r_r = s_r = 1 when amax_r is 0 or 448 / amax_r is not finite.
    Returns (codes uint8 [R, K], scales float32 [R])."""
    M = np.asarray(M, dtype=np.float32)
    amax = np.max(np.abs(M), axis=1) if M.shape[1] else np.zeros(M.shape[0], np.float32)
    with np.errstate(divide="ignore", over="ignore"):
        rcp = (np.float32(E4M3_MAX) / amax).astype(np.float32)
    ok = (amax > 0) & np.isfinite(rcp)
    rcp = np.where(ok, rcp, np.float32(1.0)).astype(np.float32)
    sc = np.where(ok, (amax / np.float32(E4M3_MAX)).astype(np.float32), np.float32(1.0))
    q = (M * rcp[:, None]).astype(np.float32)
    return e4m3_encode(q), sc.astype(np.float32)


def fp8_product(Xc, sx, Wc, sw) -> np.ndarray:
    """diag(sx) (dec(Xc) dec(Wc)^T) diag(sw): the frozen product on E4M3 operands with per-row
    scales of X's rows and W's rows (the contraction runs over the columns of both)."""
    return (_f64(sx)[:, None] * (e4m3_decode(Xc) @ e4m3_decode(Wc).T)) * _f64(sw)[None, :]


def lora_forward_fp8(X, W, A, B, s: float, keep=None, q: float = 1.0) -> Forward:
    """Y = fp8 frozen product of (X, W) + s q (Xd A^T) B^T: the frozen term runs on the per-row
    E4M3 quantisations of X (per token) and W (per output row); the adapter branch reads the
    bf16 X unchanged."""
    Xc, sx = quantize_rows_e4m3(X)
    Wc, sw = quantize_rows_e4m3(W)
    X64, A, B = _f64(X), _f64(A), _f64(B)
    Xd = X64 if keep is None else keep * X64
    H = Xd @ A.T
    Y = fp8_product(Xc, sx, Wc, sw) + (s * q) * (H @ B.T)
    return Forward(Y, H, Y)


def lora_dx_fp8(dY, W, A, G, s: float, keep=None, q: float = 1.0) -> np.ndarray:
    """dX = fp8 product of (dY, W^T) + s q (G A) * M: the frozen term runs on the per-token
    E4M3 quantisation of dY and the per-row quantisation of W^T (one scale per input column
    of W); G = dY B is taken in full precision as in lora_backward."""
    Dc, sd = quantize_rows_e4m3(dY)
    Wtc, swt = quantize_rows_e4m3(np.asarray(W, np.float32).T)
    M = 1.0 if keep is None else keep
    return fp8_product(Dc, sd, Wtc, swt) + (s * q) * (_f64(G) @ _f64(A)) * M


# ----------------------------------------------------------------------------------------------
# grad prepare and optimizer  ("4.3. Training Guide" / Gradient clipping, Optimizer)
# ----------------------------------------------------------------------------------------------
@dataclass
class Prepared:
    status: int
    scale: float     # combined normalise x clip factor c applied to every gradient element
    norm: float      # L2 norm of the normalised gradient (gamma * ||g||), before clipping


def grad_prepare(grads: Sequence, grad_scale: float, max_norm: float) -> Prepared:
    """Pass 1: S = sum of g^2 over every element of every gradient tensor, in double; a
    non-finite S rejects the step. Pass 2's single factor: gamma = grad_scale (1 / prediction
    tokens, or 1 / adapter_global_batch_size per slot); norm = gamma * sqrt(S);
    c = gamma * max_norm / norm if max_norm > 0 and norm > max_norm, else gamma."""
    S = 0.0
    for g in grads:
        g = _f64(g).ravel()
        S += float(np.dot(g, g))
    if not math.isfinite(S):
        return Prepared(STATUS_NONFINITE, float("nan"), float("nan"))
    gamma = float(grad_scale)
    norm = math.sqrt(S) * gamma
    c = gamma * (max_norm / norm) if (max_norm > 0.0 and norm > max_norm) else gamma
    return Prepared(STATUS_OK, c, norm)


@dataclass
class AdamHP:
    lr: float
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    wd: float = 0.01
    plus_ratio: float = 1.0
    step: int = 0       # completed updates before this one


def adamw_update(p, g, m, v, kind: int, c: float, hp: AdamHP):
    """One decoupled AdamW update of one tensor, given the prepared factor c.

    g_hat = c g; m = b1 m + (1-b1) g_hat; v = b2 v + (1-b2) g_hat^2; k = step + 1;
    u = (m / (1 - b1^k)) / (sqrt(v / (1 - b2^k)) + eps).
    A:   p - lr u - lr wd p_pre   (decay on A only, from the pre-update value, scheduled lr)
    B:   p - lr rho u             (LoRA+ ratio rho, never decayed)
    MAG: p - lr u                 (DoRA magnitude: ratio 1, no decay)
    Returns fp32 (p, m, v)."""
    p, g, m, v = _f64(p), _f64(g), _f64(m), _f64(v)
    k = hp.step + 1
    gh = c * g
    m1 = hp.beta1 * m + (1.0 - hp.beta1) * gh
    v1 = hp.beta2 * v + (1.0 - hp.beta2) * gh * gh
    u = (m1 / (1.0 - hp.beta1 ** k)) / (np.sqrt(v1 / (1.0 - hp.beta2 ** k)) + hp.eps)
    if kind == KIND_A:
        p1 = p - hp.lr * u - hp.lr * hp.wd * p
    elif kind == KIND_B:
        p1 = p - hp.lr * hp.plus_ratio * u
    elif kind == KIND_MAG:
        p1 = p - hp.lr * u
    else:
        raise ValueError(kind)
    return p1.astype(np.float32), m1.astype(np.float32), v1.astype(np.float32)


# ----------------------------------------------------------------------------------------------
# adapter-state maintenance  ("4.3. Training Guide" / Validation early stopping: the best A/B
# are snapshotted and restored, and the optimizer is reset after the restore; "Multi-LoRA
# Training Example (fully-async)": a finished adapter is retired, its slot cleared, its optimizer
# state and retained gradients zeroed and its partial accumulation discarded)
# ----------------------------------------------------------------------------------------------
def group_ranges(groups: Sequence[Tuple[int, int]]):
    """(offset, count) pairs -> the flat index ranges they cover."""
    return [range(off, off + cnt) for off, cnt in groups]


def snapshot(params, snap, groups: Sequence[Tuple[int, int]]) -> np.ndarray:
    """Returns snap with snap[i] = params[i] for every index i in a group; other entries kept."""
    out = np.array(snap, dtype=np.float32, copy=True)
    for r in group_ranges(groups):
        for i in r:
            out[i] = params[i]
    return out


def restore(params, snap, grads, m, v, groups: Sequence[Tuple[int, int]], zero_grads: bool):
    """Returns (params, grads, m, v) with, inside the groups: params = snap, m = v = 0 (the
    optimizer reset; the caller also restarts the update count) and grads = 0 when zero_grads.
    Entries outside the groups are kept."""
    p, g, mm, vv = (np.array(a, dtype=np.float32, copy=True) for a in (params, grads, m, v))
    for r in group_ranges(groups):
        for i in r:
            p[i] = snap[i]
            mm[i] = 0.0
            vv[i] = 0.0
            if zero_grads:
                g[i] = 0.0
    return p, g, mm, vv


def retire(params, grads, m, v, groups: Sequence[Tuple[int, int]], clear_params: bool):
    """Returns (params, grads, m, v) with, inside the groups: grads = m = v = 0 and params = 0
    when clear_params. Entries outside the groups are kept."""
    p, g, mm, vv = (np.array(a, dtype=np.float32, copy=True) for a in (params, grads, m, v))
    for r in group_ranges(groups):
        for i in r:
            g[i] = 0.0
            mm[i] = 0.0
            vv[i] = 0.0
            if clear_params:
                p[i] = 0.0
    return p, g, mm, vv


# ----------------------------------------------------------------------------------------------
# slot-keyed multi-LoRA  ("Multi-LoRA Training Example (fully-async)" / Design)
# ----------------------------------------------------------------------------------------------
def token_slots(T: int, seg_start: Sequence[int], seg_slot: Sequence[int], n_slots: int) -> np.ndarray:
    """Slot of every token: segment k covers tokens [seg_start[k], seg_start[k+1]); tokens in no
    segment, and segments whose slot id is outside [0, n_slots), get -1 (no adapter)."""
    out = np.full(T, -1, dtype=np.int32)
    for k in range(len(seg_slot)):
        a, b = int(seg_start[k]), int(seg_start[k + 1])
        a, b = max(0, min(a, T)), max(0, min(b, T))
        sl = int(seg_slot[k])
        if 0 <= sl < n_slots and b > a:
            out[a:b] = sl
    return out


@dataclass
class SlotTensors:
    A: object
    B: object
    s: float


def multi_lora_forward(X, W, slots: Sequence[SlotTensors], tok_slot: np.ndarray, keep=None,
                       q: float = 1.0) -> Tuple[np.ndarray, np.ndarray]:
    """Per token t with slot k: Y_t = X_t W^T + s_k q (Xd_t A_k^T) B_k^T; tokens with no slot get
    the frozen output only. Returns (Y, H) with H [T, max_rank] holding Xd_t A_k^T in the slot's
    first r_k columns and zeros elsewhere."""
    X, W = _f64(X), _f64(W)
    T = X.shape[0]
    M = np.ones_like(X) if keep is None else keep
    rmax = max(_f64(sl.A).shape[0] for sl in slots)
    Y = X @ W.T
    H = np.zeros((T, rmax))
    for t in range(T):
        k = int(tok_slot[t])
        if k < 0:
            continue
        A, B = _f64(slots[k].A), _f64(slots[k].B)
        h = A @ (M[t] * X[t])
        H[t, :A.shape[0]] = h
        Y[t] += slots[k].s * q * (B @ h)
    return Y, H


def multi_lora_backward(X, W, dY, slots: Sequence[SlotTensors], tok_slot: np.ndarray, keep=None,
                        q: float = 1.0):
    """Per-slot gradients summed over that slot's tokens (weight 1 per token), plus dX:
    dX_t = dY_t W + s_k q ((dY_t B_k) A_k) * M_t; dA_k = sum_t s_k q (dY_t B_k)^T (Xd_t);
    dB_k = sum_t s_k q dY_t^T (A_k Xd_t)."""
    X, W, dY = _f64(X), _f64(W), _f64(dY)
    M = np.ones_like(X) if keep is None else keep
    dX = dY @ W
    dA = [np.zeros_like(_f64(sl.A)) for sl in slots]
    dB = [np.zeros_like(_f64(sl.B)) for sl in slots]
    for t in range(X.shape[0]):
        k = int(tok_slot[t])
        if k < 0:
            continue
        A, B, sq = _f64(slots[k].A), _f64(slots[k].B), slots[k].s * q
        xd = M[t] * X[t]
        g = dY[t] @ B
        dX[t] += sq * (g @ A) * M[t]
        dA[k] += sq * np.outer(g, xd)
        dB[k] += sq * np.outer(dY[t], A @ xd)
    return dX, dA, dB


def multi_lora_backward_vectorised(X, W, dY, slots: Sequence[SlotTensors], tok_slot: np.ndarray,
                                   keep=None, q: float = 1.0):
    """Same definition as multi_lora_backward, evaluated slot by slot with matrix products over the
    slot's token rows (for full-size cases where the per-token loop is too slow)."""
    X, W, dY = _f64(X), _f64(W), _f64(dY)
    M = np.ones_like(X) if keep is None else keep
    dX = dY @ W
    dA, dB = [], []
    for k, sl in enumerate(slots):
        rows = np.nonzero(tok_slot == k)[0]
        A, B, sq = _f64(sl.A), _f64(sl.B), sl.s * q
        Xd = M[rows] * X[rows]
        G = dY[rows] @ B
        dX[rows] += sq * (G @ A) * M[rows]
        dA.append(sq * (G.T @ Xd))
        dB.append(sq * (dY[rows].T @ (Xd @ A.T)))
    return dX, dA, dB


# ----------------------------------------------------------------------------------------------
# one optimizer step over accumulation chunks  ("4.3. Training Guide" / Gradient accumulation;
# "8. LoRA Fundamentals" / The training loop, Microbatching)
# ----------------------------------------------------------------------------------------------
@dataclass
class AdapterState:
    A: np.ndarray
    B: np.ndarray
    mA: np.ndarray
    vA: np.ndarray
    mB: np.ndarray
    vB: np.ndarray
    mag: Optional[np.ndarray] = None
    mM: Optional[np.ndarray] = None
    vM: Optional[np.ndarray] = None


@dataclass
class StepResult:
    prepared: Prepared
    grads: Dict[object, Tuple[np.ndarray, np.ndarray, Optional[np.ndarray]]]   # fp32 sums
    new_state: Dict[object, AdapterState]
    outputs: Dict[object, List[Tuple[np.ndarray, np.ndarray, np.ndarray]]]     # per chunk Y, dX, H


def run_single_step(problems: Dict[object, dict], state: Dict[object, AdapterState], *, s: float,
                    chunks: int, p: float, seed: int, opt_step: int, max_norm: float, hp: AdamHP,
                    dora: bool = False, keep_outputs: bool = True) -> StepResult:
    """One optimizer step for a set of independent adapted linears.

    problems[key] = {X [T,in], W [out,in], dY [T,out], layer, proj}. Every problem's T tokens are
    split into `chunks` equal accumulation chunks processed in order; raw gradient sums accumulate
    in fp32 buffers; then grad_prepare with gamma = 1 / (total prediction tokens) over every
    adapter gradient (global clip) and, if the status is OK, one AdamW update of every tensor.
    DoRA row norms are refreshed once at the start of the step from the current A and B."""
    q = dropout_q(p) if p > 0 else 1.0
    grads, outputs = {}, {}
    n_pred = 0
    for key, pr in problems.items():
        st = state[key]
        X, W, dY = _f64(pr["X"]), _f64(pr["W"]), _f64(pr["dY"])
        T = X.shape[0]
        ct = T // chunks
        gA = np.zeros(st.A.shape, np.float32)
        gB = np.zeros(st.B.shape, np.float32)
        gM = np.zeros(st.mag.shape, np.float32) if dora else None
        rown = dora_row_norm(W, st.A, st.B, s) if dora else None
        outs = []
        for c in range(chunks):
            rows = slice(c * ct, (c + 1) * ct)
            keep = dropout_keep(p, seed, opt_step, c, pr["layer"], pr["proj"], ct, X.shape[1]) \
                if p > 0 else None
            mag = st.mag if dora else None
            f = lora_forward(X[rows], W, st.A, st.B, s, keep, q, mag, rown)
            b = lora_backward(X[rows], W, st.A, st.B, dY[rows], s, keep, q, mag, rown)
            gA = (gA.astype(np.float64) + b.dA).astype(np.float32)
            gB = (gB.astype(np.float64) + b.dB).astype(np.float32)
            if dora:
                gM = (gM.astype(np.float64) + b.dm).astype(np.float32)
            if keep_outputs:
                outs.append((f.Y, b.dX, f.H))
        grads[key] = (gA, gB, gM)
        outputs[key] = outs
    n_pred = next(iter(problems.values()))["X"].shape[0]
    flat = []
    for key in problems:
        gA, gB, gM = grads[key]
        flat += [gA, gB] + ([gM] if dora else [])
    prep = grad_prepare(flat, 1.0 / n_pred, max_norm)
    new_state = {}
    for key in problems:
        st = state[key]
        if prep.status != STATUS_OK:
            new_state[key] = st
            continue
        gA, gB, gM = grads[key]
        A1, mA1, vA1 = adamw_update(st.A, gA, st.mA, st.vA, KIND_A, prep.scale, hp)
        B1, mB1, vB1 = adamw_update(st.B, gB, st.mB, st.vB, KIND_B, prep.scale, hp)
        ns = AdapterState(A1, B1, mA1, vA1, mB1, vB1)
        if dora:
            ns.mag, ns.mM, ns.vM = adamw_update(st.mag, gM, st.mM, st.vM, KIND_MAG, prep.scale, hp)
        new_state[key] = ns
    return StepResult(prep, grads, new_state, outputs)


@dataclass
class FusedResult:
    Y: np.ndarray                      # [T, sum out_p]
    H: np.ndarray                      # [T, P * r] unscaled shrinks, projection p in columns p*r..
    dX: np.ndarray                     # [T, in] summed over the projections
    grads: List[Tuple[np.ndarray, np.ndarray]]   # per projection (dA_p, dB_p)


def fused_forward_backward(X, Ws: Sequence, As: Sequence, Bs: Sequence, dYs: Sequence, s: float,
                           keep=None, q: float = 1.0) -> FusedResult:
    """Projections that share one input, run as one fused linear ("LoRA Training and Serving",
    --lora-type: `lora` fuses the projections, `canonical_lora` keeps one adapter per projection;
    here one fused frozen weight W_cat = [W_0; W_1; ...] with one adapter per projection). The
    output is the projections' outputs side by side, and the input gradient is their sum:
        Y_cat = [Y_0 | Y_1 | ...],  Y_p = X W_p^T + s q (Xd A_p^T) B_p^T
        dX    = sum_p (dY_p W_p + s q (G_p A_p) * M),  G_p = dY_p B_p
    with one dropout mask M shared by the projections (they read the same input)."""
    ys, hs, grads = [], [], []
    dX = None
    for W, A, B, dY in zip(Ws, As, Bs, dYs):
        f = lora_forward(X, W, A, B, s, keep, q)
        b = lora_backward(X, W, A, B, dY, s, keep, q)
        ys.append(f.Y)
        hs.append(f.H)
        grads.append((b.dA, b.dB))
        dX = b.dX if dX is None else dX + b.dX
    return FusedResult(np.concatenate(ys, axis=1), np.concatenate(hs, axis=1), dX, grads)


@dataclass
class ChainResult:
    Y: np.ndarray                      # [T, d_L] output of the last layer
    dX: np.ndarray                     # [T, d_0] gradient of the first layer's input
    grads: List[Tuple[np.ndarray, np.ndarray]]   # per layer fp32 sums (dA, dB)


def chained_forward_backward(X0, Ws: Sequence, As: Sequence, Bs: Sequence, dY_top, s: float,
                             chunks: int, *, round_act=None, p: float = 0.0, seed: int = 0,
                             opt_step: int = 0, layer_ids: Optional[Sequence[int]] = None,
                             proj: int = 0) -> ChainResult:
    """A stack of adapted linears in which layer l's output is layer l + 1's input ("4.3.
    Training Guide", Truncated BPTT: the backward window is one chunk of tokens, and Gradient
    accumulation: raw sums over the chunks in order). Per chunk: the forward runs through every
    layer, then the backward runs through them in reverse, layer l's output gradient being layer
    l + 1's input gradient. Activations handed from one layer to the next pass through round_act
    (the activation dtype: identity for fp32, round to bf16 for bf16 activations), as they do
    when stored between layers. Gradient sums accumulate in fp32 as in run_single_step."""
    rnd = round_act if round_act is not None else (lambda a: a)
    X0, dY_top = _f64(X0), _f64(dY_top)
    T = X0.shape[0]
    ct = T // chunks
    nl = len(Ws)
    ids = list(layer_ids) if layer_ids is not None else list(range(nl))
    q = dropout_q(p) if p > 0 else 1.0
    grads = [(np.zeros(np.shape(As[l]), np.float32), np.zeros(np.shape(Bs[l]), np.float32))
             for l in range(nl)]
    Y_out = np.zeros((T, np.shape(Ws[-1])[0]))
    dX_in = np.zeros((T, np.shape(Ws[0])[1]))
    for c in range(chunks):
        rows = slice(c * ct, (c + 1) * ct)
        xs, keeps = [], []
        x = X0[rows]
        for l in range(nl):
            keep = dropout_keep(p, seed, opt_step, c, ids[l], proj, ct, np.shape(Ws[l])[1]) \
                if p > 0 else None
            xs.append(x)
            keeps.append(keep)
            x = rnd(lora_forward(x, Ws[l], As[l], Bs[l], s, keep, q).Y)
        Y_out[rows] = x
        g = dY_top[rows]
        for l in reversed(range(nl)):
            b = lora_backward(xs[l], Ws[l], As[l], Bs[l], g, s, keeps[l], q)
            gA, gB = grads[l]
            grads[l] = ((gA.astype(np.float64) + b.dA).astype(np.float32),
                        (gB.astype(np.float64) + b.dB).astype(np.float32))
            g = rnd(b.dX)
        dX_in[rows] = g
    return ChainResult(Y_out, dX_in, grads)


def lora_adapter_grads(X, A, B, dY, s: float, keep=None, q: float = 1.0):
    """dA and dB alone (no frozen product needed): dA = s q (dY B)^T Xd, dB = s q dY^T (Xd A^T).
    Same definitions as lora_backward, for cases where the frozen products are too large."""
    X, A, B, dY = _f64(X), _f64(A), _f64(B), _f64(dY)
    Xd = X if keep is None else keep * X
    G = dY @ B
    return (s * q) * (G.T @ Xd), (s * q) * (dY.T @ (Xd @ A.T))
