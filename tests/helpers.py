"""Shared helpers for the tests: seeded problems fed identically to the CUDA path and the oracle,
and the per-tensor error metric (max |x - r| / max |r|)."""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

import lora_inputs as LI
from oracle import lora_oracle as O

TOL_F32 = 1e-5          # fp32 frozen-W paths: every output and the post-step state
TOL_BF16 = 2e-2         # bf16 frozen-W paths: Y, dX, dA, dB
TOL_BF16_STEP = 1e-2    # bf16 frozen-W paths: post-step A / B


def rel_err(x, ref) -> float:
    x = np.asarray(x.detach().cpu().double().numpy() if hasattr(x, "detach") else x, np.float64)
    ref = np.asarray(ref.detach().cpu().double().numpy() if hasattr(ref, "detach") else ref,
                     np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(x - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den


def to64(t) -> np.ndarray:
    if hasattr(t, "detach"):
        return t.detach().cpu().double().numpy()
    return np.asarray(t, np.float64)


def lr_for(cfg: LI.LoraConfig) -> float:
    return O.lr_at(cfg.sched, cfg.lr, cfg.opt_step, cfg.warmup, cfg.total, cfg.min_lr)


def build_single(cfg: LI.LoraConfig, layers: Sequence[int], proj_idx: Sequence[int],
                 tokens: Optional[int] = None, device="cuda", n_streams: int = 1,
                 overrides: Optional[dict] = None):
    """CUDA LoraStep and the oracle's problems/state from the same seeded inputs."""
    from bwd_adapter_adamw_gb300 import binding as L
    from bwd_adapter_adamw_gb300.step import Linear, LoraStep
    T = cfg.tokens if tokens is None else tokens
    linears, problems, state, init = [], {}, {}, {}
    for l in layers:
        for pi in proj_idx:
            pr = cfg.projs[pi]
            X = LI.make_x(cfg, l, pr, tokens=T)
            W = LI.make_w(cfg, l, pr)
            dY = LI.make_dy(cfg, l, pr, tokens=T)
            A = LI.make_a(cfg, l, pr)
            B = LI.make_b(cfg, l, pr)
            linears.append(Linear(l, pi, X.to(device), W.to(device), dY.to(device)))
            problems[(l, pi)] = dict(X=X, W=W, dY=dY, layer=l, proj=pi)
            init[(l, pi)] = (A, B, W)
    s = O.lora_scale(cfg.alpha, cfg.rank, cfg.rslora)
    hp = L.make_hp(cfg.beta1, cfg.beta2, cfg.eps, cfg.wd, cfg.plus_ratio)
    step = LoraStep(linears, rank=cfg.rank, scale=s, dtype=cfg.dtype, tokens=T, chunks=cfg.chunks,
                    dropout_p=cfg.dropout_p, seed=cfg.dropout_seed, dora=cfg.dora,
                    max_norm=cfg.max_norm, hp=hp, n_streams=n_streams, device=device)
    mA, vA = LI.make_adam_state(cfg, step.n_a, "A")
    mB, vB = LI.make_adam_state(cfg, step.n_b, "B")
    na, nb = step.n_a, step.n_b
    step.arena.m[:na].copy_(mA)
    step.arena.v[:na].copy_(vA)
    step.arena.m[na:na + nb].copy_(mB)
    step.arena.v[na:na + nb].copy_(vB)
    oa, ob = 0, 0
    for lin in step.linears:
        A, B, W = init[(lin.layer, lin.proj_id)]
        lin.A.copy_(A)
        lin.B.copy_(B)
        st = O.AdapterState(A.numpy().copy(), B.numpy().copy(),
                            mA[oa:oa + A.numel()].numpy().reshape(A.shape).copy(),
                            vA[oa:oa + A.numel()].numpy().reshape(A.shape).copy(),
                            mB[ob:ob + B.numel()].numpy().reshape(B.shape).copy(),
                            vB[ob:ob + B.numel()].numpy().reshape(B.shape).copy())
        oa += A.numel()
        ob += B.numel()
        if cfg.dora:
            mag = LI.dora_magnitude_init(W)
            lin.mag.copy_(mag)
            st.mag = mag.numpy().copy()
            st.mM = np.zeros_like(st.mag)
            st.vM = np.zeros_like(st.mag)
        state[(lin.layer, lin.proj_id)] = st
    step.prepare_weights()
    torch.cuda.synchronize()
    hp_o = O.AdamHP(lr=lr_for(cfg), beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps, wd=cfg.wd,
                    plus_ratio=cfg.plus_ratio, step=cfg.opt_step)
    return step, problems, state, s, hp_o


U32 = 2.0 ** -24   # fp32 unit roundoff: the GPU accumulates every sum in fp32


def grad_bounds(pr: dict, A, B, s: float, keep, q: float):
    """Forward-error bounds of one chunk's fp32 gradient sums: |computed - exact| <= n u sum|terms|
    (the standard summation bound), with n the length of the chained sums: H = Xd A^T (in terms)
    feeding dB (T terms), G = dY B (out terms) feeding dA (T terms)."""
    X, dY = to64(pr["X"]), to64(pr["dY"])
    A, B = np.abs(np.asarray(A, np.float64)), np.abs(np.asarray(B, np.float64))
    Xd = np.abs(X if keep is None else keep * X)
    T, n_in, n_out = X.shape[0], X.shape[1], dY.shape[1]
    H_abs = Xd @ A.T
    G_abs = np.abs(dY) @ B
    dB = (T + n_in) * U32 * abs(s * q) * (np.abs(dY).T @ H_abs)
    dA = (T + n_out) * U32 * abs(s * q) * (G_abs.T @ Xd)
    return dA, dB


def check_post_step(x_gpu, p0, m0, v0, g_ref, g_bound, kind: int, c: float, hp, tol: float,
                    max_clause_frac: float = 1e-3, exclude=None):
    """Post-step parameter check. An element passes plainly when |x - r| <= tol * max|r|; near
    g_hat ~ 0 the Adam map u = m_hat / (sqrt(v_hat) + eps) has slope up to 1/eps, so an fp32
    difference in the gradient within its error bound moves the update by far more than tol.
    Such an element passes if x lies in the band of oracle results for gradients in
    [g - bound, g + bound] (widened by tol * max|r|). Returns the number of elements that needed
    the band, which must stay below max_clause_frac of the tensor."""
    x = to64(x_gpu) if hasattr(x_gpu, "detach") else np.asarray(x_gpu, np.float64)
    g = np.asarray(g_ref, np.float64)
    m0 = np.asarray(m0, np.float64)
    bound = np.asarray(g_bound, np.float64) + 1e-6 * np.abs(g)
    r = O.adamw_update(p0, g, m0, v0, kind, c, hp)[0].astype(np.float64)
    # corners: the gradient within its bound, and the first moment within the fp32 rounding of
    # m = b1 m0 + (1 - b1) c g (which can cancel to ~0, where u = m_hat / sqrt(v_hat) is steep)
    dm = 4 * U32 * (np.abs(m0) + (1 - hp.beta1) / hp.beta1 * np.abs(c * g))
    # u(g) is not monotonic (it saturates towards a constant for large |g_hat|), so the interval is
    # sampled densely, linearly and log-spaced around g, rather than at its ends only
    ts = np.concatenate([np.linspace(-1.0, 1.0, 41), np.logspace(-9, 0, 28), -np.logspace(-9, 0, 28)])
    lo, hi = r.copy(), r.copy()
    for t in ts:
        gg = g + t * bound
        for mm in (m0 - dm, m0, m0 + dm):
            y = O.adamw_update(p0, gg, mm, v0, kind, c, hp)[0].astype(np.float64)
            lo, hi = np.minimum(lo, y), np.maximum(hi, y)
    slack = tol * max(float(np.max(np.abs(r))), 1e-30)
    plain = np.abs(x - r) <= slack
    band = (x >= lo - slack) & (x <= hi + slack)
    ok = plain | band
    if exclude is not None:
        # elements whose previous update already needed the band carry that (bounded) difference
        # in their state; they are left out here and counted by the caller
        ok = ok | exclude
        plain = plain | exclude
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[np.argmax(np.abs((x - r)[~ok]))])
        detail = dict(index=i, x=x[i], r=r[i], lo=lo[i], hi=hi[i], g=g[i], bound=bound[i],
                      m0=m0[i], v0=np.asarray(v0, np.float64)[i], p0=np.asarray(p0, np.float64)[i],
                      c=c, slack=slack)
        raise AssertionError((int((~ok).sum()), float(np.max(np.abs(x - r))) / max(slack / tol, 1e-30),
                              detail))
    n_clause = int((~plain).sum())
    assert n_clause <= max(2, int(max_clause_frac * x.size)), n_clause
    return n_clause, ~(np.abs(x - r) <= slack)
