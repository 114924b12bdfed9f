"""Pins for the CPU oracle: each check ties the oracle to something other than its own formula
(hand-worked values, published test vectors, closed forms, exact identities, finite differences,
brute force), so that a dropped term, a wrong sign, index or transposed operand fails one of them.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import lora_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed=0):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------------------------------ hash
def test_mix64_matches_published_splitmix64_outputs():
    g = _golden("splitmix64_seed0.json")
    state = 0
    for want in g["outputs_hex"]:
        state = (state + O.GOLDEN_GAMMA) & ((1 << 64) - 1)
        assert O.mix64(state) == int(want, 16)


def _inv_xorshift(y, sh):
    x = y
    for _ in range(64 // sh + 1):
        x = y ^ (x >> sh)
    return x


def test_mix64_is_a_bijection_via_its_algebraic_inverse():
    M = (1 << 64) - 1
    i1 = pow(0xBF58476D1CE4E5B9, -1, 1 << 64)
    i2 = pow(0x94D049BB133111EB, -1, 1 << 64)
    rng = _rng(1)
    for z in [0, 1, M] + [int(v) for v in rng.integers(0, 2**63, 200, dtype=np.int64)]:
        y = O.mix64(z)
        x = _inv_xorshift(y, 31)
        x = (x * i2) & M
        x = _inv_xorshift(x, 27)
        x = (x * i1) & M
        x = _inv_xorshift(x, 30)
        assert x == z


def test_mix64_array_and_scalar_forms_agree():
    zs = _rng(2).integers(0, 2**63, 64, dtype=np.int64).astype(np.uint64)
    arr = O.mix64(zs)
    assert [int(v) for v in arr] == [O.mix64(int(z)) for z in zs]


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_dropout_rate_within_binomial_bounds(p):
    keep = O.dropout_keep(p, 1234, 25, 0, 3, 2, 512, 768)
    n = keep.size
    dropped = n - keep.sum()
    sigma = math.sqrt(n * p * (1 - p))
    assert abs(dropped - n * p) < 6 * sigma


def test_dropout_threshold_edges():
    assert O.dropout_threshold(0.0) == 0
    assert O.dropout_threshold(0.5) == 1 << 31
    assert O.dropout_threshold(0.25) == 1 << 30
    assert np.all(O.dropout_keep(0.0, 1, 2, 3, 4, 5, 7, 9) == 1.0)
    assert O.dropout_q(0.5) == 2.0
    assert O.dropout_q(0.1) == float(np.float32(1 / 0.9))


def test_dropout_is_deterministic_and_every_key_field_matters():
    base = dict(p=0.3, seed=42, opt_step=7, accum_ordinal=1, layer=5, proj=3, T=16, in_dim=64)
    m0 = O.dropout_keep(**base)
    assert np.array_equal(m0, O.dropout_keep(**base))
    for field, val in [("seed", 43), ("opt_step", 8), ("accum_ordinal", 2), ("layer", 6),
                       ("proj", 4)]:
        other = dict(base, **{field: val})
        assert not np.array_equal(m0, O.dropout_keep(**other)), field


def test_dropout_chunked_call_equals_per_chunk_calls():
    a = O.dropout_keep(0.2, 9, 3, 4, 1, 1, 24, 40, chunk_tokens=8)
    parts = [O.dropout_keep(0.2, 9, 3, 4 + c, 1, 1, 8, 40) for c in range(3)]
    assert np.array_equal(a, np.concatenate(parts))


def test_dropout_hash_brute_force_single_element():
    # element (t, i) of chunk `ordinal`: mix(key ^ (t*in + i)), dropped iff top 32 bits < tau
    p, seed, step, ordinal, layer, proj, in_dim = 0.37, 77, 11, 3, 9, 4, 13
    key = O.mix64(O.mix64(O.mix64(seed ^ O.GOLDEN_GAMMA) ^ step) ^ ((ordinal << 48) | (layer << 16) | proj))
    keep = O.dropout_keep(p, seed, step, ordinal, layer, proj, 5, in_dim)
    tau = int(p * 2**32)
    for t in range(5):
        for i in range(in_dim):
            h = O.mix64(key ^ (t * in_dim + i))
            assert keep[t, i] == (1.0 if (h >> 32) >= tau else 0.0)


# ---------------------------------------------------------------------------------- forward/back
def test_hand_worked_forward_backward():
    g = _golden("hand_worked.json")["lora_1x2"]
    s = O.lora_scale(g["alpha"], g["rank"], False)
    f = O.lora_forward(g["X"], g["W"], g["A"], g["B"], s)
    b = O.lora_backward(g["X"], g["W"], g["A"], g["B"], g["dY"], s)
    np.testing.assert_array_equal(f.Y, g["Y"])
    np.testing.assert_array_equal(b.dX, g["dX"])
    np.testing.assert_array_equal(b.dA, g["dA"])
    np.testing.assert_array_equal(b.dB, g["dB"])


def test_scaling_standard_and_rslora():
    assert O.lora_scale(16, 8, False) == 2.0
    assert O.lora_scale(128, 64, True) == 16.0
    assert O.lora_scale(8, 4, False) == 2.0


def _problem(T=6, n_in=5, n_out=4, r=3, seed=3):
    rng = _rng(seed)
    return (rng.standard_normal((T, n_in)), rng.standard_normal((n_out, n_in)) / 2,
            rng.standard_normal((r, n_in)), rng.standard_normal((n_out, r)),
            rng.standard_normal((T, n_out)))


def test_zero_adapter_is_a_noop_and_gives_zero_dA():
    X, W, A, B, dY = _problem()
    B0 = np.zeros_like(B)
    f = O.lora_forward(X, W, A, B0, 2.0)
    np.testing.assert_array_equal(f.Y, X @ W.T)
    b = O.lora_backward(X, W, A, B0, dY, 2.0)
    assert np.all(b.dA == 0.0)
    np.testing.assert_array_equal(b.dX, dY @ W)


def test_forward_equals_merged_weight():
    X, W, A, B, _ = _problem(T=9, n_in=7, n_out=6, r=2)
    s = 1.5
    f = O.lora_forward(X, W, A, B, s)
    merged = W + s * (B @ A)
    np.testing.assert_allclose(f.Y, np.einsum("ti,oi->to", X, merged), rtol=1e-13, atol=1e-13)


def _loss(Y, dY):
    return float(np.sum(Y * dY))


@pytest.mark.parametrize("p", [0.0, 0.4])
def test_backward_matches_central_finite_differences(p):
    X, W, A, B, dY = _problem(T=4, n_in=5, n_out=3, r=2, seed=5)
    s = 1.25
    keep = O.dropout_keep(p, 1, 2, 0, 0, 0, X.shape[0], X.shape[1]) if p > 0 else None
    q = O.dropout_q(p) if p > 0 else 1.0
    b = O.lora_backward(X, W, A, B, dY, s, keep, q)
    h = 1e-3

    def L(X_, A_, B_):
        return _loss(O.lora_forward(X_, W, A_, B_, s, keep, q).Y, dY)

    for name, arr, grad in [("X", X, b.dX), ("A", A, b.dA), ("B", B, b.dB)]:
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args_p = {"X": X, "A": A, "B": B}
            args_m = dict(args_p)
            args_p[name], args_m[name] = plus, minus
            fd[idx] = (L(args_p["X"], args_p["A"], args_p["B"]) -
                       L(args_m["X"], args_m["A"], args_m["B"])) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-8, atol=1e-9, err_msg=name)


def test_dropout_masks_only_the_adapter_branch():
    X, W, A, B, dY = _problem(T=5, n_in=6, n_out=4, r=2, seed=8)
    keep = O.dropout_keep(0.5, 3, 0, 0, 0, 0, 5, 6)
    f = O.lora_forward(X, W, A, B, 1.0, keep, 2.0)
    # frozen part unmasked, adapter part sees the masked input scaled by q
    np.testing.assert_allclose(f.Y, X @ W.T + 2.0 * ((keep * X) @ A.T) @ B.T, rtol=1e-13)
    # with an all-zero mask the output is exactly the frozen product
    f0 = O.lora_forward(X, W, A, B, 1.0, np.zeros_like(X), 2.0)
    np.testing.assert_array_equal(f0.Y, X @ W.T)


def test_adjointness_of_frozen_forward_and_transpose():
    X, W, A, B, dY = _problem(T=7, n_in=6, n_out=5, r=2, seed=11)
    B0 = np.zeros_like(B)
    y = O.lora_forward(X, W, A, B0, 1.0).Y
    dx = O.lora_backward(X, W, A, B0, dY, 1.0).dX
    assert abs(np.sum(y * dY) - np.sum(X * dx)) < 1e-12 * max(1.0, abs(np.sum(y * dY)))


# ---------------------------------------------------------------------------------------- DoRA
def test_dora_row_norm_matches_expanded_identity():
    _, W, A, B, _ = _problem(n_in=8, n_out=5, r=3, seed=12)
    s = 0.7
    n = O.dora_row_norm(W, A, B, s)
    WAt = W @ A.T
    AAt = A @ A.T
    n2 = np.sum(W * W, 1) + 2 * s * np.sum(B * WAt, 1) + s * s * np.einsum("oj,jk,ok->o", B, AAt, B)
    np.testing.assert_allclose(n, np.sqrt(n2), rtol=1e-12)


def test_dora_with_zero_adapter_and_row_norm_magnitude_is_plain():
    X, W, A, B, _ = _problem(seed=13)
    B0 = np.zeros_like(B)
    n = O.dora_row_norm(W, A, B0, 2.0)
    np.testing.assert_allclose(n, np.linalg.norm(W, axis=1), rtol=1e-14)
    f = O.lora_forward(X, W, A, B0, 2.0, mag=np.linalg.norm(W, axis=1), rownorm=n)
    np.testing.assert_allclose(f.Y, X @ W.T, rtol=1e-13, atol=1e-14)


def test_dora_backward_finite_differences_with_fixed_norm():
    X, W, A, B, dY = _problem(T=3, n_in=4, n_out=3, r=2, seed=14)
    s = 0.9
    mag = np.abs(_rng(15).standard_normal(3)) + 0.5
    n = O.dora_row_norm(W, A, B, s)
    b = O.lora_backward(X, W, A, B, dY, s, mag=mag, rownorm=n)
    h = 1e-3

    def L(X_, A_, B_, m_):
        return _loss(O.lora_forward(X_, W, A_, B_, s, mag=m_, rownorm=n).Y, dY)

    for name, grad in [("X", b.dX), ("A", b.dA), ("B", b.dB), ("m", b.dm)]:
        base = {"X": X, "A": A, "B": B, "m": mag}
        arr = base[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p_, m_ = dict(base), dict(base)
            p_[name] = arr.copy(); p_[name][idx] += h
            m_[name] = arr.copy(); m_[name][idx] -= h
            fd[idx] = (L(p_["X"], p_["A"], p_["B"], p_["m"]) - L(m_["X"], m_["A"], m_["B"], m_["m"])) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-8, atol=1e-9, err_msg=name)


# ------------------------------------------------------------------------------ clip / optimizer
def test_clip_hand_worked():
    g = _golden("hand_worked.json")
    for case in ("clip_3_4", "clip_normalise_only"):
        c = g[case]
        p = O.grad_prepare([np.array(c["grads"])], c["grad_scale"], c["max_norm"])
        assert p.status == O.STATUS_OK
        assert abs(p.scale - c["scale"]) < 1e-15 and abs(p.norm - c["norm"]) < 1e-15


def test_clip_closed_form_constant_tensors():
    # two constant tensors: S = n1 v1^2 + n2 v2^2
    g1, g2 = np.full(300, 0.5, np.float32), np.full((20, 7), -2.0, np.float32)
    S = 300 * 0.25 + 140 * 4.0
    gamma = 1.0 / 64
    for max_norm in (0.0, 0.1, 1e6):
        p = O.grad_prepare([g1, g2], gamma, max_norm)
        norm = gamma * math.sqrt(S)
        assert abs(p.norm - norm) < 1e-15
        want = gamma * min(1.0, max_norm / norm) if max_norm > 0 else gamma
        assert abs(p.scale - want) < 1e-17
    # a norm exactly at the limit is not clipped (strict test)
    p = O.grad_prepare([np.array([3.0, 4.0])], 1.0, 5.0)
    assert p.scale == 1.0


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
def test_clip_rejects_non_finite(bad):
    g = np.ones(10, np.float32)
    g[3] = bad
    assert O.grad_prepare([np.ones(4), g], 1.0, 1.0).status == O.STATUS_NONFINITE


def test_decay_touches_A_only_and_uses_pre_update_value():
    rng = _rng(20)
    A, B = rng.standard_normal(50).astype(np.float32), rng.standard_normal(50).astype(np.float32)
    z = np.zeros(50, np.float32)
    hp = O.AdamHP(lr=1e-2, wd=0.1, plus_ratio=4.0, step=0)
    A1, _, _ = O.adamw_update(A, z, z, z, O.KIND_A, 1.0, hp)
    B1, _, _ = O.adamw_update(B, z, z, z, O.KIND_B, 1.0, hp)
    np.testing.assert_array_equal(A1, (A.astype(np.float64) * (1 - 1e-2 * 0.1)).astype(np.float32))
    np.testing.assert_array_equal(B1, B)


def test_decay_uses_scheduled_not_bias_corrected_lr():
    # g = 0 with nonzero moments at step k: decay term is lr*wd*A regardless of 1/(1-b1^k)
    A = np.full(4, 2.0, np.float32)
    m = np.zeros(4, np.float32)
    v = np.zeros(4, np.float32)
    hp = O.AdamHP(lr=0.5, wd=0.2, step=3)
    A1, _, _ = O.adamw_update(A, np.zeros(4), m, v, O.KIND_A, 1.0, hp)
    np.testing.assert_array_equal(A1, np.full(4, 2.0 - 0.5 * 0.2 * 2.0, np.float32))


def test_adam_first_step_is_normalised_sign_step():
    # textbook Adam from zero moments: m_hat = g_hat, v_hat = g_hat^2, u = g_hat / (|g_hat| + eps)
    g = np.array([1e-3, -2.0, 5e-9, 0.0], np.float64)
    p = np.zeros(4, np.float32)
    z = np.zeros(4, np.float32)
    hp = O.AdamHP(lr=0.1, wd=0.0, step=0)
    for kind, ratio in ((O.KIND_A, 1.0), (O.KIND_B, 1.0)):
        p1, m1, v1 = O.adamw_update(p, g, z, z, kind, 1.0, hp)
        want = -0.1 * ratio * g / (np.abs(g) + 1e-8)
        np.testing.assert_allclose(p1, want.astype(np.float32), rtol=1e-6, atol=1e-30)
        np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-6)
        np.testing.assert_allclose(v1, 0.001 * g * g, rtol=1e-6)


def test_lora_plus_scales_B_update_exactly():
    # from B = 0 a power-of-two ratio scales the fp32 result exactly, and decay never applies
    rng = _rng(21)
    B = np.zeros(64, np.float32)
    g = rng.standard_normal(64)
    m = (rng.standard_normal(64) * 1e-3).astype(np.float32)
    v = (rng.random(64) * 1e-6).astype(np.float32)
    d = {}
    for rho in (1.0, 16.0):
        hp = O.AdamHP(lr=1e-3, wd=0.5, plus_ratio=rho, step=4)
        d[rho], _, _ = O.adamw_update(B, g, m, v, O.KIND_B, 0.3, hp)
    np.testing.assert_array_equal(d[16.0], 16.0 * d[1.0])
    assert np.all(d[1.0] != 0)


def test_magnitude_update_has_no_decay_and_ratio_one():
    mag = np.full(8, 3.0, np.float32)
    z = np.zeros(8, np.float32)
    hp = O.AdamHP(lr=0.5, wd=0.9, plus_ratio=10.0, step=0)
    m1, _, _ = O.adamw_update(mag, np.zeros(8), z, z, O.KIND_MAG, 1.0, hp)
    np.testing.assert_array_equal(m1, mag)
    g = np.full(8, 2.0)
    m2, _, _ = O.adamw_update(mag, g, z, z, O.KIND_MAG, 1.0, hp)
    np.testing.assert_allclose(m2, 3.0 - 0.5 * 2.0 / (2.0 + 1e-8), rtol=1e-7)


# ------------------------------------------------------------------------------------- schedule
def test_schedule_closed_forms():
    base, mn = 1e-4, 1e-6
    assert O.lr_at("constant", base, 12345, 10, 100, mn) == base
    assert O.lr_at("cosine", base, 0, 10, 100, mn) == pytest.approx(base / 10, rel=1e-15)
    assert O.lr_at("cosine", base, 9, 10, 100, mn) == pytest.approx(base, rel=1e-15)
    assert O.lr_at("cosine", base, 10, 10, 100, mn) == pytest.approx(base, rel=1e-15)
    assert O.lr_at("cosine", base, 55, 10, 100, mn) == pytest.approx((base + mn) / 2, rel=1e-14)
    assert O.lr_at("cosine", base, 100, 10, 100, mn) == pytest.approx(mn, rel=1e-12)
    assert O.lr_at("cosine", base, 1000, 10, 100, mn) == pytest.approx(mn, rel=1e-12)
    g = _golden("hand_worked.json")["cosine_at_25"]
    assert O.lr_at("cosine", base, 25, 10, 100, mn) == pytest.approx(g["lr"], rel=1e-14)
    seq = [O.lr_at("cosine", base, k, 10, 100, mn) for k in range(10, 101)]
    assert all(a >= b for a, b in zip(seq, seq[1:]))


# ---------------------------------------------------------------------------------- accumulation
def _small_problems(T, seed, n_layers=2, dora=False):
    rng = _rng(seed)
    problems, state = {}, {}
    for l in range(n_layers):
        X = rng.standard_normal((T, 8))
        W = rng.standard_normal((6, 8)) / 3
        dY = rng.standard_normal((T, 6))
        A = rng.uniform(-0.8, 0.8, (2, 8)).astype(np.float32)
        B = (rng.standard_normal((6, 2)) * 0.1).astype(np.float32)
        problems[l] = dict(X=X, W=W, dY=dY, layer=l, proj=0)
        z = lambda a: np.zeros_like(a)
        st = O.AdapterState(A, B, z(A), z(A), z(B), z(B))
        if dora:
            st.mag = np.linalg.norm(W, axis=1).astype(np.float32)
            st.mM, st.vM = z(st.mag), z(st.mag)
        state[l] = st
    return problems, state


def test_accumulated_chunks_equal_concatenated_batch():
    problems, state = _small_problems(T=12, seed=30)
    kw = dict(s=2.0, p=0.0, seed=0, opt_step=0, max_norm=1.0, hp=O.AdamHP(lr=1e-3))
    r3 = O.run_single_step(problems, state, chunks=3, **kw)
    r1 = O.run_single_step(problems, state, chunks=1, **kw)
    for k in problems:
        for a, b in zip(r3.grads[k][:2], r1.grads[k][:2]):
            np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-6)
    assert r3.prepared.scale == pytest.approx(r1.prepared.scale, rel=1e-6)
    # gamma = 1 / total prediction tokens
    sq = sum(float(np.sum(np.float64(g) ** 2)) for k in problems for g in r1.grads[k][:2])
    assert r1.prepared.norm == pytest.approx(math.sqrt(sq) / 12, rel=1e-12)


def test_step_rejects_non_finite_without_mutation():
    problems, state = _small_problems(T=4, seed=31)
    problems[1]["dY"] = problems[1]["dY"].copy()
    problems[1]["dY"][2, 3] = np.nan
    r = O.run_single_step(problems, state, s=1.0, chunks=2, p=0.0, seed=0, opt_step=0,
                          max_norm=1.0, hp=O.AdamHP(lr=1e-3))
    assert r.prepared.status == O.STATUS_NONFINITE
    for k in problems:
        assert r.new_state[k] is state[k]


# ------------------------------------------------------------------------------------ multi-LoRA
def test_token_slots_brute_force():
    seg_start = [0, 3, 3, 7, 10]
    seg_slot = [1, 0, 2, 9]
    ts = O.token_slots(12, seg_start, seg_slot, 3)
    assert list(ts) == [1, 1, 1, 2, 2, 2, 2, -1, -1, -1, -1, -1]


def test_multi_single_slot_equals_single_lora():
    X, W, A, B, dY = _problem(T=8, n_in=6, n_out=5, r=3, seed=40)
    keep = O.dropout_keep(0.25, 1, 0, 0, 0, 0, 8, 6)
    q = O.dropout_q(0.25)
    slots = [O.SlotTensors(A, B, 1.5)]
    ts = O.token_slots(8, [0, 8], [0], 1)
    Y, H = O.multi_lora_forward(X, W, slots, ts, keep, q)
    f = O.lora_forward(X, W, A, B, 1.5, keep, q)
    np.testing.assert_allclose(Y, f.Y, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(H, f.H, rtol=1e-13, atol=1e-13)
    dX, dA, dB = O.multi_lora_backward(X, W, dY, slots, ts, keep, q)
    b = O.lora_backward(X, W, A, B, dY, 1.5, keep, q)
    np.testing.assert_allclose(dX, b.dX, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dA[0], b.dA, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dB[0], b.dB, rtol=1e-12, atol=1e-12)


def test_multi_slot_gradient_equals_that_slot_training_alone():
    rng = _rng(41)
    T, n_in, n_out = 20, 6, 4
    X, W, dY = rng.standard_normal((T, n_in)), rng.standard_normal((n_out, n_in)), rng.standard_normal((T, n_out))
    slots = [O.SlotTensors(rng.standard_normal((r, n_in)), rng.standard_normal((n_out, r)), s)
             for r, s in ((2, 1.0), (3, 2.0), (1, 0.5))]
    seg_start, seg_slot = [0, 5, 9, 14, 20], [2, 0, 2, 1]
    ts = O.token_slots(T, seg_start, seg_slot, 3)
    dX, dA, dB = O.multi_lora_backward(X, W, dY, slots, ts)
    dXv, dAv, dBv = O.multi_lora_backward_vectorised(X, W, dY, slots, ts)
    np.testing.assert_allclose(dX, dXv, rtol=1e-12, atol=1e-12)
    for k, sl in enumerate(slots):
        rows = ts == k
        alone = O.lora_backward(X[rows], W, sl.A, sl.B, dY[rows], sl.s)
        np.testing.assert_allclose(dA[k], alone.dA, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dB[k], alone.dB, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dAv[k], alone.dA, rtol=1e-12, atol=1e-12)
    # the 1/adapter_global_batch_size scaled update of a slot is what it would get alone
    gbs = 64
    p_multi = O.grad_prepare([dA[1], dB[1]], 1.0 / gbs, 1.0)
    p_alone = O.grad_prepare([O.lora_backward(X[ts == 1], W, slots[1].A, slots[1].B, dY[ts == 1], 2.0).dA,
                              O.lora_backward(X[ts == 1], W, slots[1].A, slots[1].B, dY[ts == 1], 2.0).dB],
                             1.0 / gbs, 1.0)
    assert p_multi.scale == pytest.approx(p_alone.scale, rel=1e-12)


# ---- adapter-state maintenance ("4.3. Training Guide", Validation early stopping; "Multi-LoRA
# Training Example (fully-async)", adapter retirement) ----
def _arenas(n=64, seed=7):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal(n).astype(np.float32) for _ in range(4)]


def test_restore_returns_the_snapshot_and_a_fresh_optimizer():
    # snapshot, two updates that move params and moments, restore: params are the snapshot bit for
    # bit inside the groups, moments are zero there, everything outside the groups is untouched
    p, g, m, v = _arenas()
    v = np.abs(v)                          # a second moment is non-negative
    groups = [(4, 20), (32, 13)]
    snap = O.snapshot(p, np.full_like(p, np.nan), groups)
    hp = O.AdamHP(lr=0.05, wd=0.01)
    p1, m1, v1 = p.copy(), m.copy(), v.copy()
    for k in range(2):
        hp.step = k
        p1, m1, v1 = O.adamw_update(p1, g, m1, v1, O.KIND_A, 1.0, hp)
    pr, gr, mr, vr = O.restore(p1, snap, g, m1, v1, groups, zero_grads=True)
    inside = np.zeros(p.size, bool)
    for off, cnt in groups:
        inside[off:off + cnt] = True
    assert np.array_equal(pr[inside], p[inside])
    assert not np.any(mr[inside]) and not np.any(vr[inside]) and not np.any(gr[inside])
    assert np.array_equal(pr[~inside], p1[~inside])
    assert np.array_equal(mr[~inside], m1[~inside]) and np.array_equal(gr[~inside], g[~inside])
    assert np.all(np.isnan(snap[~inside]))


def test_step_after_restore_is_the_normalised_sign_step_from_the_snapshot():
    # after the reset the next update (update count restarted at 0) is Adam's first step from
    # zero moments, whatever the moments were before: p_snap - lr * g / (|g| + eps) for B
    p, g, m, v = _arenas(seed=11)
    v = np.abs(v) + 1.0                   # stale moments that would change the update
    groups = [(0, 64)]
    snap = O.snapshot(p, np.zeros_like(p), groups)
    pr, _, mr, vr = O.restore(p + 1.0, snap, g, m, v, groups, zero_grads=False)
    p1, _, _ = O.adamw_update(pr, g, mr, vr, O.KIND_B, 1.0, O.AdamHP(lr=0.1, wd=0.0, step=0))
    g64 = g.astype(np.float64)
    want = p.astype(np.float64) - 0.1 * g64 / (np.abs(g64) + 1e-8)
    np.testing.assert_allclose(p1, want.astype(np.float32), rtol=1e-6, atol=1e-7)


def test_retire_clears_only_the_retired_slot():
    p, g, m, v = _arenas(seed=3)
    slots = [(0, 16), (16, 24), (40, 24)]
    pr, gr, mr, vr = O.retire(p, g, m, v, [slots[1]], clear_params=True)
    for (off, cnt), retired in zip(slots, (False, True, False)):
        sl = slice(off, off + cnt)
        if retired:
            assert not np.any(pr[sl]) and not np.any(gr[sl]) and not np.any(mr[sl]) and not np.any(vr[sl])
        else:
            for a, b in ((pr, p), (gr, g), (mr, m), (vr, v)):
                assert np.array_equal(a[sl], b[sl])
    pk, _, _, _ = O.retire(p, g, m, v, [slots[1]], clear_params=False)
    assert np.array_equal(pk, p)


# ---- chained layers ("4.3. Training Guide", Truncated BPTT, Gradient accumulation) ----
def _chain(seed=5, dims=(6, 5, 7), r=2, T=4, zero_b=False):
    rng = np.random.default_rng(seed)
    Ws = [rng.standard_normal((dims[l + 1], dims[l])) / math.sqrt(dims[l]) for l in range(len(dims) - 1)]
    As = [rng.standard_normal((r, dims[l])) for l in range(len(dims) - 1)]
    Bs = [np.zeros((dims[l + 1], r)) if zero_b else 0.3 * rng.standard_normal((dims[l + 1], r))
          for l in range(len(dims) - 1)]
    X0 = rng.standard_normal((T, dims[0]))
    dY = rng.standard_normal((T, dims[-1]))
    return Ws, As, Bs, X0, dY


def test_chain_equals_product_of_merged_weights():
    Ws, As, Bs, X0, dY = _chain()
    s = 1.5
    res = O.chained_forward_backward(X0, Ws, As, Bs, dY, s, chunks=2)
    M = [W + s * B @ A for W, A, B in zip(Ws, As, Bs)]
    want_Y = X0 @ M[0].T @ M[1].T
    want_dX = dY @ M[1] @ M[0]
    np.testing.assert_allclose(res.Y, want_Y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res.dX, want_dX, rtol=1e-12, atol=1e-12)


def test_chain_with_zero_adapters_gives_zero_dA_and_frozen_products():
    Ws, As, Bs, X0, dY = _chain(zero_b=True)
    res = O.chained_forward_backward(X0, Ws, As, Bs, dY, 2.0, chunks=1)
    for gA, _ in res.grads:
        assert not np.any(gA)
    np.testing.assert_allclose(res.Y, X0 @ Ws[0].T @ Ws[1].T, rtol=1e-12, atol=1e-12)


def test_chain_gradients_match_central_finite_differences():
    Ws, As, Bs, X0, dY = _chain(seed=9)
    s = 0.7
    res = O.chained_forward_backward(X0, Ws, As, Bs, dY, s, chunks=2)

    def loss(As_, Bs_):
        Y = X0
        for W, A, B in zip(Ws, As_, Bs_):
            Y = Y @ (W + s * B @ A).T
        return float(np.sum(Y * dY))

    h = 1e-5
    for l in range(2):
        for name, idx in (("A", (1, 3)), ("B", (2, 0))):
            Ap = [a.copy() for a in As]
            Am = [a.copy() for a in As]
            Bp = [b.copy() for b in Bs]
            Bm = [b.copy() for b in Bs]
            if name == "A":
                Ap[l][idx] += h
                Am[l][idx] -= h
            else:
                Bp[l][idx] += h
                Bm[l][idx] -= h
            fd = (loss(Ap, Bp) - loss(Am, Bm)) / (2 * h)
            got = res.grads[l][0 if name == "A" else 1][idx]
            assert abs(got - fd) <= 1e-5 * max(1.0, abs(fd))


def test_chain_chunking_changes_only_the_summation_order():
    Ws, As, Bs, X0, dY = _chain(seed=13, T=8)
    one = O.chained_forward_backward(X0, Ws, As, Bs, dY, 1.0, chunks=1)
    four = O.chained_forward_backward(X0, Ws, As, Bs, dY, 1.0, chunks=4)
    np.testing.assert_allclose(one.Y, four.Y, rtol=1e-13, atol=1e-13)
    for (a1, b1), (a4, b4) in zip(one.grads, four.grads):
        np.testing.assert_allclose(a1, a4, rtol=1e-6, atol=1e-6)
        np.testing.assert_allclose(b1, b4, rtol=1e-6, atol=1e-6)


# ---- FP8 E4M3 frozen base ----
def test_e4m3_reference_values():
    # OCP 8-bit float E4M3: 448 largest finite, 2^-6 smallest normal, 2^-9 smallest subnormal,
    # 1.0 = 0x38, S.1111.111 is NaN (no infinities)
    dec = O.e4m3_decode(np.array([0x7E, 0xFE, 0x38, 0x08, 0x01, 0x00, 0x80, 0x77, 0x3C],
                                 np.uint8))
    np.testing.assert_array_equal(dec, [448.0, -448.0, 1.0, 2.0 ** -6, 2.0 ** -9, 0.0, -0.0,
                                        240.0, 1.5])
    assert np.isnan(O.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_round_trip_and_monotone():
    codes = np.arange(256, dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    fin = ~np.isnan(vals)
    assert np.array_equal(O.e4m3_encode(vals[fin].astype(np.float32)), codes[fin])
    xs = np.linspace(0.0, 500.0, 20001).astype(np.float32)
    dec = O.e4m3_decode(O.e4m3_encode(xs))
    assert np.all(np.diff(dec) >= 0)


def test_e4m3_ties_to_even_and_saturation():
    x = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -11, 463.9, 464.0, 1e6, -1e6, -0.0],
                 np.float32)
    np.testing.assert_array_equal(O.e4m3_encode(x), [0x38, 0x3A, 0x00, 0x01, 0x7E, 0x7E, 0x7E,
                                                     0xFE, 0x80])


def test_e4m3_relative_error_bound():
    # three mantissa bits: round-to-nearest error <= 2^-4 of the value in the normal range
    rng = np.random.default_rng(0)
    x = np.exp(rng.uniform(np.log(2.0 ** -6), np.log(448.0), 5000)).astype(np.float32)
    err = np.abs(O.e4m3_decode(O.e4m3_encode(x)) - x) / x
    assert err.max() <= 2.0 ** -4 + 1e-12


def test_quantize_rows_maps_each_row_max_to_448():
    rng = np.random.default_rng(1)
    M = (rng.standard_normal((16, 40)) * np.exp(rng.uniform(-5, 5, (16, 1)))).astype(np.float32)
    M[3] = 0.0
    codes, sc = O.quantize_rows_e4m3(M)
    assert sc[3] == 1.0 and not np.any(codes[3] & 0x7F)
    for r in range(16):
        if r == 3:
            continue
        assert np.max(np.abs(O.e4m3_decode(codes[r]))) == 448.0
        assert sc[r] == np.float32(np.max(np.abs(M[r])) / np.float32(448.0))


def test_fp8_product_brute_force_and_error_bound():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((3, 20)).astype(np.float32)
    W = rng.standard_normal((4, 20)).astype(np.float32)
    Xc, sx = O.quantize_rows_e4m3(X)
    Wc, sw = O.quantize_rows_e4m3(W)
    got = O.fp8_product(Xc, sx, Wc, sw)
    for t in range(3):
        for n in range(4):
            acc = 0.0
            for k in range(20):
                acc += O.e4m3_decode([Xc[t, k]])[0] * O.e4m3_decode([Wc[n, k]])[0]
            assert abs(got[t, n] - float(sx[t]) * acc * float(sw[n])) <= 1e-12 * max(1.0, abs(acc))
    # each operand is within 2^-4 (relative) of its value, or within half a subnormal step
    bound = (np.abs(X) @ np.abs(W).T) * (2 * 2.0 ** -4 + 2.0 ** -8) \
        + 2.0 ** -10 * (sx[:, None] * (np.abs(W).sum(1))[None, :] + (np.abs(X).sum(1))[:, None] * sw[None, :])
    assert np.all(np.abs(got - X.astype(np.float64) @ W.T.astype(np.float64)) <= bound)


def test_fp8_forward_with_zero_adapter_is_the_fp8_product():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((5, 16)).astype(np.float32)
    W = rng.standard_normal((6, 16)).astype(np.float32)
    A = rng.standard_normal((4, 16)).astype(np.float32)
    B = np.zeros((6, 4), np.float32)
    f = O.lora_forward_fp8(X, W, A, B, 2.0)
    Xc, sx = O.quantize_rows_e4m3(X)
    Wc, sw = O.quantize_rows_e4m3(W)
    np.testing.assert_array_equal(f.Y, O.fp8_product(Xc, sx, Wc, sw))


# ---- fused projections ("LoRA Training and Serving", --lora-type lora / canonical_lora) ----
def test_fused_projections_equal_the_stacked_effective_weight():
    # one fused linear with the effective weight W_eff = [W_p + s B_p A_p]_p stacked by rows:
    # Y_cat = X W_eff^T and dX = dY_cat W_eff (closed forms, p = 0)
    rng = np.random.default_rng(17)
    T, d_in, outs, r, s = 5, 12, (8, 4, 4), 3, 0.5
    X = rng.standard_normal((T, d_in))
    Ws = [rng.standard_normal((o, d_in)) for o in outs]
    As = [rng.standard_normal((r, d_in)) for _ in outs]
    Bs = [rng.standard_normal((o, r)) for o in outs]
    dYs = [rng.standard_normal((T, o)) for o in outs]
    res = O.fused_forward_backward(X, Ws, As, Bs, dYs, s)
    W_eff = np.concatenate([W + s * B @ A for W, A, B in zip(Ws, As, Bs)], axis=0)
    np.testing.assert_allclose(res.Y, X @ W_eff.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res.dX, np.concatenate(dYs, axis=1) @ W_eff, rtol=1e-12, atol=1e-12)
    # each projection's adapter gradient sees only its own output columns
    for (gA, gB), W, A, B, dY in zip(res.grads, Ws, As, Bs, dYs):
        np.testing.assert_allclose(gB, s * dY.T @ (X @ A.T), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(gA, s * (dY @ B).T @ X, rtol=1e-12, atol=1e-12)


# ---- FP8 dX ("LoRA Training and Serving", Quantized rollout: E4M3 frozen base) ----
def _e4m3_col_scaled(W):
    """Independent per-input-column quantisation of W (the layout the dX product contracts
    over the output rows of W): amax_i = max_o |W[o, i]|, codes e4m3(W[o, i] * 448 / amax_i)."""
    W = np.asarray(W, np.float32)
    amax = np.max(np.abs(W), axis=0)
    rcp = (np.float32(448.0) / amax).astype(np.float32)
    codes = O.e4m3_encode((W * rcp[None, :]).astype(np.float32))
    return codes, (amax / np.float32(448.0)).astype(np.float32)


def _fp8_dx_problem(seed=21, T=3, n_out=24, n_in=5, r=2):
    rng = np.random.default_rng(seed)
    dY = rng.standard_normal((T, n_out)).astype(np.float32)
    # input columns of W with scales 10^-5 .. 10^1: a per-output-row quantisation of W (the
    # forward's layout, wrong for dX) flushes the small columns to zero, far outside the
    # per-column bound below
    W = (rng.standard_normal((n_out, n_in)) * np.logspace(-5, 1, n_in)[None, :]).astype(np.float32)
    A = rng.standard_normal((r, n_in)).astype(np.float32)
    B = rng.standard_normal((n_out, r)).astype(np.float32)
    return dY, W, A, B


def test_fp8_dx_brute_force_over_decoded_codes():
    dY, W, A, B = _fp8_dx_problem()
    s = 1.5
    G = dY.astype(np.float64) @ B.astype(np.float64)
    got = O.lora_dx_fp8(dY, W, A, G, s)
    Dc, sd = O.quantize_rows_e4m3(dY)          # per token (row of dY)
    Wc, sw = _e4m3_col_scaled(W)                 # per input column of W
    T, n_out = dY.shape
    n_in = W.shape[1]
    for t in range(T):
        for i in range(n_in):
            acc = 0.0
            for o in range(n_out):
                acc += float(O.e4m3_decode([Dc[t, o]])[0]) * float(O.e4m3_decode([Wc[o, i]])[0])
            lora = sum(G[t, j] * float(A[j, i]) for j in range(A.shape[0]))
            want = float(sd[t]) * acc * float(sw[i]) + s * lora
            assert abs(got[t, i] - want) <= 1e-12 * max(1.0, abs(want)), (t, i)


def test_fp8_dx_with_zero_adapter_is_the_fp8_product_of_dY_and_W_transposed():
    dY, W, A, _ = _fp8_dx_problem(seed=22)
    G0 = np.zeros((dY.shape[0], A.shape[0]))
    got = O.lora_dx_fp8(dY, W, A, G0, 2.0)
    Dc, sd = O.quantize_rows_e4m3(dY)
    Wtc, swt = O.quantize_rows_e4m3(np.ascontiguousarray(W.T))
    np.testing.assert_array_equal(got, O.fp8_product(Dc, sd, Wtc, swt))


def test_fp8_dx_within_the_e4m3_bound_of_the_exact_backward():
    dY, W, A, B = _fp8_dx_problem(seed=23, T=4)
    rng = np.random.default_rng(24)
    X = rng.standard_normal((dY.shape[0], W.shape[1])).astype(np.float32)
    s, p = 0.75, 0.3
    keep = O.dropout_keep(p, 5, 1, 0, 2, 1, X.shape[0], X.shape[1])
    q = O.dropout_q(p)
    ref = O.lora_backward(X, W, A, B, dY, s, keep, q)
    got = O.lora_dx_fp8(dY, W, A, ref.G, s, keep, q)
    # each quantised operand is within 2^-4 of its value (relative) or half a subnormal step
    # (2^-10 in code units) of it; the adapter term is exact in both
    sd = np.max(np.abs(dY), axis=1) / 448.0
    sw = np.max(np.abs(W), axis=0) / 448.0
    bound = (np.abs(dY).astype(np.float64) @ np.abs(W)) * (2 * 2.0 ** -4 + 2.0 ** -8) \
        + 2.0 ** -10 * (sd[:, None] * np.abs(W).sum(0)[None, :] + np.abs(dY).sum(1)[:, None] * sw[None, :])
    assert np.all(np.abs(got - ref.dX) <= bound + 1e-12)
    # and a per-output-row quantisation of W would not be: its small input columns lose
    # everything, so the same bound fails there
    Wc_row, sw_row = O.quantize_rows_e4m3(W)
    Dc, sdq = O.quantize_rows_e4m3(dY)
    wrong = (sdq[:, None] * (O.e4m3_decode(Dc) @ (O.e4m3_decode(Wc_row) * sw_row[:, None].astype(np.float64))))
    frozen = dY.astype(np.float64) @ W.astype(np.float64)
    assert np.any(np.abs(wrong - frozen) > bound)


# ---- adapter gradients alone ("Backward Bug Hunts and Vulkan Tiled GEMM", Bug #1 / #2) ----
@pytest.mark.parametrize("p", [0.0, 0.35])
def test_adapter_grads_equal_the_full_backward(p):
    X, W, A, B, dY = _problem(T=7, n_in=6, n_out=5, r=3, seed=31)
    s = 1.7
    keep = O.dropout_keep(p, 9, 4, 1, 3, 2, X.shape[0], X.shape[1]) if p > 0 else None
    q = O.dropout_q(p) if p > 0 else 1.0
    dA, dB = O.lora_adapter_grads(X, A, B, dY, s, keep, q)
    ref = O.lora_backward(X, W, A, B, dY, s, keep, q)
    np.testing.assert_allclose(dA, ref.dA, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dB, ref.dB, rtol=1e-13, atol=1e-13)


def test_adapter_grads_match_central_finite_differences():
    X, W, A, B, dY = _problem(T=5, n_in=4, n_out=3, r=2, seed=32)
    s, p = 0.9, 0.5
    keep = O.dropout_keep(p, 2, 0, 1, 0, 4, X.shape[0], X.shape[1])
    q = O.dropout_q(p)
    dA, dB = O.lora_adapter_grads(X, A, B, dY, s, keep, q)
    h = 1e-3

    def L(A_, B_):
        return _loss(O.lora_forward(X, W, A_, B_, s, keep, q).Y, dY)

    for arr, grad, which in ((A, dA, "A"), (B, dB, "B")):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            fd[idx] = ((L(plus, B) - L(minus, B)) if which == "A" else (L(A, plus) - L(A, minus))) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-8, atol=1e-9, err_msg=which)


# ---- Adam bias correction at k > 1 ("4.3. Training Guide", Optimizer) ----
def test_adam_constant_gradient_gives_the_normalised_sign_step_at_every_k():
    # from zero moments and a constant g_hat, after k updates m = (1 - b1^k) g_hat and
    # v = (1 - b2^k) g_hat^2, so the corrected moments are g_hat and g_hat^2 and every update is
    # -lr g_hat / (|g_hat| + eps); a bias correction with the wrong power (or none) breaks this
    g = np.array([3e-2, -1.5, 4e-6, 0.25], np.float64)
    lr = 1e-2
    p = np.zeros(4, np.float32)
    m = np.zeros(4, np.float32)
    v = np.zeros(4, np.float32)
    want = -lr * g / (np.abs(g) + 1e-8)
    for k in range(12):
        hp = O.AdamHP(lr=lr, wd=0.0, step=k)
        p1, m, v = O.adamw_update(p, g, m, v, O.KIND_B, 1.0, hp)
        np.testing.assert_allclose(p1.astype(np.float64) - p.astype(np.float64), want,
                                   rtol=2e-5, atol=1e-12, err_msg=f"update {k + 1}")
        np.testing.assert_allclose(m, (1 - 0.9 ** (k + 1)) * g, rtol=1e-5)
        np.testing.assert_allclose(v, (1 - 0.999 ** (k + 1)) * g * g, rtol=1e-5)
        p = p1
