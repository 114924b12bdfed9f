"""Parity at the benchmark's full sizes, in the launch configuration bench.py times: the step on 4
streams, captured in a CUDA graph and replayed once from the seeded initial state.

Frozen products at these sizes are too large for the float64 oracle over every token, so the
per-token outputs (Y, H, dX) are checked on sampled tokens (each token's outputs depend on that
token alone), while the adapter gradients and the post-step adapters, which sum over all tokens,
are checked in full against the oracle's adapter-gradient form."""
import numpy as np
import pytest
import torch

import lora_inputs as LI
from oracle import lora_oracle as O

from tests.helpers import (TOL_BF16, TOL_BF16_STEP, TOL_F32, build_single, check_post_step,
                           grad_bounds, rel_err, to64)

pytestmark = pytest.mark.gpu

N_SAMPLE = 48


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_adapter_adamw_gb300 import binding
    return binding


def _sample_rows(T: int, seed: int, extra=()):
    """Sorted token indices: a seeded sample plus the ends and the given boundaries (a torch
    index tensor on the CPU)."""
    rng = np.random.default_rng(seed)
    rows = set(int(x) for x in rng.choice(T, size=min(T, N_SAMPLE), replace=False))
    rows.update([0, T - 1])
    rows.update(int(x) for x in extra if 0 <= x < T)
    return torch.tensor(sorted(rows), dtype=torch.long)


def _rows_of(t, rows):
    return t[rows.to(t.device)]


def _replay_once(fn):
    """Capture fn in a CUDA graph (nothing runs during capture) and replay it once."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()


def _warm_library(L):
    """Run the library once outside any capture (lazy kernel attributes, tensor-map encoder)."""
    for name in ("c1", "c3"):
        cfg = LI.with_overrides(LI.CONFIGS[name], tokens=64, chunks=1)
        step, *_ = build_single(cfg, [0], [0])
        step.run(cfg.opt_step, 1e-4, zero_grads=False)
    torch.cuda.synchronize()


@pytest.mark.parametrize("name,layers", [("c2", None), ("c4", [0]), ("c4dora", [0])])
def test_fullsize_single_sampled(L, name, layers):
    cfg = LI.CONFIGS[name]
    layers = list(range(cfg.layers)) if layers is None else layers
    tol, tol_step = (TOL_F32, TOL_F32) if cfg.dtype == "f32" else (TOL_BF16, TOL_BF16_STEP)
    _warm_library(L)
    step, problems, state, s, hp_o = build_single(cfg, layers, range(len(cfg.projs)),
                                                  n_streams=4)
    assert cfg.dropout_p == 0.0   # the full-size configs with a single adapter have no dropout
    _replay_once(lambda: step.run(cfg.opt_step, hp_o.lr, zero_grads=False))
    assert int(step.status.item()) == O.STATUS_OK
    T = cfg.tokens
    ct = T // cfg.chunks
    edges = [c * ct for c in range(cfg.chunks)] + [c * ct - 1 for c in range(1, cfg.chunks)]
    rows = _sample_rows(T, 7, extra=edges)
    grads, errs = [], {}
    for lin in step.linears:
        key = (lin.layer, lin.proj_id)
        pr, st = problems[key], state[key]
        mag = rown = None
        dY = pr["dY"]
        if cfg.dora:
            mag = st.mag
            rown = O.dora_row_norm(pr["W"], st.A, st.B, s)
        # sampled per-token outputs
        f = O.lora_forward(_rows_of(pr["X"], rows), pr["W"], st.A, st.B, s, mag=mag, rownorm=rown)
        b = O.lora_backward(_rows_of(pr["X"], rows), pr["W"], st.A, st.B, _rows_of(dY, rows), s,
                            mag=mag, rownorm=rown)
        errs[(key, "Y")] = rel_err(_rows_of(lin.Y, rows), f.Y)
        errs[(key, "H")] = rel_err(_rows_of(lin.H, rows), s * f.H)
        errs[(key, "dX")] = rel_err(_rows_of(lin.dX, rows), b.dX)
        # adapter gradients over all tokens: dY' = dY * m / n in DoRA mode
        dYp = to64(dY) * (mag / rown)[None, :] if cfg.dora else dY
        gA, gB = O.lora_adapter_grads(pr["X"], st.A, st.B, dYp, s)
        errs[(key, "dA")] = rel_err(lin.gA, gA)
        errs[(key, "dB")] = rel_err(lin.gB, gB)
        grads.append((key, [gA, gB]))
    for k, e in errs.items():
        assert e <= tol, (k, e, name)
    if cfg.dora:
        # dm = sum_t dY * Y / m needs the full frozen product over every token, beyond the
        # oracle at this size; dm, the DoRA clip norm and the DoRA post-step state are checked
        # at T = 256 in test_gpu_parity
        return
    # global clip over every adapter of the step, then AdamW from the initial state
    prep = O.grad_prepare([g.astype(np.float32) for _, gl in grads for g in gl], 1.0 / T,
                          cfg.max_norm)
    sn = step.scale_norm.cpu().numpy()
    tol_norm = 1e-5 if cfg.dtype == "f32" else 1e-3
    assert abs(sn[0] - prep.scale) <= tol_norm * abs(prep.scale)
    assert abs(sn[1] - prep.norm) <= tol_norm * abs(prep.norm)
    # post-step A and B: the per-tensor bar, with the Adam-conditioning band near g_hat ~ 0 (the
    # gradients' fp32 forward-error bounds, as in test_gpu_parity)
    n_clause = 0
    for lin in step.linears:
        key = (lin.layer, lin.proj_id)
        st = state[key]
        gl = dict(grads)[key]
        bA, bB = grad_bounds(problems[key], st.A, st.B, s, None, 1.0)
        nA, _ = check_post_step(lin.A, st.A, st.mA, st.vA, gl[0], bA, O.KIND_A, prep.scale, hp_o,
                                tol_step)
        nB, _ = check_post_step(lin.B, st.B, st.mB, st.vB, gl[1], bB, O.KIND_B, prep.scale, hp_o,
                                tol_step)
        n_clause += nA + nB
    if cfg.dtype != "f32":
        assert n_clause == 0


def test_fullsize_fp8_sampled(L):
    """c4 with the E4M3 frozen product, layer 0's wq at full size (T 8192, 4096 x 4096): the
    per-token outputs on sampled tokens against the oracle's E4M3 product (codes per token row,
    so a sampled row quantises as it does in the full batch), the adapter gradients in full."""
    cfg = LI.CONFIGS["c4fp8"]
    _warm_library(L)
    step, problems, state, s, hp_o = build_single(cfg, [0], [0], n_streams=4)
    _replay_once(lambda: step.run(cfg.opt_step, hp_o.lr, zero_grads=False))
    assert int(step.status.item()) == O.STATUS_OK
    rows = _sample_rows(cfg.tokens, 11)
    lin = step.linears[0]
    pr, st = problems[(0, 0)], state[(0, 0)]
    X = _rows_of(pr["X"], rows).float().numpy()
    dY = _rows_of(pr["dY"], rows).float().numpy()
    W = pr["W"].float().numpy()
    f = O.lora_forward_fp8(X, W, st.A, st.B, s)
    b = O.lora_backward(X, W, st.A, st.B, dY, s)
    assert rel_err(_rows_of(lin.Y, rows), f.Y) <= TOL_BF16
    assert rel_err(_rows_of(lin.H, rows), s * f.H) <= TOL_BF16
    assert rel_err(_rows_of(lin.dX, rows), O.lora_dx_fp8(dY, W, st.A, b.G, s)) <= TOL_BF16
    gA, gB = O.lora_adapter_grads(pr["X"], st.A, st.B, pr["dY"], s)
    assert rel_err(lin.gA, gA) <= TOL_BF16
    assert rel_err(lin.gB, gB) <= TOL_BF16


def test_fullsize_multi_sampled(L):
    from bwd_adapter_adamw_gb300.step import MultiLinear, MultiLoraStep
    cfg = LI.CONFIGS["c5"]
    T = cfg.tokens
    r = LI.make_routing(cfg, T)
    ranks = r.slot_rank
    scales = [O.lora_scale(a, rk, cfg.rslora) for a, rk in zip(r.slot_alpha, ranks)]
    _warm_library(L)
    lins, host = [], {}
    for pi, pr in enumerate(cfg.projs):
        X = LI.make_x(cfg, 0, pr, tokens=T)
        W = LI.make_w(cfg, 0, pr)
        dY = LI.make_dy(cfg, 0, pr, tokens=T)
        lins.append(MultiLinear(pi, X.cuda(), W.cuda(), dY.cuda()))
        host[pi] = dict(X=X, W=W, dY=dY,
                        slots=[(LI.make_a(cfg, 0, pr, rank=rk, tag=f"slot{k}"),
                                LI.make_b(cfg, 0, pr, rank=rk, tag=f"slot{k}"))
                               for k, rk in enumerate(ranks)])
    hp = L.make_hp(cfg.beta1, cfg.beta2, cfg.eps, cfg.wd, cfg.plus_ratio)
    step = MultiLoraStep(lins, slot_ranks=ranks, slot_scales=scales, dtype=cfg.dtype, tokens=T,
                         seg_start=torch.tensor(r.seg_start, device="cuda"),
                         seg_slot=torch.tensor(r.seg_slot, device="cuda"),
                         max_norm=cfg.max_norm, hp=hp, n_streams=4)
    for lin in step.linears:
        for k, (A, B) in enumerate(host[lin.proj_id]["slots"]):
            lin.A[k].copy_(A)
            lin.B[k].copy_(B)
    step.prepare_weights()
    torch.cuda.synchronize()
    ready = [k for k in range(len(ranks)) if LI.slot_ready(r, k)]
    lrs = [cfg.lr] * len(ranks)

    def run():
        step.forward_backward(0)
        step.optimizer_step(ready, r.slot_gbs, lrs, r.slot_step, zero_grads=False)

    before = step.arena.params.clone()
    _replay_once(run)
    tok = O.token_slots(T, r.seg_start, r.seg_slot, len(ranks))
    rows = _sample_rows(T, 11, extra=list(r.seg_start[:40]))
    grads = {}
    for lin in step.linears:
        h = host[lin.proj_id]
        X, W, dY = h["X"], h["W"], h["dY"]
        Yr, Hr, dXr = [], [], []
        for t in rows.tolist():
            k = int(tok[t])
            if k >= 0:
                A, B = h["slots"][k]
                sc = scales[k]
            else:   # no adapter: the frozen product alone (B = 0)
                A, B = h["slots"][0]
                B, sc = torch.zeros_like(B), scales[0]
            f = O.lora_forward(X[t:t + 1], W, A, B, sc)
            b = O.lora_backward(X[t:t + 1], W, A, B, dY[t:t + 1], sc)
            Yr.append(f.Y[0])
            Hr.append(sc * f.H[0] if k >= 0 else 0.0 * f.H[0])
            dXr.append(b.dX[0])
        assert rel_err(_rows_of(lin.Y, rows), np.stack(Yr)) <= TOL_BF16
        Hg = _rows_of(lin.H, rows).detach().cpu().double().numpy()
        Hs = np.zeros_like(Hg)
        for i, t in enumerate(rows.tolist()):
            k = int(tok[t])
            if k >= 0:
                Hs[i, :ranks[k]] = Hr[i]
        assert rel_err(Hg, Hs) <= TOL_BF16
        assert rel_err(_rows_of(lin.dX, rows), np.stack(dXr)) <= TOL_BF16
        gk = {}
        for k in range(len(ranks)):
            sel = np.nonzero(tok == k)[0]
            A, B = h["slots"][k]
            if sel.size == 0:
                assert float(lin.gA[k].abs().max()) == 0.0
                gk[k] = (np.zeros(A.shape), np.zeros(B.shape))
                continue
            si = torch.from_numpy(sel)
            gA, gB = O.lora_adapter_grads(X[si], A, B, dY[si], scales[k])
            assert rel_err(lin.gA[k], gA) <= TOL_BF16, ("dA", k)
            assert rel_err(lin.gB[k], gB) <= TOL_BF16, ("dB", k)
            gk[k] = (gA, gB)
        grads[lin.proj_id] = gk
    st = step.status.cpu().numpy()
    for i, k in enumerate(ready):
        assert st[i] == O.STATUS_OK
        glist = []
        for lin in step.linears:
            glist += [grads[lin.proj_id][k][0], grads[lin.proj_id][k][1]]
        prep = O.grad_prepare([g.astype(np.float32) for g in glist], 1.0 / r.slot_gbs[k],
                              cfg.max_norm)
        hpo = O.AdamHP(lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps, wd=cfg.wd,
                       plus_ratio=cfg.plus_ratio, step=r.slot_step[k])
        for lin in step.linears:
            A0, B0 = host[lin.proj_id]["slots"][k]
            z = np.zeros
            A1, _, _ = O.adamw_update(A0, grads[lin.proj_id][k][0].astype(np.float32),
                                      z(A0.shape), z(A0.shape), O.KIND_A, prep.scale, hpo)
            B1, _, _ = O.adamw_update(B0, grads[lin.proj_id][k][1].astype(np.float32),
                                      z(B0.shape), z(B0.shape), O.KIND_B, prep.scale, hpo)
            assert rel_err(lin.A[k], A1) <= TOL_BF16_STEP
            assert rel_err(lin.B[k], B1) <= TOL_BF16_STEP
    for k in range(len(ranks)):
        if k not in ready:
            o, n = step.slot_off[k], step.slot_na[k] + step.slot_nb[k]
            assert torch.equal(step.arena.params[o:o + n], before[o:o + n])
