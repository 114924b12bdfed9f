"""Snapshot / restore / retirement of adapter state through the C ABI, against the CPU oracle
("4.3. Training Guide", Validation early stopping; "Multi-LoRA Training Example (fully-async)",
adapter retirement).

The calls only copy and zero, so their results must be bit-exact; the update after a restore
(update count restarted) must match the oracle's AdamW from the snapshot with zero moments.
"""
import numpy as np
import pytest
import torch

from oracle import lora_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_adapter_adamw_gb300 import binding
    return binding


# ragged groups with gaps between them: counts that are not multiples of 4 exercise the tails,
# and one group spans several CTAs (4096 elements each)
GROUPS = [dict(offset=4, n_a=37, n_b=22, grad_scale=1.0),
          dict(offset=100, n_a=5000, n_b=3003, n_mag=9, grad_scale=1.0),
          dict(offset=8200, n_a=16, n_b=0, grad_scale=1.0)]
N = 8300


def _ranges():
    return [(g["offset"], g.get("n_a", 0) + g.get("n_b", 0) + g.get("n_mag", 0)) for g in GROUPS]


def _arenas(seed):
    rng = np.random.default_rng(seed)
    p = rng.standard_normal(N).astype(np.float32)
    g = rng.standard_normal(N).astype(np.float32)
    m = (0.1 * rng.standard_normal(N)).astype(np.float32)
    v = (0.01 * np.abs(rng.standard_normal(N)) + 1e-4).astype(np.float32)
    return p, g, m, v


def _dev(*arrs):
    return [torch.from_numpy(a.copy()).cuda() for a in arrs]


def test_snapshot_copies_exactly_the_group_ranges(L):
    p, _, _, _ = _arenas(1)
    snap0 = np.full(N, -7.0, np.float32)
    dp, dsnap = _dev(p, snap0)
    L.lora_snapshot(dp, dsnap, L.make_groups(GROUPS))
    torch.cuda.synchronize()
    want = O.snapshot(p, snap0, _ranges())
    assert np.array_equal(dsnap.cpu().numpy(), want)


@pytest.mark.parametrize("zero_grads", [False, True])
def test_restore_matches_oracle_bit_for_bit(L, zero_grads):
    p, g, m, v = _arenas(2)
    snap = _arenas(3)[0]
    dp, dsnap, dg, dm, dv = _dev(p, snap, g, m, v)
    L.lora_restore(dp, dsnap, dg, dm, dv, L.make_groups(GROUPS), zero_grads=zero_grads)
    torch.cuda.synchronize()
    want = O.restore(p, snap, g, m, v, _ranges(), zero_grads)
    for got, ref in zip((dp, dg, dm, dv), want):
        assert np.array_equal(got.cpu().numpy(), ref)


@pytest.mark.parametrize("clear_params", [False, True])
def test_retire_matches_oracle_bit_for_bit(L, clear_params):
    p, g, m, v = _arenas(4)
    dp, dg, dm, dv = _dev(p, g, m, v)
    retired = [GROUPS[1]]
    L.lora_retire(dp, dg, dm, dv, L.make_groups(retired), clear_params=clear_params)
    torch.cuda.synchronize()
    want = O.retire(p, g, m, v, [(GROUPS[1]["offset"], 5000 + 3003 + 9)], clear_params)
    for got, ref in zip((dp, dg, dm, dv), want):
        assert np.array_equal(got.cpu().numpy(), ref)


def test_train_snapshot_train_restore_then_step(L):
    """Two AdamW updates after a snapshot, then restore: the next update (count restarted at 0)
    equals the oracle's first update from the snapshot with zero moments."""
    p, g, m, v = _arenas(5)
    dp, dg, dm, dv = _dev(p, g, m, v)
    dsnap = torch.zeros_like(dp)
    hp = L.make_hp(weight_decay=0.01, plus_ratio=4.0)
    hp_o = dict(wd=0.01, plus_ratio=4.0)
    sn = torch.tensor([1.0, 1.0] * len(GROUPS), dtype=torch.float64, device="cuda")
    st = torch.zeros(len(GROUPS), dtype=torch.int32, device="cuda")
    L.lora_snapshot(dp, dsnap, L.make_groups(GROUPS))
    for k in range(2):
        gs = [dict(gr, lr=1e-2, step=k) for gr in GROUPS]
        L.lora_adamw_step(dp, dg, dm, dv, L.make_groups(gs), hp, sn, st)
    torch.cuda.synchronize()
    assert not torch.equal(dp, torch.from_numpy(p).cuda())
    L.lora_restore(dp, dsnap, dg, dm, dv, L.make_groups(GROUPS), zero_grads=False)
    gs = [dict(gr, lr=1e-2, step=0) for gr in GROUPS]
    L.lora_adamw_step(dp, dg, dm, dv, L.make_groups(gs), hp, sn, st)
    torch.cuda.synchronize()
    got = dp.cpu().numpy()
    for gr in GROUPS:
        off, na, nb, nm = gr["offset"], gr.get("n_a", 0), gr.get("n_b", 0), gr.get("n_mag", 0)
        z = np.zeros(na + nb + nm, np.float32)
        for kind, a, b in ((O.KIND_A, off, off + na), (O.KIND_B, off + na, off + na + nb),
                           (O.KIND_MAG, off + na + nb, off + na + nb + nm)):
            if b == a:
                continue
            ref, _, _ = O.adamw_update(p[a:b], g[a:b], z[:b - a], z[:b - a], kind, 1.0,
                                       O.AdamHP(lr=1e-2, step=0, **hp_o))
            np.testing.assert_allclose(got[a:b], ref, rtol=1e-6, atol=1e-7)


def test_maintenance_rejects_bad_arguments(L):
    dp = torch.zeros(64, device="cuda")
    bad_offset = L.make_groups([dict(offset=2, n_a=8, grad_scale=1.0)])
    assert L.lora_snapshot(dp, dp, bad_offset, check=False) == L.LORA_ERR_ALIGN
    ok = L.make_groups([dict(offset=0, n_a=8, grad_scale=1.0)])
    assert L.lora_restore(dp, None, dp, dp, dp, ok, check=False) == L.LORA_ERR_INVALID
    assert L.lora_retire(None, dp, dp, dp, ok, clear_params=True, check=False) == L.LORA_ERR_INVALID
    assert L.lora_retire(None, dp, dp, dp, ok, clear_params=False, check=False) == L.LORA_OK
    torch.cuda.synchronize()


def test_step_snapshot_restore_through_the_orchestration(L):
    import lora_inputs as LI
    from tests.helpers import build_single
    cfg = LI.with_overrides(LI.CONFIGS["c3"], tokens=512)
    step, problems, state, s, hp_o = build_single(cfg, [0], [0])
    step.run(cfg.opt_step, hp_o.lr)
    snap = step.snapshot()
    params0 = step.arena.params.clone()
    for k in range(2):
        step.run(cfg.opt_step + 1 + k, hp_o.lr)
    torch.cuda.synchronize()
    assert not torch.equal(step.arena.params, params0)
    step.restore(snap)
    torch.cuda.synchronize()
    assert torch.equal(step.arena.params, params0)
    assert not step.arena.m.any() and not step.arena.v.any() and not step.arena.grads.any()


def test_multi_retire_clears_one_slot_and_leaves_the_others(L):
    import lora_inputs as LI
    from tests.test_gpu_parity import _build_multi
    cfg = LI.CONFIGS["c5"]
    step, host, r, scales = _build_multi(cfg, [1], 900)
    step.forward_backward(0)
    ready = list(range(step.n_slots))
    step.optimizer_step(ready, [64] * step.n_slots, [1e-3] * step.n_slots, [0] * step.n_slots,
                        zero_grads=False)
    torch.cuda.synchronize()
    before = [t.clone() for t in (step.arena.params, step.arena.grads, step.arena.m, step.arena.v)]
    k = 2
    step.retire([k], clear_params=True)
    torch.cuda.synchronize()
    a, b = step.slot_off[k], step.slot_off[k] + step.slot_na[k] + step.slot_nb[k]
    for t, t0 in zip((step.arena.params, step.arena.grads, step.arena.m, step.arena.v), before):
        assert not t[a:b].any()
        assert torch.equal(t[:a], t0[:a]) and torch.equal(t[b:], t0[b:])
