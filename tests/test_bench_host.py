"""Host-side logic of the benchmark: the flat input buffer behind the end-to-end copies, the
per-group byte model, and the chained workload's stability caps (CPU only)."""
import math

import pytest
import torch

import bench
import lora_inputs as LI


def test_pack_inputs_keeps_values_and_aliases():
    gen = torch.Generator().manual_seed(3)
    a = torch.randn(5, 7, generator=gen)
    b = torch.randn(3, 8, generator=gen).to(torch.bfloat16)
    c = torch.randn(11, generator=gen)
    ref = [a.clone(), b.clone(), c.clone()]
    holder = {"x": a}   # another reference to the same tensor object
    inputs = [a, b, a, c]
    flat, offs = bench.pack_inputs(inputs, "cpu")
    assert len(inputs) == 3            # the repeated tensor is packed once
    for t, r in zip(inputs, ref):
        assert torch.equal(t, r)
    assert holder["x"].data_ptr() == a.data_ptr()
    # every input is a view of the flat buffer at a 256-byte aligned offset
    base = flat.data_ptr()
    for t, o in zip(inputs, offs):
        assert o % 256 == 0
        assert t.data_ptr() == base + o
    # writing the flat buffer is writing the inputs
    flat.zero_()
    assert all(float(t.float().abs().sum()) == 0.0 for t in inputs)


def test_rebind_moves_inputs_to_a_second_buffer():
    a = torch.arange(12, dtype=torch.float32).reshape(3, 4)
    b = torch.arange(6, dtype=torch.float32)
    inputs = [a, b]
    flat, offs = bench.pack_inputs(inputs, "cpu")
    second = flat.clone()
    second.view(torch.uint8).zero_()
    bench.rebind_inputs(inputs, second, offs)
    assert a.data_ptr() == second.data_ptr() + offs[0]
    assert float(a.sum()) == 0.0 and float(b.sum()) == 0.0
    bench.rebind_inputs(inputs, flat, offs)
    assert torch.equal(a, torch.arange(12, dtype=torch.float32).reshape(3, 4))
    assert torch.equal(b, torch.arange(6, dtype=torch.float32))


def test_memory_counts_groups_count_shared_inputs_once():
    cfg = LI.CONFIGS["c4"]
    per_proj = bench.memory_counts(cfg, 1)
    grouped = bench.memory_counts(cfg, 1, bench.fused_groups(cfg))
    T = cfg.tokens
    # q/k/v and gate/up share X: the grouped shrink reads X 4 times instead of 7
    x_reads = lambda m: m["shrink"]
    saved = (3 - 1) * T * 4096 * 2 + (2 - 1) * T * 4096 * 2
    # the adapters and Hs columns are the same in both counts; only the X reads differ
    assert x_reads(per_proj) - x_reads(grouped) == saved
    # the reductions: dY' and the adapters are the same in both counts, and the grouped dA reads
    # X once per group (the o and down groups reduce dB and dA in one launch, class "red")
    red = lambda m: m["redB"] + m["redA"] + m.get("red", 0)
    assert red(per_proj) - red(grouped) == saved
    assert per_proj["adamw"] == grouped["adamw"]


def test_memory_counts_fused_classes_follow_the_launches():
    """bf16 fused groups of 2 to 4 projections time their dB and their shared dA as classes of
    their own; every other group (one projection here) reduces dB and dA in one launch ("red").
    fp32 groups run as one adapter of rank n r, so all of them count as "red"."""
    cfg = LI.CONFIGS["c4"]
    groups = bench.fused_groups(cfg)
    bf = bench.memory_counts(cfg, 1, groups)
    sizes = sorted(len(g) for g in groups)
    assert sizes == [1, 1, 2, 3]
    T, a, r = cfg.tokens, 2, cfg.rank
    # the o and down groups: dY' and X read once each, Hs and Gs, dB and dA read and written
    want_red = 0
    for g in groups:
        if len(g) == 1:
            p = cfg.projs[g[0]]
            want_red += (T * p.out_dim * a + T * r * 4 + 2 * r * p.out_dim * 4 +
                         T * p.in_dim * a + T * r * 4 + 2 * r * p.in_dim * 4)
    assert bf["red"] == want_red
    f32 = bench.memory_counts(LI.with_overrides(cfg, dtype="f32"), 1, groups)
    assert f32["redB"] == 0 and f32["redA"] == 0 and f32["red"] > 0
    # the unfused count has no merged class of its own: the bench derives it from dB + dA
    assert "red" not in bench.memory_counts(cfg, 1)


@pytest.mark.parametrize("name", ["c2", "c4"])
def test_chain_config_caps_the_adapter_gain(name):
    base = LI.CONFIGS[name]
    cfg = bench.chain_config(base)
    assert len(cfg.projs) == 1 and cfg.projs[0].in_dim == cfg.projs[0].out_dim
    s = cfg.alpha / (math.sqrt(cfg.rank) if cfg.rslora else cfg.rank)
    assert 2.0 * s * s * cfg.rank * cfg.b_var <= 0.01 * (1 + 1e-9)
    assert cfg.lr <= base.lr
    # Adam moves an entry by about lr per update: 50 replayed updates stay near B's scale
    assert 50 * cfg.lr * max(1.0, cfg.plus_ratio) <= 1.0 * math.sqrt(cfg.b_var) + 1e-12
