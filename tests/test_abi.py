"""The C-ABI library on the host: it builds, loads, exports every symbol include/lora_gb300.h
declares, and rejects bad arguments before launching anything (no GPU needed: every call here
returns during host-side validation or is a host-only helper)."""
import ctypes as C
import os
import re

import pytest

from oracle import lora_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora_gb300.h")


@pytest.fixture(scope="module")
def L():
    from bwd_adapter_adamw_gb300 import build
    build.build()
    from bwd_adapter_adamw_gb300 import binding
    return binding


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n.startswith(("lora_", "multi_lora_"))))


def test_header_symbols_are_exported(L):
    names = _declared()
    assert len(names) >= 16
    lib = C.CDLL(L.library_path())
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(L.EXPORTED) == names


def test_status_strings(L):
    for code in range(7):
        assert L.status_string(code)
    assert "non-finite" in L.status_string(L.LORA_ERR_NONFINITE)


def test_host_scale_and_schedule_match_oracle(L):
    for a, r, rs in [(8, 4, False), (16, 8, False), (128, 64, True), (32, 16, False), (7, 3, True)]:
        assert L.lora_scale(a, r, rs) == O.lora_scale(a, r, rs)
    for k in range(0, 120, 7):
        assert L.lora_lr_at(L.LORA_SCHED_WARMUP_COSINE, 1e-4, k, 10, 100, 1e-6) == pytest.approx(
            O.lr_at("cosine", 1e-4, k, 10, 100, 1e-6), rel=1e-14)
        assert L.lora_lr_at(L.LORA_SCHED_CONSTANT, 2e-4, k, 10, 100, 1e-6) == 2e-4


FAKE = 1 << 20   # an aligned non-null address; never dereferenced (validation fails first)


def _fwd(L, d, T=16, ws_bytes=1 << 30, **kw):
    args = dict(X=FAKE, W=FAKE, Wp=FAKE, A=FAKE, B=FAKE, dm=None, dn=None, Y=FAKE, H=FAKE, ws=FAKE)
    args.update(kw)
    return L.lora_forward(d, None, T, args["X"], args["W"], args["Wp"], args["A"], args["B"], args["dm"],
                          args["dn"], args["Y"], args["H"], args["ws"], ws_bytes, stream=0,
                          check=False)


def test_forward_argument_errors(L):
    ok = L.make_desc(64, 64, 4, 2.0, L.LORA_F32)
    assert _fwd(L, L.make_desc(64, 64, 0, 2.0, L.LORA_F32)) == L.LORA_ERR_INVALID
    assert _fwd(L, L.make_desc(64, 64, 68, 2.0, L.LORA_F32)) == L.LORA_ERR_UNSUPPORTED
    assert _fwd(L, L.make_desc(64, 64, 6, 2.0, L.LORA_F32)) == L.LORA_ERR_UNSUPPORTED
    assert _fwd(L, L.make_desc(60, 64, 4, 2.0, L.LORA_F32)) == L.LORA_ERR_ALIGN
    assert _fwd(L, L.make_desc(64, 64, 4, 2.0, 7)) == L.LORA_ERR_INVALID
    assert _fwd(L, L.make_desc(64, 64, 4, 2.0, L.LORA_F32, dropout_p=1.0)) == L.LORA_ERR_INVALID
    assert _fwd(L, L.make_desc(64, 64, 4, 2.0, L.LORA_F32, proj_id=70000)) == L.LORA_ERR_INVALID
    assert _fwd(L, ok, T=-1) == L.LORA_ERR_INVALID
    assert _fwd(L, ok, X=None) == L.LORA_ERR_INVALID
    assert _fwd(L, ok, Wp=None) == L.LORA_ERR_INVALID
    assert _fwd(L, ok, Wp=FAKE + 8) == L.LORA_ERR_ALIGN
    assert _fwd(L, ok, Y=FAKE + 4) == L.LORA_ERR_ALIGN
    assert _fwd(L, ok, ws_bytes=16) == L.LORA_ERR_WORKSPACE
    dora = L.make_desc(64, 64, 4, 2.0, L.LORA_F32, dora=True)
    assert _fwd(L, dora) == L.LORA_ERR_INVALID          # magnitudes missing
    # more chunks in one call than the key table holds
    c = L.make_ctx(0, 0, 1)
    st = L.lora_forward(ok, c, 65, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, FAKE,
                        1 << 30, stream=0, check=False)
    assert st == L.LORA_ERR_UNSUPPORTED
    c = L.make_ctx(0, 65535, 8)
    st = L.lora_forward(ok, c, 16, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, FAKE,
                        1 << 30, stream=0, check=False)
    assert st == L.LORA_ERR_INVALID


def test_fused_workspace_dtypes(L):
    """Fused projections: bf16 needs 256-wide projections; fp32 runs the group as one adapter of
    rank n_proj * rank, at most 64 (host-side checks only, no launch)."""
    import torch
    A = torch.zeros(8, 256)
    B1, B2 = torch.zeros(384, 8), torch.zeros(128, 8)
    projs = L.make_projs([dict(A=A, B=B1, out=384), dict(A=A, B=B2, out=128)])
    assert L.lora_fused_workspace_size(L.make_desc(256, 512, 8, 1.0, L.LORA_F32), 64, projs) > 0
    assert L.lora_fused_workspace_size(L.make_desc(256, 512, 8, 1.0, L.LORA_BF16), 64, projs) == 0
    A40 = torch.zeros(40, 256)
    B40 = torch.zeros(384, 40)
    projs = L.make_projs([dict(A=A40, B=B40, out=384), dict(A=A40, B=B40, out=128)])
    assert L.lora_fused_workspace_size(L.make_desc(256, 512, 40, 1.0, L.LORA_F32), 64, projs) == 0


def test_prepared_weight_size(L):
    assert L.lora_prepared_weight_size(L.make_desc(2048, 256, 8, 2.0, L.LORA_F32)) == 8 * 2048 * 256
    assert L.lora_prepared_weight_size(L.make_desc(1536, 4096, 16, 2.0, L.LORA_BF16)) == 2 * 1536 * 4096
    assert L.lora_prepared_weight_size(L.make_desc(1536, 4096, 0, 2.0, L.LORA_BF16)) == 0


def test_workspace_sizes(L):
    d = L.make_desc(1536, 4096, 16, 2.0, L.LORA_BF16, 0.1, 1234)
    n = L.lora_workspace_size(d, 4096)
    assert n > 4096 * 16 * 4
    assert L.lora_workspace_size(L.make_desc(1536, 4096, 0, 2.0, L.LORA_BF16), 4096) == 0
    assert L.lora_workspace_size(d, 8192) > n


def test_multi_argument_errors(L):
    d = L.make_desc(2560, 4096, 64, 0.0, L.LORA_BF16)
    slots = L.make_slots([dict(A=FAKE, B=FAKE, dA=FAKE, dB=FAKE, rank=8, scale=1.0),
                          dict(A=FAKE, B=FAKE, dA=FAKE, dB=FAKE, rank=64, scale=2.0)])
    assert L.multi_lora_workspace_size(d, 1024, 5, slots) > 0
    bad = L.make_slots([dict(A=FAKE, B=FAKE, dA=FAKE, dB=FAKE, rank=72, scale=1.0)])
    assert L.multi_lora_workspace_size(d, 1024, 5, bad) == 0
    st = L.multi_lora_forward(L.make_desc(2560, 4096, 64, 0.0, L.LORA_BF16, dora=True), None, 16,
                              FAKE, FAKE, FAKE, 1, FAKE, FAKE, slots, FAKE, FAKE, FAKE, 1 << 30,
                              stream=0, check=False)
    assert st == L.LORA_ERR_UNSUPPORTED
    st = L.multi_lora_forward(d, None, 16, FAKE, FAKE, FAKE, 1, None, FAKE, slots, FAKE, FAKE, FAKE,
                              1 << 30, stream=0, check=False)
    assert st == L.LORA_ERR_INVALID
    st = L.multi_lora_backward(d, None, 16, FAKE, FAKE, 1, FAKE, FAKE, slots, FAKE, FAKE, None, FAKE,
                               16, stream=0, check=False)
    assert st == L.LORA_ERR_WORKSPACE


def test_plan_argument_errors(L):
    """The routing plan's calls validate their arguments on the host, before any launch."""
    assert L.multi_lora_plan_size(16384, 30, 8) > 0
    assert L.multi_lora_plan_size(16384, 0, 8) == 0
    assert L.multi_lora_plan_size(16384, 30, 0) == 0
    assert L.multi_lora_plan_size(16384, 30, L.LORA_MAX_SLOTS + 1) == 0
    # more segments take more room; T = 0 still has a layout
    assert L.multi_lora_plan_size(16384, 300, 8) > L.multi_lora_plan_size(16384, 30, 8)
    assert L.multi_lora_plan_size(0, 1, 1) > 0
    size = L.multi_lora_plan_size(1024, 5, 2)
    assert L.multi_lora_plan_build(1024, 5, None, FAKE, 2, FAKE, size, stream=0,
                                   check=False) == L.LORA_ERR_INVALID
    assert L.multi_lora_plan_build(1024, 5, FAKE, FAKE, 2, None, size, stream=0,
                                   check=False) == L.LORA_ERR_INVALID
    assert L.multi_lora_plan_build(1024, 5, FAKE, FAKE, 2, FAKE + 8, size, stream=0,
                                   check=False) == L.LORA_ERR_ALIGN
    assert L.multi_lora_plan_build(1024, 5, FAKE, FAKE, 2, FAKE, size - 16, stream=0,
                                   check=False) == L.LORA_ERR_WORKSPACE
    assert L.multi_lora_plan_build(0, 5, FAKE, FAKE, 2, FAKE, size, stream=0,
                                   check=False) == L.LORA_OK   # no tokens: nothing to build
    d = L.make_desc(2560, 4096, 64, 0.0, L.LORA_BF16)
    slots = L.make_slots([dict(A=FAKE, B=FAKE, dA=FAKE, dB=FAKE, rank=8, scale=1.0),
                          dict(A=FAKE, B=FAKE, dA=FAKE, dB=FAKE, rank=64, scale=2.0)])
    st = L.multi_lora_forward_planned(d, None, 16, 0, FAKE, FAKE, FAKE, FAKE, slots, FAKE, FAKE,
                                      FAKE, 1 << 30, stream=0, check=False)
    assert st == L.LORA_ERR_INVALID   # a plan needs at least one segment
    st = L.multi_lora_forward_planned(d, None, 16, 1, None, FAKE, FAKE, FAKE, slots, FAKE, FAKE,
                                      FAKE, 1 << 30, stream=0, check=False)
    assert st == L.LORA_ERR_INVALID
    st = L.multi_lora_backward_planned(d, None, 16, 1, FAKE, FAKE, FAKE, slots, FAKE, FAKE, None,
                                       FAKE, 16, stream=0, check=False)
    assert st == L.LORA_ERR_WORKSPACE


def test_optimizer_argument_errors(L):
    g1 = L.make_groups([dict(offset=0, n_a=100, n_b=50, grad_scale=0.1, max_norm=1.0),
                        dict(offset=148, n_a=8, grad_scale=0.1, max_norm=1.0)])
    assert L.lora_grad_prepare(FAKE, g1, FAKE, FAKE, FAKE, 1 << 20, stream=0, check=False) == \
        L.LORA_ERR_INVALID   # overlapping groups
    g2 = L.make_groups([dict(offset=2, n_a=100, grad_scale=0.1)])
    assert L.lora_grad_prepare(FAKE, g2, FAKE, FAKE, FAKE, 1 << 20, stream=0, check=False) == \
        L.LORA_ERR_ALIGN
    g3 = L.make_groups([dict(offset=0, n_a=100, grad_scale=0.1)])
    assert L.lora_grad_prepare(FAKE, g3, FAKE, FAKE, FAKE, 8, stream=0, check=False) == \
        L.LORA_ERR_WORKSPACE
    g4 = L.make_groups([dict(offset=0, n_a=100, grad_scale=0.1, max_norm=-1.0)])
    assert L.lora_grad_prepare(FAKE, g4, FAKE, FAKE, FAKE, 1 << 20, stream=0, check=False) == \
        L.LORA_ERR_INVALID
    many = L.make_groups([dict(offset=4 * i, n_a=4, grad_scale=1.0) for i in range(65)])
    assert L.lora_grad_prepare(FAKE, many, FAKE, FAKE, FAKE, 1 << 20, stream=0, check=False) == \
        L.LORA_ERR_UNSUPPORTED
    hp = L.make_hp(beta1=1.0)
    assert L.lora_adamw_step(FAKE, FAKE, FAKE, FAKE, g3, hp, FAKE, FAKE, stream=0, check=False) == \
        L.LORA_ERR_INVALID
    assert L.lora_grad_prepare_workspace_size(g3) > 0


def test_fused_entries_check_arguments_before_launch(L):
    """Host-side argument checks of the fused entries (no launch happens on these paths)."""
    import torch
    A = torch.zeros(8, 256)
    B1, B2 = torch.zeros(384, 8), torch.zeros(128, 8)
    projs = L.make_projs([dict(A=A, B=B1, dA=A, dB=B1, out=384), dict(A=A, B=B2, dA=A, dB=B2, out=128)])
    d = L.make_desc(256, 512, 8, 1.0, L.LORA_F32)
    c = L.make_ctx(0, 0, 64)
    args = dict(X=FAKE, W=FAKE, Wp=FAKE, Y=FAKE, H=FAKE, ws=FAKE)

    def fwd(**kw):
        a = dict(args, **kw)
        return L.lora_fused_forward(d, c, 64, a["X"], a["W"], a["Wp"], projs, a["Y"], a["H"],
                                    a["ws"], ws_bytes=1 << 30, stream=0, check=False)

    assert fwd(Wp=None) == L.LORA_ERR_INVALID       # the fp32 forward reads the prepared weight
    assert fwd(X=None) == L.LORA_ERR_INVALID
    assert L.lora_fused_forward(d, c, 64, FAKE, FAKE, FAKE, projs, FAKE, FAKE, FAKE, ws_bytes=16,
                                stream=0, check=False) == L.LORA_ERR_WORKSPACE
    st = L.lora_fused_backward(d, c, 64, FAKE, None, projs, FAKE, FAKE, None, FAKE,
                               ws_bytes=1 << 30, stream=0, check=False)
    assert st == L.LORA_ERR_INVALID                 # W_prep missing
