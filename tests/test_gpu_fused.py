"""Fused projections through the C ABI against the CPU oracle ("LoRA Training and Serving",
--lora-type: one frozen product over the stacked q/k/v or gate/up weights, one adapter per
projection, the input gradient summed over the projections). bf16 bars: 2e-2 per tensor; fp32
1e-5."""
import numpy as np
import pytest
import torch

from oracle import lora_oracle as O
from tests.helpers import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_adapter_adamw_gb300 import binding
    return binding


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("T,in_d,outs,r,p", [(384, 512, (512, 256, 256), 16, 0.0),
                                             (256, 256, (768, 768), 64, 0.1),
                                             (640, 768, (256,), 8, 0.0),
                                             # one shrink over the group's adapters side by side:
                                             # 3 x 64 and 4 x 64 columns (two MMAs per K-step)
                                             (520, 512, (512, 256, 256), 64, 0.1),
                                             (300, 256, (256, 256, 256, 256), 64, 0.0),
                                             # five projections: no group dA, ten reduction
                                             # jobs over three shared launches
                                             (264, 256, (256, 256, 512, 256, 256), 16, 0.1)])
def test_fused_projections_match_oracle(L, T, in_d, outs, r, p):
    from bwd_adapter_adamw_gb300.step import FusedGroup, FusedLoraStep
    rng = np.random.default_rng(T + in_d + sum(outs) + r)
    X = _bf16(rng.standard_normal((T, in_d)))
    Ws = [_bf16(rng.standard_normal((o, in_d)) / np.sqrt(in_d)) for o in outs]
    dYs = [_bf16(0.1 * rng.standard_normal((T, o))) for o in outs]
    As = [rng.uniform(-np.sqrt(6 / in_d), np.sqrt(6 / in_d), (r, in_d)).astype(np.float32)
          for _ in outs]
    Bs = [(0.1 * rng.standard_normal((o, r))).astype(np.float32) for o in outs]
    s = O.lora_scale(2.0 * r, r, False)
    g = FusedGroup(3, 7, X.cuda(), torch.cat(Ws, 0).cuda(), torch.cat(dYs, 1).cuda(), tuple(outs))
    step = FusedLoraStep([g], rank=r, scale=s, dtype="bf16", tokens=T, chunks=1, dropout_p=p,
                         seed=11, device="cuda")
    for k in range(len(outs)):
        g.A[k].copy_(torch.from_numpy(As[k]))
        g.B[k].copy_(torch.from_numpy(Bs[k]))
    step.prepare_weights()
    step.forward_backward(opt_step=4)
    torch.cuda.synchronize()
    keep = O.dropout_keep(p, 11, 4, 0, 3, 7, T, in_d) if p > 0 else None
    q = O.dropout_q(p) if p > 0 else 1.0
    res = O.fused_forward_backward(X.float().numpy(), [W.float().numpy() for W in Ws], As, Bs,
                                   [d.float().numpy() for d in dYs], s, keep, q)
    assert rel_err(g.Y, res.Y) <= TOL_BF16
    assert rel_err(g.dX, res.dX) <= TOL_BF16
    assert rel_err(g.H, (s * q) * res.H) <= TOL_BF16
    for k, (dA, dB) in enumerate(res.grads):
        assert rel_err(g.gA[k], dA) <= TOL_BF16
        assert rel_err(g.gB[k], dB) <= TOL_BF16


@pytest.mark.parametrize("T,in_d,outs,r,p", [(300, 256, (256, 128), 8, 0.0),
                                             (1024, 512, (512, 256), 8, 0.1),
                                             (257, 384, (136, 64, 200), 16, 0.0)])
def test_fused_projections_f32_match_oracle(L, T, in_d, outs, r, p):
    """fp32: the group as one adapter of rank n r with a block-diagonal up-projection; every
    output within the fp32 bound."""
    from bwd_adapter_adamw_gb300.step import FusedGroup, FusedLoraStep
    rng = np.random.default_rng(7 * T + in_d + sum(outs) + r)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32))
    X = f32(rng.standard_normal((T, in_d)))
    Ws = [f32(rng.standard_normal((o, in_d)) / np.sqrt(in_d)) for o in outs]
    dYs = [f32(rng.standard_normal((T, o))) for o in outs]
    As = [rng.uniform(-np.sqrt(6 / in_d), np.sqrt(6 / in_d), (r, in_d)).astype(np.float32)
          for _ in outs]
    Bs = [(0.1 * rng.standard_normal((o, r))).astype(np.float32) for o in outs]
    s = O.lora_scale(2.0 * r, r, False)
    g = FusedGroup(2, 5, X.cuda(), torch.cat(Ws, 0).cuda(), torch.cat(dYs, 1).cuda(), tuple(outs))
    step = FusedLoraStep([g], rank=r, scale=s, dtype="f32", tokens=T, chunks=1, dropout_p=p,
                         seed=5, device="cuda")
    for k in range(len(outs)):
        g.A[k].copy_(torch.from_numpy(As[k]))
        g.B[k].copy_(torch.from_numpy(Bs[k]))
    step.prepare_weights()
    step.forward_backward(opt_step=3)
    torch.cuda.synchronize()
    keep = O.dropout_keep(p, 5, 3, 0, 2, 5, T, in_d) if p > 0 else None
    q = O.dropout_q(p) if p > 0 else 1.0
    res = O.fused_forward_backward(X.numpy(), [W.numpy() for W in Ws], As, Bs,
                                   [d.numpy() for d in dYs], s, keep, q)
    assert rel_err(g.Y, res.Y) <= TOL_F32
    assert rel_err(g.dX, res.dX) <= TOL_F32
    assert rel_err(g.H, (s * q) * res.H) <= TOL_F32
    for k, (dA, dB) in enumerate(res.grads):
        assert rel_err(g.gA[k], dA) <= TOL_F32
        assert rel_err(g.gB[k], dB) <= TOL_F32


def test_fused_rejects_unaligned_projection_widths(L):
    d = L.make_desc(256, 384, 8, 1.0, L.LORA_BF16)
    A = torch.zeros(8, 256, device="cuda")
    B1, B2 = torch.zeros(256, 8, device="cuda"), torch.zeros(128, 8, device="cuda")
    projs = L.make_projs([dict(A=A, B=B1, out=256), dict(A=A, B=B2, out=128)])
    assert L.lora_fused_workspace_size(d, 64, projs) == 0
    d = L.make_desc(256, 512, 8, 1.0, L.LORA_BF16)
    projs = L.make_projs([dict(A=A, B=B1, out=256), dict(A=A, B=B1, out=128)])   # sum != out
    assert L.lora_fused_workspace_size(d, 64, projs) == 0
