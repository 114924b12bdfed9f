"""Chained stack of adapted linears (layer l's output is layer l + 1's input), processed one
accumulation chunk at a time, through the C ABI against the CPU oracle ("4.3. Training Guide",
Truncated BPTT and Gradient accumulation).

fp32 activations: within 1e-5 per tensor; bf16 activations (rounded to bf16 between layers on
both sides): within 2e-2. The post-step A/B must follow the oracle's clip and AdamW.
"""
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


def _bf16_round(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def _inputs(dims, r, T, seed, dtype):
    rng = np.random.default_rng(seed)
    Ws = [(rng.standard_normal((dims[l + 1], dims[l])) / np.sqrt(dims[l])).astype(np.float32)
          for l in range(len(dims) - 1)]
    As = [rng.uniform(-np.sqrt(6.0 / dims[l]), np.sqrt(6.0 / dims[l]), (r, dims[l])).astype(np.float32)
          for l in range(len(dims) - 1)]
    Bs = [(0.1 * rng.standard_normal((dims[l + 1], r))).astype(np.float32)
          for l in range(len(dims) - 1)]
    X0 = rng.standard_normal((T, dims[0])).astype(np.float32)
    dY = rng.standard_normal((T, dims[-1])).astype(np.float32)
    if dtype == "bf16":   # the activations and frozen weights live in bf16: both sides see these
        Ws = [_bf16_round(W).astype(np.float32) for W in Ws]
        X0 = _bf16_round(X0).astype(np.float32)
        dY = _bf16_round(dY).astype(np.float32)
    return Ws, As, Bs, X0, dY


@pytest.mark.parametrize("dtype,dims,r,T,chunks,p", [
    ("f32", (256, 384, 256, 256), 8, 256, 2, 0.0),
    ("bf16", (512, 768, 512), 16, 512, 2, 0.1),
    ("bf16", (256, 256, 256, 256, 256), 8, 384, 3, 0.0),
])
def test_chain_matches_oracle(L, dtype, dims, r, T, chunks, p):
    from bwd_adapter_adamw_gb300.step import ChainStep
    Ws, As, Bs, X0, dY = _inputs(dims, r, T, seed=len(dims) * 31 + r, dtype=dtype)
    s = O.lora_scale(2.0 * r, r, False)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    dev = "cuda"
    step = ChainStep([torch.from_numpy(W).to(dev, tdt) for W in Ws],
                     torch.from_numpy(X0).to(dev, tdt), torch.from_numpy(dY).to(dev, tdt),
                     layer_ids=list(range(len(Ws))), rank=r, scale=s, dtype=dtype, chunks=chunks,
                     dropout_p=p, seed=77, max_norm=1.0, hp=L.make_hp(weight_decay=0.01),
                     device=dev)
    for lin, A, B in zip(step.linears, As, Bs):
        lin.A.copy_(torch.from_numpy(A))
        lin.B.copy_(torch.from_numpy(B))
    step.prepare_weights()
    step.forward_backward(opt_step=3)
    torch.cuda.synchronize()
    ref = O.chained_forward_backward(X0, Ws, As, Bs, dY, s, chunks,
                                     round_act=_bf16_round if dtype == "bf16" else None, p=p,
                                     seed=77, opt_step=3, layer_ids=list(range(len(Ws))))
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert rel_err(step.linears[-1].Y, ref.Y) <= tol
    assert rel_err(step.linears[0].dX, ref.dX) <= tol
    for lin, (gA, gB) in zip(step.linears, ref.grads):
        assert rel_err(lin.gA, gA) <= tol
        assert rel_err(lin.gB, gB) <= tol
    # the optimizer step over the whole stack: one global clip, A-only decay
    grads = [lin.gA.clone() for lin in step.linears], [lin.gB.clone() for lin in step.linears]
    A0 = [lin.A.clone() for lin in step.linears]
    step.optimizer_step(lr=1e-3, step=0)
    torch.cuda.synchronize()
    flat = [g.cpu().numpy() for pair in zip(*grads) for g in pair]
    prep = O.grad_prepare(flat, 1.0 / T, 1.0)
    assert int(step.status.item()) == prep.status
    for lin, gA, a0 in zip(step.linears, grads[0], A0):
        z = np.zeros(a0.shape, np.float32)
        want, _, _ = O.adamw_update(a0.cpu().numpy(), gA.cpu().numpy(), z, z, O.KIND_A,
                                    prep.scale, O.AdamHP(lr=1e-3, wd=0.01, step=0))
        assert rel_err(lin.A, want) <= 1e-5


def test_chain_rejects_widths_that_do_not_chain(L):
    from bwd_adapter_adamw_gb300.step import ChainStep
    W1 = torch.zeros(64, 32, device="cuda")
    W2 = torch.zeros(16, 48, device="cuda")
    with pytest.raises(ValueError):
        ChainStep([W1, W2], torch.zeros(32, 32, device="cuda"), torch.zeros(32, 16, device="cuda"),
                  rank=4, scale=1.0, dtype="f32", chunks=1)
