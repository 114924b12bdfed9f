"""E4M3 frozen base (LORA_BF16_FP8) through the C ABI against the CPU oracle.

The quantised codes and scales are integer/byte work decided in fp32 on both sides and must be
bit-exact; the frozen products and the adapter gradients are floating point and must meet the
bf16 bars (2e-2 per tensor), the frozen term compared with the oracle's product of the same
codes.
"""
import numpy as np
import pytest
import torch

import lora_inputs as LI
from oracle import lora_oracle as O
from tests.helpers import TOL_BF16, rel_err, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_adapter_adamw_gb300 import binding
    return binding


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("rows,K", [(7, 16), (33, 48), (64, 1536), (5, 14336)])
def test_quantize_rows_bit_exact(L, rows, K):
    rng = np.random.default_rng(rows * 131 + K)
    M = rng.standard_normal((rows, K)) * np.exp(rng.uniform(-12, 12, (rows, 1)))
    M[0] = 0.0                                     # an all-zero row: scale 1, codes 0
    if rows > 2:
        M[1, 3] = 1e30                             # one huge element
        M[2] *= 1e-30                              # tiny row (448 / amax still finite)
    Mb = _bf16(M)
    codes = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    L.lora_quantize_e4m3(Mb.cuda(), codes, scales)
    torch.cuda.synchronize()
    want_c, want_s = O.quantize_rows_e4m3(Mb.float().numpy())
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(scales.cpu().numpy(), want_s)


def test_prepared_weight_codes_bit_exact(L):
    out_d, in_d = 96, 160
    W = _bf16(np.random.default_rng(3).standard_normal((out_d, in_d)) / np.sqrt(in_d))
    d = L.make_desc(in_d, out_d, 8, 1.0, L.LORA_BF16_FP8, 0.0, 0, 0, 0, 0)
    nbytes = L.lora_prepared_weight_size(d)
    Wp = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    L.lora_prepare_weight(d, W.cuda(), Wp)
    torch.cuda.synchronize()
    buf = Wp.cpu().numpy()
    up = lambda b: (b + 15) // 16 * 16
    o1 = up(out_d * in_d)
    o2 = o1 + up(out_d * 4)
    o3 = o2 + up(in_d * out_d)
    W8 = buf[:out_d * in_d].reshape(out_d, in_d)
    sw = buf[o1:o1 + out_d * 4].view(np.float32)
    WT8 = buf[o2:o2 + in_d * out_d].reshape(in_d, out_d)
    swT = buf[o3:o3 + in_d * 4].view(np.float32)
    c, sc = O.quantize_rows_e4m3(W.float().numpy())
    ct, sct = O.quantize_rows_e4m3(W.float().numpy().T)
    assert np.array_equal(W8, c) and np.array_equal(sw, sc)
    assert np.array_equal(WT8, ct) and np.array_equal(swT, sct)
    assert nbytes == o3 + up(in_d * 4)


@pytest.mark.parametrize("T,in_d,out_d,r,p", [(384, 256, 384, 16, 0.0), (512, 512, 256, 8, 0.1),
                                              (256, 1024, 512, 64, 0.0)])
def test_fp8_forward_backward_matches_oracle(L, T, in_d, out_d, r, p):
    from bwd_adapter_adamw_gb300.step import Linear, LoraStep
    rng = np.random.default_rng(T + in_d + out_d)
    X = _bf16(rng.standard_normal((T, in_d)))
    W = _bf16(rng.standard_normal((out_d, in_d)) / np.sqrt(in_d))
    dY = _bf16(0.1 * rng.standard_normal((T, out_d)))
    A = rng.uniform(-np.sqrt(6 / in_d), np.sqrt(6 / in_d), (r, in_d)).astype(np.float32)
    B = (0.1 * rng.standard_normal((out_d, r))).astype(np.float32)
    s = O.lora_scale(2.0 * r, r, False)
    lin = Linear(0, 0, X.cuda(), W.cuda(), dY.cuda())
    step = LoraStep([lin], rank=r, scale=s, dtype="bf16fp8", tokens=T, chunks=1, dropout_p=p,
                    seed=5, max_norm=1.0, hp=L.make_hp(), device="cuda")
    lin.A.copy_(torch.from_numpy(A))
    lin.B.copy_(torch.from_numpy(B))
    step.prepare_weights()
    step.forward_backward(opt_step=2)
    torch.cuda.synchronize()
    keep = O.dropout_keep(p, 5, 2, 0, 0, 0, T, in_d) if p > 0 else None
    q = O.dropout_q(p) if p > 0 else 1.0
    Xf, Wf, dYf = X.float().numpy(), W.float().numpy(), dY.float().numpy()
    f = O.lora_forward_fp8(Xf, Wf, A, B, s, keep, q)
    b = O.lora_backward(Xf, Wf, A, B, dYf, s, keep, q)
    dX = O.lora_dx_fp8(dYf, Wf, A, b.G, s, keep, q)
    assert rel_err(lin.Y, f.Y) <= TOL_BF16
    assert rel_err(lin.dX, dX) <= TOL_BF16
    assert rel_err(lin.gA, b.dA) <= TOL_BF16
    assert rel_err(lin.gB, b.dB) <= TOL_BF16
    # the E4M3 frozen term really is the quantised one: the bf16 product is measurably off
    ref_bf16 = to64(Xf) @ to64(Wf).T
    fp8_only = O.lora_forward_fp8(Xf, Wf, A, np.zeros_like(B), s).Y
    assert rel_err(fp8_only, ref_bf16) > 1e-3


def test_fp8_rejects_unsupported_descriptors(L):
    d = L.make_desc(24, 64, 8, 1.0, L.LORA_BF16_FP8, 0.0, 0, 0, 0, 0)   # in % 16 != 0
    assert L.lora_prepared_weight_size(d) == 0
    d = L.make_desc(64, 64, 8, 1.0, L.LORA_BF16_FP8, 0.0, 0, 0, 0, 1)   # DoRA
    assert L.lora_prepared_weight_size(d) == 0
