"""The fp32 frozen products run as three bf16 products of a two-term bf16 split of each operand
(hi = bf16(x), lo = bf16(x - hi); the product is hi*hi' + hi*lo' + lo*hi'). This checks, in
float64 on the CPU and independently of the CUDA path, that the arithmetic this reading rests on
holds: the split keeps 16 significant bits, and on the fp32 workloads' shapes and value
distributions the three-product form stays well inside the fp32 paths' 1e-5 relative bound
(max |diff| / max |ref|), leaving room for the tensor core's fp32 accumulation."""
import numpy as np
import pytest


def _bf16_rne(x):
    """Round float32 values to bf16 (nearest, ties to even), returned as float32."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _split(x):
    x = np.asarray(x, np.float32)
    hi = _bf16_rne(x)
    lo = _bf16_rne((x - hi).astype(np.float32))
    return hi.astype(np.float64), lo.astype(np.float64)


def test_two_term_split_keeps_sixteen_bits():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200000), rng.uniform(-1e3, 1e3, 200000),
                        rng.standard_normal(1000) * 1e-20]).astype(np.float32)
    hi, lo = _split(x)
    x64 = x.astype(np.float64)
    assert np.all(np.abs(x64 - hi - lo) <= 2.0 ** -16 * np.abs(x64))
    # hi alone is a bf16 rounding: within half a unit in its 8th bit
    assert np.all(np.abs(x64 - hi) <= 2.0 ** -8 * np.abs(x64))


@pytest.mark.parametrize("T,K,N", [(256, 2048, 512), (256, 2048, 256), (256, 256, 1024),
                                   (32, 64, 64)])
def test_three_product_form_within_fp32_bound(T, K, N):
    """Shapes of the fp32 workloads (TinyLlama wq / wv forward and dX, the tiny linear) at a
    reduced token count; X ~ N(0, 1), W ~ N(0, 1/K)."""
    rng = np.random.default_rng(T + K + N)
    X = rng.standard_normal((T, K)).astype(np.float32)
    W = (rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    xh, xl = _split(X)
    wh, wl = _split(W)
    three = xh @ wh.T + xh @ wl.T + xl @ wh.T
    err = np.max(np.abs(three - ref)) / np.max(np.abs(ref))
    assert err <= 6e-6, err
    # dropping the lo terms altogether (a plain bf16 product) is far outside the bound, so the
    # check above can fail
    plain = xh @ wh.T
    assert np.max(np.abs(plain - ref)) / np.max(np.abs(ref)) > 1e-4
