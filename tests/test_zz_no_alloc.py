"""The allocation-free grad-prepare entry point, for callers that cannot allocate device memory
(another framework's allocator owns the device pool, no allocation is allowed after
initialisation, or a CUDA graph is being captured around the call). It must give the same
results as the workspace entry point, call after call, since all calls share one fixed device
array. This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process (the first call sets up the array's
device address)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_adapter_adamw_gb300 import binding
    return binding


def _groups(L, sizes, gammas, max_norms):
    out, off = [], 0
    for n, g, mx in zip(sizes, gammas, max_norms):
        out.append(dict(offset=off, n_a=n // 2, n_b=n - n // 2, grad_scale=g, max_norm=mx))
        off += (n + 3) // 4 * 4
    return L.make_groups(out), off


def test_noalloc_prepare_matches_workspace_prepare_twice(L):
    sizes = [1_000_003, 16384 * 3, 7, 0, 2_500_000]
    groups, total = _groups(L, sizes, [1 / 1024, 1 / 64, 1.0, 0.5, 1 / 8192], [1.0, 0.0, 1.0, 1.0, 1e9])
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    for call in range(2):
        grads = torch.randn(total, device="cuda", generator=gen) * (10.0 ** call)
        n = len(sizes)
        want_sn = torch.zeros(2 * n, dtype=torch.float64, device="cuda")
        want_st = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        ws = torch.empty(L.lora_grad_prepare_workspace_size(groups), dtype=torch.uint8, device="cuda")
        L.lora_grad_prepare(grads, groups, want_sn, want_st, ws)
        got_sn = torch.full((2 * n,), float("nan"), dtype=torch.float64, device="cuda")
        got_st = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        L.lora_grad_prepare_noalloc(grads, groups, got_sn, got_st)
        torch.cuda.synchronize()
        assert torch.equal(got_st, want_st)
        w, g = want_sn.cpu().numpy(), got_sn.cpu().numpy()
        assert np.all(np.abs(g - w) <= 1e-12 * np.abs(w)), (call, g, w)


def test_noalloc_prepare_nonfinite_and_size_limit(L):
    groups, total = _groups(L, [4096, 4096], [1.0, 1.0], [1.0, 1.0])
    grads = torch.ones(total, device="cuda")
    grads[5000] = float("nan")
    sn = torch.zeros(4, dtype=torch.float64, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    L.lora_grad_prepare_noalloc(grads, groups, sn, st)
    torch.cuda.synchronize()
    assert st.tolist() == [L.LORA_OK, L.LORA_ERR_NONFINITE]
    assert abs(sn[1].item() - 64.0) < 1e-12
    # beyond the fixed array: rejected on the host, nothing launched
    big = L.make_groups([dict(offset=0, n_a=16384 * 16384 + 1, grad_scale=1.0)])
    assert L.lora_grad_prepare_noalloc(1 << 20, big, 1 << 20, 1 << 20, stream=0, check=False) == \
        L.LORA_ERR_UNSUPPORTED
