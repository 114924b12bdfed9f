"""The bounded-wait path of the tensor-core frozen products, on a correct launch.

Every pipeline wait of the frozen-product kernel gives up after a bound, sets a bit in the
device error word and lets the kernel return, so that a stalled pipeline cannot hang the GPU and
the caller learns that the outputs are invalid. Here the bound is shortened (a test hook) to one
cycle, so that an ordinary launch's waits run out; nothing is broken on purpose. The kernel must
then report the timeout (lora_device_check returns LORA_ERR_TIMEOUT, lora_device_error shows the
bits), and with the default bound back the same call on the same context must match the oracle.
"""
import numpy as np
import pytest
import torch

import lora_inputs as LI
from oracle import lora_oracle as O
from tests.helpers import TOL_BF16, build_single, rel_err, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_adapter_adamw_gb300 import binding
    return binding


def test_short_wait_bound_reports_timeout_and_context_stays_usable(L):
    # one Llama-style wq projection (4096 -> 4096, rank 64, bf16), 1024 tokens: each output tile
    # accumulates 64 K-blocks, far longer than one cycle
    cfg = LI.with_overrides(LI.CONFIGS["c4"], tokens=1024, chunks=1)
    step, problems, state, s, _ = build_single(cfg, [0], [0], device="cuda")
    lin = step.linears[0]
    assert L.lora_device_error(reset=True) == 0
    assert L.lora_device_check() == L.LORA_OK
    try:
        L.lora_set_wait_limit(1)
        lin.Y.zero_()
        step.forward_backward(cfg.opt_step)
        status = L.lora_device_check()
    finally:
        L.lora_set_wait_limit(0)
    flags = L.lora_device_error(reset=True)
    assert status == L.LORA_ERR_TIMEOUT
    assert flags != 0 and (flags & ~0x7) == 0, hex(flags)
    # default bound again: the same call completes and matches the oracle
    step.arena.grads.zero_()
    step.forward_backward(cfg.opt_step)
    assert L.lora_device_check() == L.LORA_OK
    assert L.lora_device_error(reset=True) == 0
    pr = problems[(0, 0)]
    A, B = state[(0, 0)].A, state[(0, 0)].B
    ref = O.lora_forward(to64(pr["X"]), to64(pr["W"]), A, B, s)
    assert rel_err(lin.Y, ref.Y) <= TOL_BF16
