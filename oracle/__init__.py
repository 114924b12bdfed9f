"""CPU oracle (test infrastructure only).

A plain float64 restatement of the LoRA-linear training step, used by the tests, the smoke
check and the benchmark's CPU-baseline leg to check and time the CUDA path. It shares no code
with the CUDA path and the product path never imports it.
"""
