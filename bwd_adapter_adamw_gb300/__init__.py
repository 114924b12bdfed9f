"""GB300-native LoRA-linear training step: forward, backward, two-pass clip and A-only AdamW.

The compute lives in liblora_gb300.so (hand-written sm_103a CUDA behind a C ABI, declared in
include/lora_gb300.h). `binding` marshals arguments to it; `step` sequences the calls for one
optimizer step. Importing `binding` fails loudly when the library has not been built.
"""
import importlib

__all__ = ["binding", "step", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
