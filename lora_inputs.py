"""Seeded synthetic inputs for the LoRA-linear training step.

This module is shared by the CUDA path (tests, bench) and by the CPU oracle.
It draws random numbers and fixes shapes; it holds none of the method's
arithmetic (no forward, backward, hash, clip or optimizer math).

Workload shapes follow the pages:
  * "4.3. Training Guide" (Juno) -- accumulation chunks, clip 1.0, lr 1e-4.
  * "8. LoRA Fundamentals" (Juno) -- TinyLlama wq/wv targets, rank 8,
    Kaiming-uniform A, B = 0 at the start, the seven "all" projections.
  * "Backward Bug Hunts and Vulkan Tiled GEMM" -- the rank-16 1536 -> 4096
    LoRA-B shape, 4096 context, dropout-free vs dropout runs.
  * "Multi-LoRA Training Example (fully-async)" -- per-slot rank/alpha,
    adapter_global_batch_size, Qwen3-4B-shaped base.

Every tensor gets its own seed, derived from the config seed and the tensor's
name, so that any single (layer, projection) can be regenerated on its own.
N(mu, v) below always means variance v.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

KIND_A, KIND_B, KIND_MAG = 0, 1, 2


@dataclass(frozen=True)
class Proj:
    name: str
    in_dim: int
    out_dim: int
    x_group: str  # projections with the same x_group read the same X (q/k/v, gate/up)


@dataclass(frozen=True)
class LoraConfig:
    name: str
    index: int
    projs: Tuple[Proj, ...]
    layers: int
    rank: int
    alpha: float
    rslora: bool
    dtype: str                 # "f32", "bf16", or "bf16fp8" (bf16 with an E4M3 frozen product)
    tokens: int                # tokens per optimizer step
    chunks: int                # accumulation chunks per step
    x_var: float = 1.0
    dy_var: float = 1.0
    dy_tail: int = 0           # 0: dY normal; k > 0: Student-t with k degrees of freedom, scaled by sqrt(dy_var)
    b_var: float = 0.01
    b_zero: bool = False
    dropout_p: float = 0.0
    dropout_seed: int = 0
    dora: bool = False
    max_norm: float = 1.0
    lr: float = 1e-4
    wd: float = 0.01
    plus_ratio: float = 1.0
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    sched: str = "constant"    # "constant" | "cosine"
    warmup: int = 0
    total: int = 0
    min_lr: float = 0.0
    opt_step: int = 0          # completed optimizer updates before this step
    adam_state: str = "zero"   # "zero" | "synthetic"
    # slot-keyed multi-LoRA
    slot_ranks: Optional[Tuple[int, ...]] = None
    seg_len_range: Tuple[int, int] = (64, 1024)
    gbs_choices: Tuple[int, ...] = (64, 128, 256)

    @property
    def seed(self) -> int:
        return 1234 + self.index

    @property
    def chunk_tokens(self) -> int:
        return self.tokens // self.chunks

    @property
    def multi(self) -> bool:
        return self.slot_ranks is not None


LLAMA_PROJS = (
    Proj("wq", 4096, 4096, "attn_in"), Proj("wk", 4096, 1024, "attn_in"),
    Proj("wv", 4096, 1024, "attn_in"), Proj("wo", 4096, 4096, "attn_out"),
    Proj("wgate", 4096, 14336, "mlp_in"), Proj("wup", 4096, 14336, "mlp_in"),
    Proj("wdown", 14336, 4096, "mlp_out"),
)
QWEN3_4B_PROJS = (
    Proj("wq", 2560, 4096, "attn_in"), Proj("wk", 2560, 1024, "attn_in"),
    Proj("wv", 2560, 1024, "attn_in"), Proj("wo", 4096, 2560, "attn_out"),
    Proj("wgate", 2560, 9728, "mlp_in"), Proj("wup", 2560, 9728, "mlp_in"),
    Proj("wdown", 9728, 2560, "mlp_out"),
)

CONFIGS: Dict[str, LoraConfig] = {
    # Tiny single LoRA linear, fp32, 2 chunks of 16 tokens.
    "c1": LoraConfig("c1", 1, (Proj("lin", 64, 64, "x"),), 1, rank=4, alpha=8, rslora=False,
                     dtype="f32", tokens=32, chunks=2, lr=1e-3, wd=0.01),
    # TinyLlama-1.1B-shaped wq + wv over 22 layers, fp32 frozen W, B = 0 at step 0.
    "c2": LoraConfig("c2", 2, (Proj("wq", 2048, 2048, "attn_in"), Proj("wv", 2048, 256, "attn_in")),
                     22, rank=8, alpha=16, rslora=False, dtype="f32", tokens=1024, chunks=4,
                     b_zero=True, lr=2e-4, wd=0.01),
    # Rank-16 1536 -> 4096 bf16 projection, dropout 0.1, LoRA+ 16, warmup-cosine at update 25.
    "c3": LoraConfig("c3", 3, (Proj("lin", 1536, 4096, "x"),), 1, rank=16, alpha=32, rslora=False,
                     dtype="bf16", tokens=4096, chunks=1, dy_var=1e-2, dropout_p=0.1,
                     dropout_seed=1234, plus_ratio=16.0, lr=1e-4, sched="cosine", warmup=10,
                     total=100, min_lr=1e-6, opt_step=25, adam_state="synthetic"),
    # Llama-style layer, all seven projections, 32 layers, rank 64 rsLoRA, 8 chunks of 1024.
    "c4": LoraConfig("c4", 4, LLAMA_PROJS, 32, rank=64, alpha=128, rslora=True, dtype="bf16",
                     tokens=8192, chunks=8, dy_var=1e-2),
    "c4dora": LoraConfig("c4dora", 4, LLAMA_PROJS, 32, rank=64, alpha=128, rslora=True,
                         dtype="bf16", tokens=8192, chunks=8, dy_var=1e-2, dora=True),
    # c4's workload (same seeded inputs) with the frozen products on E4M3 tensor cores.
    "c4fp8": LoraConfig("c4fp8", 4, LLAMA_PROJS, 32, rank=64, alpha=128, rslora=True,
                        dtype="bf16fp8", tokens=8192, chunks=8, dy_var=1e-2),
    # Slot-keyed multi-LoRA on one Qwen3-4B-shaped layer, 8 slots.
    "c5": LoraConfig("c5", 5, QWEN3_4B_PROJS, 1, rank=64, alpha=128, rslora=False, dtype="bf16",
                     tokens=16384, chunks=1, dy_var=1e-2,
                     slot_ranks=(8, 16, 16, 32, 32, 64, 64, 64)),
}


def with_overrides(cfg: LoraConfig, **kw) -> LoraConfig:
    """A copy of cfg with some fields replaced (used for smaller parity cases)."""
    d = {f: getattr(cfg, f) for f in cfg.__dataclass_fields__}
    d.update(kw)
    return LoraConfig(**d)


# ----------------------------------------------------------------------------------------------
# seeding
# ----------------------------------------------------------------------------------------------
def tensor_seed(cfg_seed: int, *parts) -> int:
    """Stable 63-bit seed for one named tensor of one config."""
    key = "/".join(str(p) for p in (cfg_seed,) + tuple(parts)).encode()
    return int.from_bytes(hashlib.blake2b(key, digest_size=8).digest(), "little") >> 1


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, var, seed, device, dtype) -> torch.Tensor:
    g = _gen(seed, device)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if var != 1.0:
        t.mul_(math.sqrt(var))
    return t.to(dtype)


def _student_t(shape, dof: int, var, seed, device, dtype) -> torch.Tensor:
    """Student-t with `dof` degrees of freedom times sqrt(var): z / sqrt(chi2_dof / dof), the
    chi-square drawn as a sum of dof squared normals from the same seeded generator."""
    g = _gen(seed, device)
    z = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    chi = torch.zeros(tuple(shape), device=device, dtype=torch.float32)
    for _ in range(dof):
        u = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
        chi.add_(u * u)
    t = z / torch.sqrt(chi / dof)
    if var != 1.0:
        t.mul_(math.sqrt(var))
    return t.to(dtype)


def _uniform(shape, bound, seed, device) -> torch.Tensor:
    g = _gen(seed, device)
    t = torch.rand(tuple(shape), generator=g, device=device, dtype=torch.float32)
    return t.mul_(2.0 * bound).sub_(bound)


def act_dtype(cfg: LoraConfig) -> torch.dtype:
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


# ----------------------------------------------------------------------------------------------
# single-adapter tensors
# ----------------------------------------------------------------------------------------------
def make_x(cfg: LoraConfig, layer: int, proj: Proj, device="cpu", tokens: Optional[int] = None):
    """X [T, in]: N(0, x_var) in the activation dtype; shared by projections of one x_group."""
    T = cfg.tokens if tokens is None else tokens
    return _normal((T, proj.in_dim), cfg.x_var, tensor_seed(cfg.seed, layer, "X", proj.x_group),
                   device, act_dtype(cfg))


def make_w(cfg: LoraConfig, layer: int, proj: Proj, device="cpu"):
    """Frozen W [out, in]: N(0, 1/in) in the activation dtype (nn.Linear layout)."""
    return _normal((proj.out_dim, proj.in_dim), 1.0 / proj.in_dim,
                   tensor_seed(cfg.seed, layer, "W", proj.name), device, act_dtype(cfg))


def make_a(cfg: LoraConfig, layer: int, proj: Proj, rank: Optional[int] = None, tag="", device="cpu"):
    """A [r, in] fp32, Kaiming-uniform U(-sqrt(6/in), +sqrt(6/in))."""
    r = cfg.rank if rank is None else rank
    return _uniform((r, proj.in_dim), math.sqrt(6.0 / proj.in_dim),
                    tensor_seed(cfg.seed, layer, "A", proj.name, tag), device)


def make_b(cfg: LoraConfig, layer: int, proj: Proj, rank: Optional[int] = None, tag="", device="cpu"):
    """B [out, r] fp32: zeros when the config starts from a fresh adapter, else N(0, b_var)."""
    r = cfg.rank if rank is None else rank
    if cfg.b_zero:
        return torch.zeros((proj.out_dim, r), dtype=torch.float32, device=device)
    return _normal((proj.out_dim, r), cfg.b_var, tensor_seed(cfg.seed, layer, "B", proj.name, tag),
                   device, torch.float32)


def make_dy(cfg: LoraConfig, layer: int, proj: Proj, device="cpu", tokens: Optional[int] = None):
    """Upstream gradient dY [T, out]: N(0, dy_var) in the activation dtype (or, with dy_tail = k,
    a heavy-tailed Student-t with k degrees of freedom at the same scale)."""
    T = cfg.tokens if tokens is None else tokens
    seed = tensor_seed(cfg.seed, layer, "dY", proj.name)
    if cfg.dy_tail > 0:
        return _student_t((T, proj.out_dim), cfg.dy_tail, cfg.dy_var, seed, device, act_dtype(cfg))
    return _normal((T, proj.out_dim), cfg.dy_var, seed, device, act_dtype(cfg))


def make_adam_state(cfg: LoraConfig, n: int, tag: str, device="cpu"):
    """Adam moments (m, v) for n parameters: zeros, or a seeded well-conditioned mid-run state
    (m ~ N(0, 1e-6), v = 1e-6 * (0.5 + z^2))."""
    if cfg.adam_state == "zero":
        z = torch.zeros(n, dtype=torch.float32, device=device)
        return z, z.clone()
    m = _normal((n,), 1e-6, tensor_seed(cfg.seed, "adam_m", tag), device, torch.float32)
    z = _normal((n,), 1.0, tensor_seed(cfg.seed, "adam_v", tag), device, torch.float32)
    v = (z * z + 0.5) * 1e-6
    return m, v


def dora_magnitude_init(W: torch.Tensor) -> torch.Tensor:
    """Canonical DoRA starts the magnitude at the frozen row norm ||W_o||_2 (input preparation,
    computed once in double on the host before any step)."""
    return W.double().pow(2).sum(1).sqrt().float()


# ----------------------------------------------------------------------------------------------
# slot-keyed multi-LoRA routing inputs
# ----------------------------------------------------------------------------------------------
@dataclass
class MultiRouting:
    seg_start: np.ndarray   # int32 [n_seg + 1], seg_start[0] = 0, seg_start[-1] = T
    seg_slot: np.ndarray    # int32 [n_seg]
    slot_rank: List[int]
    slot_alpha: List[float]
    slot_gbs: List[int]
    slot_count_before: List[int]   # samples already accumulated before this batch
    slot_step: List[int]           # completed optimizer updates per slot

    @property
    def n_seg(self) -> int:
        return len(self.seg_slot)

    def seg_count(self, slot: int) -> int:
        return int(np.sum(self.seg_slot == slot))


def make_routing(cfg: LoraConfig, tokens: Optional[int] = None) -> MultiRouting:
    """Segments of uniform-random length in seg_len_range until the sum reaches T (the last one is
    truncated), each tagged with a uniform-random slot. alpha_s = r_s for even slots, 2 r_s for odd.
    adapter_global_batch_size per slot from gbs_choices; one segment is one sample of weight 1.
    Counts are set so that even slots fill exactly on this batch and odd slots do not."""
    assert cfg.slot_ranks is not None
    T = cfg.tokens if tokens is None else tokens
    rng = np.random.Generator(np.random.PCG64(tensor_seed(cfg.seed, "routing", T)))
    lo, hi = cfg.seg_len_range
    starts = [0]
    while starts[-1] < T:
        starts.append(min(T, starts[-1] + int(rng.integers(lo, hi + 1))))
    n_slots = len(cfg.slot_ranks)
    seg_slot = rng.integers(0, n_slots, size=len(starts) - 1).astype(np.int32)
    ranks = list(cfg.slot_ranks)
    alphas = [float(r if s % 2 == 0 else 2 * r) for s, r in enumerate(ranks)]
    gbs = [int(x) for x in rng.choice(np.array(cfg.gbs_choices), size=n_slots)]
    steps = [int(x) for x in rng.permutation(np.arange(3, 3 + 5 * n_slots, 5))[:n_slots]]
    count_before = []
    for s in range(n_slots):
        n_here = int(np.sum(seg_slot == s))
        if s % 2 == 0:
            count_before.append(gbs[s] - n_here)
        else:
            count_before.append(max(0, gbs[s] - n_here - 1 - int(rng.integers(0, 8))))
    return MultiRouting(np.asarray(starts, dtype=np.int32), seg_slot, ranks, alphas, gbs,
                        count_before, steps)


def slot_ready(routing: MultiRouting, slot: int) -> bool:
    """A slot steps exactly when its adapter batch is full after this batch."""
    return routing.slot_count_before[slot] + routing.seg_count(slot) >= routing.slot_gbs[slot]


def tensor_nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()
