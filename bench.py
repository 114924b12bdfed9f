"""Benchmark: one optimizer step of LoRA-adapted linears (forward + backward over every
accumulation chunk, two-pass clip, A-only AdamW) through the C ABI on GB300.

Default workload: the Llama-style layer, all seven projections (wq, wk, wv, wo, wgate, wup,
wdown; hidden 4096, kv 1024, intermediate 14336) over 32 layers, bf16 frozen W, rank 64, alpha 128
(rsLoRA), T = 8192 tokens per step in 8 accumulation chunks, global clip 1.0. `--config
c2|c3|c4dora|c5|...` selects the other workloads. Inputs are seeded synthetic tensors.

Prints ONE JSON line (rank 0). `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import lora_inputs as LI  # noqa: E402

METRIC = "LoRA linear fwd+bwd+step tokens/s on 1 GB300; % of tensor/HBM roofline"
UNIT = "tokens/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", default="c4", choices=sorted(LI.CONFIGS))
    p.add_argument("--layers", type=int, default=0, help="override the layer count (0 = config's)")
    p.add_argument("--streams", type=int, default=4,
                   help="CUDA streams over the independent adapted linears of the step")
    p.add_argument("--chain", action="store_true",
                   help="stack the config's first square projection over its layers, each "
                        "layer's output feeding the next (one stream)")
    p.add_argument("--fused", action="store_true",
                   help="run projections that share an input (q/k/v, gate/up) as one fused "
                        "linear each")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--prof-class", type=int, default=0, help="kernel class to time (0 = auto)")
    p.add_argument("--oracle-single-thread", action="store_true", help=argparse.SUPPRESS)
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, world, device="cpu"):
    """Element-wise maximum of per-rank timings over all ranks (every rank gets the result)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_rate(world, steps, tokens, ms):
    """Tokens per second of the whole job: every rank processes `tokens` per step (weak scaling),
    and the job takes the slowest rank's time."""
    return world * steps * tokens / (ms / 1e3)


# --------------------------------------------------------------------------------- algorithmic counts
def counts(cfg: LI.LoraConfig, layers: int):
    """Per-step algorithmic flops/bytes: frozen = 2 T in out per product,
    fused LoRA terms = 2 T r out (forward) / 2 T r in (dX); optimizer = 32 B/param."""
    T, r = cfg.tokens, cfg.rank
    a = 4 if cfg.dtype == "f32" else 2
    fwd = sum(2 * T * p.in_dim * p.out_dim + 2 * T * r * p.out_dim for p in cfg.projs) * layers
    dx = sum(2 * T * p.in_dim * p.out_dim + 2 * T * r * p.in_dim for p in cfg.projs) * layers
    lowrank = sum(6 * T * r * (p.in_dim + p.out_dim) for p in cfg.projs) * layers
    params = sum(r * (p.in_dim + p.out_dim) for p in cfg.projs) * layers
    return dict(fwd_flops_per_launch=fwd / (len(cfg.projs) * layers),
                dx_flops_per_launch=dx / (len(cfg.projs) * layers),
                fwd_flops=fwd, dx_flops=dx, lowrank_flops=lowrank, params=params,
                opt_bytes=32 * params, act_bytes=a)


def memory_counts(cfg: LI.LoraConfig, layers: int, groups=None):
    """Algorithmic HBM bytes per step of the memory-bound kernel classes (each array the class
    must touch, once): shrink reads X and A and writes Hs (and, on the fp32 path, the bf16 split
    of X); G reads dY' and B and writes Gs (and the split of dY'); the dB / dA reductions read dY'
    or X and Hs or Gs and update dB / dA; grad-prepare reads 4 B and AdamW moves 32 B per
    parameter (p, g, m, v read; p, m, v written; g cleared). With `groups` (fused projections:
    lists of projection indices that read one input), a group's input and output gradient are
    counted once, with the group's adapters side by side. The bf16 fused backward times the dB of
    groups of 2 to 4 projections and their shared dA as classes of their own ("redB", "redA");
    every other fused group reduces dB and dA in one launch ("red")."""
    T = cfg.tokens
    a = 4 if cfg.dtype == "f32" else 2
    split = 4 if cfg.dtype == "f32" else 0   # bf16 hi + lo per element
    if cfg.multi:
        ranks = list(LI.make_routing(cfg).slot_rank)
        r_all, layers = sum(ranks), 1
        r_row = max(ranks)
    else:
        r_all = r_row = cfg.rank
    out = {"shrink": 0, "G": 0, "redB": 0, "redA": 0}
    if groups:
        out["red"] = 0
    for idx in (groups or [[k] for k in range(len(cfg.projs))]):
        i = cfg.projs[idx[0]].in_dim
        o = sum(cfg.projs[k].out_dim for k in idx)
        n = len(idx)   # adapters of the group: n r columns of Hs / G, n A's of [r, in]
        out["shrink"] += T * i * a + n * r_all * i * 4 + T * n * r_row * 4 + split * T * i
        out["G"] += T * o * a + r_all * o * 4 + T * n * r_row * 4 + split * T * o
        if cfg.dtype != "f32" and not cfg.multi:
            # the bf16 G product also writes the transposed bf16 split of Gs (for dA) and, as a
            # side task, reads the saved Hs and writes its transposed split (for dB), per adapter
            out["G"] += 3 * 4 * T * n * r_row
        red_b = T * o * a + T * n * r_row * 4 + 2 * r_all * o * 4
        red_a = T * i * a + T * n * r_row * 4 + 2 * n * r_all * i * 4
        if groups and not (cfg.dtype != "f32" and 2 <= n <= 4 and 2 * r_row <= 128):
            out["red"] += red_b + red_a
        else:
            out["redB"] += red_b
            out["redA"] += red_a
    out = {k: v * layers for k, v in out.items()}
    r_step = r_all
    if cfg.multi:   # only the slots whose adapter batch is full take a step
        rt = LI.make_routing(cfg)
        r_step = sum(rk for k, rk in enumerate(rt.slot_rank) if LI.slot_ready(rt, k))
    params = sum(r_step * (p.in_dim + p.out_dim) for p in cfg.projs) * layers
    out["prepare"] = 4 * params
    out["adamw"] = 32 * params
    return out


# DRAM bytes per launch of the dominant kernel class (dram__bytes_read.sum + dram__bytes_write.sum,
# one ncu capture, caches flushed by ncu), averaged over the class's launch shapes, keyed by
# (workload, kernel class); valid only while the kernel source still hashes to the recorded
# value. Captured with `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum` on
# `python bench.py --layers 1 --steps 2 --warmup 3 --no-cpu-baseline --streams 1`.
NCU_TRAFFIC = {
    ("c4", 1): {"source": "gemm_tc.cu", "sha256_16": "4819c92179bf6c02",
                "bytes": 384.9e6,
                "note": "one-layer capture (profiles/launch_list_c4_llama_bf16.md): the seven "
                        "forward launches move 152.9, 78.3, 78.3, 153.9, 546.1, 548.6 and "
                        "1136.2 MB (read + write); the wide and long shapes re-read operands "
                        "while compute-bound"},
    ("c2", 1): {"source": "gemm_tc_f32.cu", "sha256_16": "0cfe552134b8e004",
                "bytes": (25.32e6 + 10.58e6) / 2,
                "note": "wq fwd 25.32 MB, wv fwd (4-way split K) 10.58 MB read (the bf16 hi / lo "
                        "splits of X and W, once), ~0 written (outputs stay in L2)"},
}


def traffic_for(cfg_name, prof_class):
    ent = NCU_TRAFFIC.get((cfg_name, prof_class))
    if ent is None:
        return None, "no ncu capture for this workload"
    path = os.path.join(ROOT, "bwd_adapter_adamw_gb300", "csrc", ent["source"])
    try:
        with open(path, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None, "kernel source not found"
    if sha != ent["sha256_16"]:
        return None, "kernel changed since the ncu capture"
    return ent["bytes"], ent["note"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}, "fallback"


# --------------------------------------------------------------------------------- clocks sampler
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------------- workload
def pack_inputs(inputs, device):
    """Rebind every input tensor (same values) to a view of one flat device buffer, so that a
    step's whole input batch moves host -> device in one copy. Drops repeated tensors from
    `inputs` (in place) and returns the flat buffer and each tensor's byte offset in it."""
    import torch
    uniq = {id(t): t for t in inputs}
    inputs[:] = list(uniq.values())
    offs, total = [], 0
    for t in inputs:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    flat = torch.empty(total, dtype=torch.uint8, device=device)
    for t, o in zip(inputs, offs):
        nb = t.numel() * t.element_size()
        flat[o:o + nb].view(t.dtype).view(t.shape).copy_(t)
    rebind_inputs(inputs, flat, offs)
    return flat, offs


def rebind_inputs(inputs, flat, offs):
    """Point every input tensor at its slice of the flat buffer `flat` (pack_inputs' layout)."""
    for t, o in zip(inputs, offs):
        nb = t.numel() * t.element_size()
        v = flat[o:o + nb].view(t.dtype).view(t.shape)
        t.set_(v.untyped_storage(), v.storage_offset(), v.shape, v.stride())


def _scale(cfg, L):
    return L.lora_scale(cfg.alpha, cfg.rank, cfg.rslora)


def make_single(cfg, layers, streams, device):
    import torch
    from bwd_adapter_adamw_gb300 import binding as L
    from bwd_adapter_adamw_gb300.step import Linear, LoraStep
    linears, xs = [], {}
    for l in range(layers):
        for pi, pr in enumerate(cfg.projs):
            key = (l, pr.x_group)
            if key not in xs:
                xs[key] = LI.make_x(cfg, l, pr, device=device)
            linears.append(Linear(l, pi, xs[key], LI.make_w(cfg, l, pr, device=device),
                                  LI.make_dy(cfg, l, pr, device=device)))
    hp = L.make_hp(cfg.beta1, cfg.beta2, cfg.eps, cfg.wd, cfg.plus_ratio)
    step = LoraStep(linears, rank=cfg.rank, scale=_scale(cfg, L), dtype=cfg.dtype,
                    tokens=cfg.tokens, chunks=cfg.chunks, dropout_p=cfg.dropout_p,
                    seed=cfg.dropout_seed, dora=cfg.dora, max_norm=cfg.max_norm, hp=hp,
                    n_streams=streams, device=device)
    for lin in step.linears:
        pr = cfg.projs[lin.proj_id]
        lin.A.copy_(LI.make_a(cfg, lin.layer, pr, device=device))
        lin.B.copy_(LI.make_b(cfg, lin.layer, pr, device=device))
        if cfg.dora:
            lin.mag.copy_(LI.dora_magnitude_init(lin.W))
    m, v = LI.make_adam_state(cfg, step.arena.n, "all", device=device)
    step.arena.m.copy_(m)
    step.arena.v.copy_(v)
    step.prepare_weights()
    inputs = list(xs.values()) + [lin.dY for lin in step.linears]
    lr = L.lora_lr_at(1 if cfg.sched == "cosine" else 0, cfg.lr, cfg.opt_step, cfg.warmup,
                      cfg.total, cfg.min_lr)

    def run():
        step.run(cfg.opt_step, lr)

    return step, run, inputs, [step.scale_norm, step.status]


def chain_config(cfg):
    """The chained workload of a config: its first square projection stacked over the config's
    layers (layer l's output is layer l + 1's input), one accumulation chunk per backward
    window."""
    sq = [pr for pr in cfg.projs if pr.in_dim == pr.out_dim]
    if not sq or cfg.multi or cfg.dora:
        raise SystemExit(f"--chain needs a single-adapter config with a square projection "
                         f"({cfg.name} has none)")
    # Stacked, each layer's adapter term multiplies the activations' variance by about
    # 1 + 2 s^2 r b_var (H = Xd A^T has variance 2 per element under the Kaiming-uniform A); with
    # the configs' independent-layer b_var (c4: 2 * 16^2 * 64 * 0.01 = 328) 32 layers overflow and
    # every step is rejected as non-finite. The chained workload caps that factor at 1.01, and
    # its learning rate so that the bench's few dozen replayed updates of the same batch (Adam
    # moves each entry by about lr per update) leave B near that scale. The step's cost does not
    # depend on either.
    s = 1.0 * cfg.alpha / (math.sqrt(cfg.rank) if cfg.rslora else cfg.rank)
    b_var = min(cfg.b_var, 0.01 / (2.0 * s * s * cfg.rank))
    lr = min(cfg.lr, 0.02 * math.sqrt(b_var) / max(1.0, cfg.plus_ratio))
    return LI.with_overrides(cfg, projs=(sq[0],), b_var=b_var, lr=lr)


def make_chain(cfg, layers, device):
    from bwd_adapter_adamw_gb300 import binding as L
    from bwd_adapter_adamw_gb300.step import ChainStep
    pr = cfg.projs[0]
    X0 = LI.make_x(cfg, 0, pr, device=device)
    dY = LI.make_dy(cfg, layers - 1, pr, device=device)
    Ws = [LI.make_w(cfg, l, pr, device=device) for l in range(layers)]
    hp = L.make_hp(cfg.beta1, cfg.beta2, cfg.eps, cfg.wd, cfg.plus_ratio)
    step = ChainStep(Ws, X0, dY, rank=cfg.rank, scale=_scale(cfg, L), dtype=cfg.dtype,
                     chunks=cfg.chunks, dropout_p=cfg.dropout_p, seed=cfg.dropout_seed,
                     max_norm=cfg.max_norm, hp=hp, device=device)
    for lin in step.linears:
        lin.A.copy_(LI.make_a(cfg, lin.layer, pr, device=device))
        lin.B.copy_(LI.make_b(cfg, lin.layer, pr, device=device))
    m, v = LI.make_adam_state(cfg, step.arena.n, "all", device=device)
    step.arena.m.copy_(m)
    step.arena.v.copy_(v)
    step.prepare_weights()
    lr = L.lora_lr_at(1 if cfg.sched == "cosine" else 0, cfg.lr, cfg.opt_step, cfg.warmup,
                      cfg.total, cfg.min_lr)

    def run():
        step.run(cfg.opt_step, lr)

    return step, run, [X0, dY], [step.scale_norm, step.status]


def fused_groups(cfg):
    """The config's projections grouped by the input they read (q/k/v, gate/up), in order."""
    groups = []
    for pi, pr in enumerate(cfg.projs):
        if groups and cfg.projs[groups[-1][0]].x_group == pr.x_group:
            groups[-1].append(pi)
        else:
            groups.append([pi])
    return groups


def make_fused(cfg, layers, streams, device):
    import torch
    from bwd_adapter_adamw_gb300 import binding as L
    from bwd_adapter_adamw_gb300.step import FusedGroup, FusedLoraStep
    if cfg.multi or cfg.dora or cfg.dtype not in ("bf16", "f32"):
        raise SystemExit(f"--fused needs a single-adapter bf16 or fp32 config without DoRA "
                         f"({cfg.name})")
    groups, xs = [], []
    for l in range(layers):
        for idx in fused_groups(cfg):
            prs = [cfg.projs[i] for i in idx]
            X = LI.make_x(cfg, l, prs[0], device=device)
            W = torch.cat([LI.make_w(cfg, l, pr, device=device) for pr in prs], 0)
            dY = torch.cat([LI.make_dy(cfg, l, pr, device=device) for pr in prs], 1)
            groups.append(FusedGroup(l, idx[0], X, W, dY, tuple(pr.out_dim for pr in prs)))
            xs.append(X)
    hp = L.make_hp(cfg.beta1, cfg.beta2, cfg.eps, cfg.wd, cfg.plus_ratio)
    step = FusedLoraStep(groups, rank=cfg.rank, scale=_scale(cfg, L), dtype=cfg.dtype,
                         tokens=cfg.tokens, chunks=cfg.chunks, dropout_p=cfg.dropout_p,
                         seed=cfg.dropout_seed, max_norm=cfg.max_norm, hp=hp, n_streams=streams,
                         device=device)
    members = {idx[0]: idx for idx in fused_groups(cfg)}   # group key: its first projection
    for g in step.fgroups:
        for k, i in enumerate(members[g.proj_id]):
            g.A[k].copy_(LI.make_a(cfg, g.layer, cfg.projs[i], device=device))
            g.B[k].copy_(LI.make_b(cfg, g.layer, cfg.projs[i], device=device))
    m, v = LI.make_adam_state(cfg, step.arena.n, "all", device=device)
    step.arena.m.copy_(m)
    step.arena.v.copy_(v)
    step.prepare_weights()
    lr = L.lora_lr_at(1 if cfg.sched == "cosine" else 0, cfg.lr, cfg.opt_step, cfg.warmup,
                      cfg.total, cfg.min_lr)

    def run():
        step.run(cfg.opt_step, lr)

    return step, run, xs + [g.dY for g in step.fgroups], [step.scale_norm, step.status]


def make_multi(cfg, streams, device):
    import torch
    from bwd_adapter_adamw_gb300 import binding as L
    from bwd_adapter_adamw_gb300.step import MultiLinear, MultiLoraStep
    r = LI.make_routing(cfg)
    xs, lins = {}, []
    for pi, pr in enumerate(cfg.projs):
        if pr.x_group not in xs:
            xs[pr.x_group] = LI.make_x(cfg, 0, pr, device=device)
        lins.append(MultiLinear(pi, xs[pr.x_group], LI.make_w(cfg, 0, pr, device=device),
                                LI.make_dy(cfg, 0, pr, device=device)))
    scales = [L.lora_scale(a, rk, cfg.rslora) for a, rk in zip(r.slot_alpha, r.slot_rank)]
    hp = L.make_hp(cfg.beta1, cfg.beta2, cfg.eps, cfg.wd, cfg.plus_ratio)
    step = MultiLoraStep(lins, slot_ranks=r.slot_rank, slot_scales=scales, dtype=cfg.dtype,
                         tokens=cfg.tokens, seg_start=torch.tensor(r.seg_start, device=device),
                         seg_slot=torch.tensor(r.seg_slot, device=device), max_norm=cfg.max_norm,
                         hp=hp, n_streams=streams, device=device)
    for lin in step.linears:
        pr = cfg.projs[lin.proj_id]
        for k, rk in enumerate(r.slot_rank):
            lin.A[k].copy_(LI.make_a(cfg, 0, pr, rank=rk, tag=f"slot{k}", device=device))
            lin.B[k].copy_(LI.make_b(cfg, 0, pr, rank=rk, tag=f"slot{k}", device=device))
    step.prepare_weights()
    ready = [k for k in range(len(r.slot_rank)) if LI.slot_ready(r, k)]
    lrs = [cfg.lr] * len(r.slot_rank)

    def run():
        step.forward_backward(0)
        step.optimizer_step(ready, r.slot_gbs, lrs, r.slot_step)

    inputs = list(xs.values()) + [lin.dY for lin in step.linears]
    return step, run, inputs, [step.scale_norm, step.status]


# --------------------------------------------------------------------------------- CPU baseline
def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def _oracle_problem(cfg, layer, tokens):
    """One layer's problems and adapter state for the oracle (inputs from lora_inputs)."""
    import numpy as np
    from oracle import lora_oracle as O
    problems, state = {}, {}
    for pi, pr in enumerate(cfg.projs):
        A = LI.make_a(cfg, layer, pr)
        B = LI.make_b(cfg, layer, pr)
        problems[pi] = dict(X=LI.make_x(cfg, layer, pr, tokens=tokens),
                            W=LI.make_w(cfg, layer, pr),
                            dY=LI.make_dy(cfg, layer, pr, tokens=tokens), layer=layer, proj=pi)
        z = lambda a: np.zeros(tuple(a.shape), np.float32)
        st = O.AdapterState(A.numpy(), B.numpy(), z(A), z(A), z(B), z(B))
        if cfg.dora:
            st.mag = LI.dora_magnitude_init(problems[pi]["W"]).numpy()
            st.mM, st.vM = np.zeros_like(st.mag), np.zeros_like(st.mag)
        state[pi] = st
    return problems, state


def _oracle_step_seconds(cfg, problems, state, chunks):
    from oracle import lora_oracle as O
    s = O.lora_scale(cfg.alpha, cfg.rank, cfg.rslora)
    hp = O.AdamHP(lr=O.lr_at(cfg.sched, cfg.lr, cfg.opt_step, cfg.warmup, cfg.total, cfg.min_lr),
                  beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps, wd=cfg.wd,
                  plus_ratio=cfg.plus_ratio, step=cfg.opt_step)
    t0 = time.perf_counter()
    O.run_single_step(problems, state, s=s, chunks=chunks, p=cfg.dropout_p,
                      seed=cfg.dropout_seed, opt_step=cfg.opt_step, max_norm=cfg.max_norm,
                      hp=hp, dora=cfg.dora, keep_outputs=False)
    return time.perf_counter() - t0


def oracle_single_thread():
    """Single-thread oracle times of two whole workloads: the tiny fp32 linear (64 x 64, T 32 in
    two chunks) and one rank-16 projection (1536 -> 4096, T 4096, dropout 0.1). Run in a child
    process whose BLAS is limited to one thread before numpy loads."""
    out = {}
    for name in ("c1", "c3"):
        cfg = LI.CONFIGS[name]
        problems, state = _oracle_problem(cfg, 0, cfg.tokens)
        sec = _oracle_step_seconds(cfg, problems, state, cfg.chunks)
        out[name] = {"seconds": sec, "tokens_per_s": cfg.tokens / sec,
                     "workload": f"{name}: 1 layer x {cfg.projs[0].in_dim}->{cfg.projs[0].out_dim}, "
                                 f"T={cfg.tokens}, whole step"}
    return out


def run_single_thread_probe():
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
              "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-single-thread"],
                           capture_output=True, text=True, timeout=300, env=env)
        return json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else None
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None


def cpu_baseline(cfg: LI.LoraConfig, layers: int, budget_s: float = 20.0, single_thread=True):
    """The oracle, as it stands, on a bounded sample of the workload: whole steps over a subset of
    the layers (all chunks, all projections; large workloads also a token sample). `value` is the
    sample's time scaled to the whole step (per layer x layers, x tokens / sampled tokens), and
    the measured part and the scale factor are reported beside it."""
    done_layers, elapsed = 0, 0.0
    tokens = cfg.tokens
    if cfg.multi or cfg.tokens * max(p.in_dim for p in cfg.projs) > 8192 * 4096:
        tokens = 512   # large workloads: a token sample, scaled by tokens
    t_all = time.perf_counter()
    while done_layers < layers:
        problems, state = _oracle_problem(cfg, done_layers, tokens)
        chunks = cfg.chunks if tokens == cfg.tokens else 1
        elapsed += _oracle_step_seconds(cfg, problems, state, chunks)
        done_layers += 1
        if time.perf_counter() - t_all > budget_s:
            break
    scale = (layers / done_layers) * (cfg.tokens / tokens)
    per_step = elapsed * scale
    cores = len(os.sched_getaffinity(0))
    out = {"value": cfg.tokens / per_step, "unit": UNIT, "cores": cores, "kind": "oracle",
           "cpu_model": cpu_model(),
           "sample": (f"{done_layers} of {layers} layers x {len(cfg.projs)} projections, "
                      f"{tokens} of {cfg.tokens} tokens, float64 numpy oracle (BLAS threads "
                      f"= all {cores} cores), whole step per layer"),
           "measured": {"seconds": elapsed, "layers": done_layers, "tokens": tokens,
                        "tokens_per_s": done_layers * tokens / elapsed / layers
                        if elapsed > 0 else None},
           "extrapolation": {"factor": scale,
                             "rule": f"x {layers}/{done_layers} layers x {cfg.tokens}/{tokens} "
                                     "tokens (the oracle's cost is linear in both)",
                             "per_step_s": per_step},
           "seconds": elapsed}
    if single_thread:
        out["single_thread"] = run_single_thread_probe()
    return out


# --------------------------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cfg = LI.CONFIGS[args.config]
    if args.chain:
        cfg = chain_config(cfg)   # same per-layer arithmetic; the chain only orders the layers
    layers = args.layers or cfg.layers
    budget = 240.0 / max(1, args.steps + args.warmup)
    vals = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(cfg, layers, budget_s=min(budget, 20.0), single_thread=False)
        if i >= args.warmup:
            vals.append(r)
    value = statistics.median(v["value"] for v in vals)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * cfg.tokens / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_name(cfg, layers, args.chain),
                       "tokens_per_step": cfg.tokens},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": vals[0]["cores"],
                             "kind": "oracle", "sample": vals[0]["sample"],
                             "cpu_model": vals[0]["cpu_model"],
                             "extrapolation": vals[0]["extrapolation"]["rule"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def step_stats(per_step):
    """Median, 10th and 90th percentile of the timed steps' durations (ms), this rank's clock."""
    xs = sorted(per_step)
    if not xs:
        return None
    q = statistics.quantiles(xs, n=10, method="inclusive") if len(xs) > 1 else [xs[0]] * 9
    return {"median": statistics.median(xs), "p10": q[0], "p90": q[8], "n": len(xs)}


def workload_name(cfg, layers, chained=False, fused=False):
    projs = "+".join(f"{p.name}:{p.in_dim}->{p.out_dim}" for p in cfg.projs)
    extra = []
    if cfg.multi:
        extra.append(f"slots ranks {list(cfg.slot_ranks)}")
    else:
        extra.append(f"rank {cfg.rank} alpha {cfg.alpha:g}{' rsLoRA' if cfg.rslora else ''}")
    if cfg.dora:
        extra.append("DoRA")
    if cfg.dropout_p:
        extra.append(f"dropout {cfg.dropout_p}")
    if chained:
        extra.append("chained: layer l's output is layer l+1's input")
    if fused:
        names = ["+".join(cfg.projs[i].name for i in g) for g in fused_groups(cfg)]
        extra.append("fused projections " + ", ".join(names))
    return (f"{cfg.name}: {layers} layers x [{projs}], {cfg.dtype} frozen W, "
            f"{', '.join(extra)}, T={cfg.tokens} in {cfg.chunks} chunks")


# --------------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import torch.distributed as dist
    from bwd_adapter_adamw_gb300 import binding as L

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    cfg = LI.CONFIGS[args.config]
    layers = args.layers or cfg.layers
    if args.chain:
        cfg = chain_config(cfg)
        step, run, inputs, results = make_chain(cfg, layers, device)
    elif args.fused:
        step, run, inputs, results = make_fused(cfg, layers, args.streams, device)
    elif cfg.multi:
        step, run, inputs, results = make_multi(cfg, args.streams, device)
    else:
        step, run, inputs, results = make_single(cfg, layers, args.streams, device)
    flat_in, in_offs = pack_inputs(inputs, device)
    torch.cuda.synchronize()

    # launches per step (eager), then warm-up
    c0 = L.lora_launch_counter()
    run()
    torch.cuda.synchronize()
    launches_per_step = L.lora_launch_counter() - c0
    for _ in range(max(0, args.warmup - 1)):
        run()
    torch.cuda.synchronize()

    # dominant kernel: event brackets around every launch of its class inside the timed step
    prof_class = args.prof_class or L.LORA_PROF_FROZEN_FWD
    n_prof = (layers if not cfg.multi else 1) * len(cfg.projs)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_prof)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(n_prof)]
    for e in starts + stops:   # torch creates the CUDA event on first record
        e.record()
    torch.cuda.synchronize()
    L.lora_profile_arm(prof_class, starts, stops)
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                run()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        replay = graph.replay
    else:
        replay = run
    used = L.lora_profile_used()
    if graph is None:
        L.lora_profile_arm(0, [], [])   # eager: only the warm-armed launches above were bracketed
    for _ in range(2):
        replay()
    torch.cuda.synchronize()

    # timed region
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    K = args.steps
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev0.record(stream)
    for i in range(K):
        replay()
        step_ev[i].record(stream)   # per-step boundaries for the median / p10 / p90
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    per_step = [(ev0 if i == 0 else step_ev[i - 1]).elapsed_time(step_ev[i]) for i in range(K)]
    # dominant-kernel durations from the last replay
    kern_ms = [a.elapsed_time(b) for a, b in zip(starts[:used], stops[:used])] if used else []
    # end-to-end through host buffers: H2D of the step's inputs, the step, D2H of the result.
    # The inputs live in one flat device buffer (pack_inputs), so the batch is one pinned host
    # buffer and one copy (one large copy runs near the host link's rate; 88 separate 1-8 MB
    # copies measured about 15% slower).
    pinned = torch.empty(flat_in.numel(), dtype=torch.uint8, pin_memory=True)
    pinned.copy_(flat_in)
    # two pinned result sets: the host reads step k's result while step k + 1 is queued
    res_host = [[torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in results]
                for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in inputs)
    d2h = sum(t.numel() * t.element_size() for t in res_host[0])
    # As a training loop would, the next step's batch is copied host -> device on a second stream
    # while the current step runs: two input buffers take turns, each with its own captured step
    # (the second capture reads the second buffer), so the copy lands in the idle buffer. Every
    # step still copies its whole input from pinned host memory and reads its result back.
    flat_b = torch.empty_like(flat_in)
    flat_b.copy_(flat_in)
    if graph is not None:
        rebind_inputs(inputs, flat_b, in_offs)
        graph_b = torch.cuda.CUDAGraph()
        sb = torch.cuda.Stream(device=device)
        sb.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(sb):
            with torch.cuda.graph(graph_b, stream=sb):
                run()
        torch.cuda.current_stream().wait_stream(sb)
        graph_b.replay()   # warm: the first replay of a capture does one-time work
        torch.cuda.synchronize()
        rebind_inputs(inputs, flat_in, in_offs)
        steps_on = [graph.replay, graph_b.replay]
    else:
        def eager_on(buf):
            def go():
                rebind_inputs(inputs, buf, in_offs)
                run()
            return go
        steps_on = [eager_on(flat_in), eager_on(flat_b)]
    bufs = [flat_in, flat_b]
    copy_stream = torch.cuda.Stream(device=device)
    # the host link's rate for this batch, alone (context for the e2e number)
    h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h2d_alone_ms = []
    for _ in range(2):
        h0.record(copy_stream)
        with torch.cuda.stream(copy_stream):
            flat_b.copy_(pinned, non_blocking=True)
        h1.record(copy_stream)
        h1.synchronize()
        h2d_alone_ms.append(h0.elapsed_time(h1))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    Ke = max(3, K // 2)
    torch.cuda.synchronize()
    e0.record(stream)

    copy_ev = []       # (start, end) of every timed host -> device copy
    step_ev_e2e = []   # (start, end) of every step in the loop

    def h2d_into(buf, after):
        # `after`: the end of the step that last read `buf`
        if after is not None:
            copy_stream.wait_event(after)
        c0 = torch.cuda.Event(enable_timing=True)
        c0.record(copy_stream)
        with torch.cuda.stream(copy_stream):
            buf.copy_(pinned, non_blocking=True)
        done = torch.cuda.Event(enable_timing=True)
        done.record(copy_stream)
        copy_ev.append((c0, done))
        return done

    # Step k: wait for its batch, queue the next batch's copy into the other buffer (after the
    # step that last read it), run, copy the result to host memory; the host then reads step
    # k - 1's result, so that step k is already queued while the host waits (a training loop
    # that logs each step's loss one step late).
    step_end = [None, None]
    check = 0.0
    h2d_done = h2d_into(bufs[0], None)
    for k in range(Ke):
        stream.wait_event(h2d_done)
        if k + 1 < Ke:
            h2d_done = h2d_into(bufs[(k + 1) % 2], step_end[(k + 1) % 2])
        s0 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        steps_on[k % 2]()
        s1 = torch.cuda.Event(enable_timing=True)
        s1.record(stream)
        step_ev_e2e.append((s0, s1))
        for dst, src in zip(res_host[k % 2], results):
            dst.copy_(src, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(stream)
        if k >= 1:
            step_end[(k - 1) % 2].synchronize()
            check += float(res_host[(k - 1) % 2][0].double().sum())
        step_end[k % 2] = ev
    step_end[(Ke - 1) % 2].synchronize()
    check += float(res_host[(Ke - 1) % 2][0].double().sum())
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    copy_ms = [a.elapsed_time(b) for a, b in copy_ev]
    loop_step_ms = [a.elapsed_time(b) for a, b in step_ev_e2e]
    # step-end to step-end periods of the loop (a single slow host copy, for instance from other
    # traffic on the host link, shows up as one long period)
    ends = [b for _, b in step_ev_e2e]
    periods = [(e0 if k == 0 else ends[k - 1]).elapsed_time(ends[k]) for k in range(len(ends))]
    rebind_inputs(inputs, flat_in, in_offs)
    if graph is not None:
        del graph_b
    del flat_b, bufs
    clk = clocks.stop()

    # the kernel classes once more with every linear on one stream (a capture per class after
    # the timed region): the kernels' own durations, without the sharing of the multi-stream step
    def serial_times(cls, n_max):
        step.active_streams = 1
        s_starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_max)]
        s_stops = [torch.cuda.Event(enable_timing=True) for _ in range(n_max)]
        for e in s_starts + s_stops:
            e.record()
        torch.cuda.synchronize()
        L.lora_profile_arm(cls, s_starts, s_stops)
        g1 = torch.cuda.CUDAGraph()
        s1 = torch.cuda.Stream(device=device)
        s1.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s1):
            with torch.cuda.graph(g1, stream=s1):
                run()
        torch.cuda.current_stream().wait_stream(s1)
        used1 = L.lora_profile_used()
        L.lora_profile_arm(0, [], [])
        for _ in range(2):
            g1.replay()
        torch.cuda.synchronize()
        step.active_streams = step.n_streams
        del g1
        return [a.elapsed_time(b) for a, b in zip(s_starts[:used1], s_stops[:used1])]

    kern_serial, mem_times = [], {}
    if graph is not None:
        if getattr(step, "n_streams", 1) > 1:
            kern_serial = serial_times(prof_class, n_prof)
        for name, cls in (("shrink", L.LORA_PROF_SHRINK), ("G", L.LORA_PROF_G),
                          ("redB", L.LORA_PROF_RED_DB), ("redA", L.LORA_PROF_RED_DA),
                          ("red", L.LORA_PROF_RED),
                          ("prepare", L.LORA_PROF_PREPARE), ("adamw", L.LORA_PROF_ADAMW)):
            # the chained step launches each low-rank class once per chunk and layer
            mem_times[name] = serial_times(cls, max(n_prof, 8) * (cfg.chunks if args.chain else 1))

    ms, e2e_ms = max_over_ranks([ms, e2e_ms], world, device)
    tokens = cfg.tokens
    value = whole_job_rate(world, K, tokens, ms)
    e2e_value = whole_job_rate(world, Ke, tokens, e2e_ms)

    if rank == 0:
        peaks, peak_src = load_peaks()
        cnt = counts(cfg, layers if not cfg.multi else 1)
        per_launch = cnt["fwd_flops_per_launch"] if prof_class == L.LORA_PROF_FROZEN_FWD \
            else cnt["dx_flops_per_launch"]
        if args.chain:   # the chained step launches each product once per chunk
            per_launch /= cfg.chunks
        if args.fused:   # one product per group of projections
            per_launch *= len(cfg.projs) / len(fused_groups(cfg))
        avg_kern = statistics.mean(kern_ms) if kern_ms else None
        # The measured bf16 peak comes as a burst (a kernel timed alone) and as a seconds-long
        # loop under the power cap (sustained): a timed region of a second or more keeps the GPU
        # at its power limit, so its kernels are held against the sustained figure.
        sustained = ms / 1e3 >= 1.0 and "bf16_tflops_sustained" in peaks
        bf16_peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        kind = ("sustained (timed region %.1f s)" % (ms / 1e3)) if sustained else "burst"
        if cfg.dtype == "f32":
            # fp32 products as four bf16 products of the split operands
            peak = bf16_peak / 4.0
            bound, punit = "tensor", "TFLOP/s"
            note = (f"split-bf16 effective: measured bf16 {kind} {bf16_peak:.0f} / 4 products "
                    f"({peak_src})")
        elif cfg.dtype == "bf16fp8":
            # E4M3 products: the measured bf16 rate x the nominal fp8 : bf16 ratio (4.5 : 2.25)
            peak = bf16_peak * 4.5 / 2.25
            bound, punit = "tensor", "TFLOP/s"
            note = (f"fp8 effective: measured bf16 {kind} {bf16_peak:.0f} x 4.5/2.25 "
                    f"({peak_src})")
        else:
            peak = bf16_peak
            bound, punit = "tensor", "TFLOP/s"
            note = f"dense bf16 cuBLAS {kind}, {peak_src}"
        avg_serial = statistics.mean(kern_serial) if kern_serial else None
        # the roofline takes the kernel's own launch durations: from the single-stream capture
        # when the step runs on several streams (there, concurrent launches stretch each
        # other's event brackets), else from the timed step itself
        own = kern_serial if kern_serial else kern_ms
        avg_own = statistics.mean(own) if own else None
        achieved = per_launch / (avg_own / 1e3) / 1e12 if avg_own else None
        achieved_overlap = per_launch / (avg_kern / 1e3) / 1e12 if avg_kern else None
        mem = memory_counts(cfg, layers if not cfg.multi else 1,
                            fused_groups(cfg) if args.fused else None)
        memory_bound = {}
        # "red": the dB and dA reductions of a linear in one launch, both classes' bytes (fused
        # groups count their own)
        class_bytes = dict(mem)
        class_bytes.setdefault("red", mem["redB"] + mem["redA"])
        for name, ts in mem_times.items():
            if ts:
                gbs = class_bytes[name] / (sum(ts) / 1e3) / 1e9
                memory_bound[name] = {"achieved_gbs": gbs, "frac": gbs / peaks["hbm_gbs"],
                                      "launches": len(ts), "ms_total": sum(ts),
                                      "bytes_per_step": class_bytes[name]}
        # step-level bound: every frozen product at the tensor peak plus every memory-bound
        # class's algorithmic bytes at the HBM peak, against the measured step
        t_tensor = (cnt["fwd_flops"] + cnt["dx_flops"]) / (peak * 1e12) * 1e3
        t_hbm = sum(mem.values()) / (peaks["hbm_gbs"] * 1e9) * 1e3
        step_roofline = {"t_bound_ms": t_tensor + t_hbm, "t_tensor_ms": t_tensor,
                         "t_hbm_ms": t_hbm, "t_measured_ms": ms / K,
                         "frac": (t_tensor + t_hbm) / (ms / K)}
        traffic, traffic_note = traffic_for(cfg.name, prof_class)
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(cfg, layers)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
            "step_ms": step_stats(per_step),
            "step_roofline": step_roofline,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {"f32": "f32", "bf16": "bf16"}.get(cfg.dtype, "e4m3 frozen, bf16 adapter"),
            "data": "synthetic",
            "config": {"workload": workload_name(cfg, layers, args.chain, args.fused),
                       "tokens_per_step": tokens,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (frozen W alone exceeds 129 MB)"
                       if cfg.name != "c1" else "inputs fit in L2",
                       "cuda_graph": graph is not None,
                       "streams": 1 if args.chain else args.streams},
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": punit,
                         "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                         "traffic_note": traffic_note,
                         "kernel": {1: "frozen forward GEMM", 2: "frozen dX GEMM"}.get(
                             prof_class, f"class {prof_class}"),
                         "launches_timed": len(own), "avg_launch_ms": avg_own,
                         "sum_launch_ms": sum(own) if own else None,
                         "flops_per_launch": per_launch,
                         "timing": "single-stream capture of the same step (CUDA events on the "
                                   "launching stream around every launch of the class)"
                                   if kern_serial else "the timed step's launches (one stream)",
                         "peak_source": note},
            "roofline_overlapped": None if not kern_serial or achieved_overlap is None else {
                "achieved": achieved_overlap, "frac": achieved_overlap / peak,
                "avg_launch_ms": avg_kern, "launches_timed": len(kern_ms),
                "note": "event brackets inside the multi-stream timed step, where concurrent "
                        "launches overlap: not the kernel's own duration"},
            "memory_bound": {"peak_gbs": peaks["hbm_gbs"], "kernels": memory_bound,
                             "note": "algorithmic bytes per step / summed launch times, "
                                     "single-stream capture"} if memory_bound else None,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "h2d_alone_gbs": h2d / (min(h2d_alone_ms) / 1e3) / 1e9 if h2d_alone_ms else None,
                    "h2d_in_loop_ms": sorted(copy_ms)[len(copy_ms) // 2] if copy_ms else None,
                    "step_in_loop_ms": sorted(loop_step_ms)[len(loop_step_ms) // 2]
                    if loop_step_ms else None,
                    "period_ms": {"median": statistics.median(periods), "max": max(periods)}
                    if periods else None,
                    # every step's result (clip scale and norm) was read on the host
                    "results_finite": math.isfinite(check)},
            "gpu_launches": launches_per_step * K,
            # the last step's optimizer status (0: every group updated; non-zero: a group's
            # gradients were non-finite and its update was skipped) and gradient norm
            "step_status": int(results[1].max().item()) if results[1].numel() else None,
            "grad_norm": float(results[0][1].item()) if results[0].numel() > 1 else None,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.oracle_single_thread:
        print(json.dumps(oracle_single_thread()), flush=True)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
