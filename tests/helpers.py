"""Shared helpers for the tests: seeded problems fed identically to the CUDA path and the oracle,
and the per-tensor error metric (max |x - r| / max |r|)."""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

import lora_inputs as LI
from oracle import lora_oracle as O

TOL_F32 = 1e-5          # fp32 frozen-W paths: every output and the post-step state
TOL_BF16 = 2e-2         # bf16 frozen-W paths: Y, dX, dA, dB
TOL_BF16_STEP = 1e-2    # bf16 frozen-W paths: post-step A / B


def rel_err(x, ref) -> float:
    x = np.asarray(x.detach().cpu().double().numpy() if hasattr(x, "detach") else x, np.float64)
    ref = np.asarray(ref.detach().cpu().double().numpy() if hasattr(ref, "detach") else ref,
                     np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(x - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den


def to64(t) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def lr_for(cfg: LI.LoraConfig) -> float:
    return O.lr_at(cfg.sched, cfg.lr, cfg.opt_step, cfg.warmup, cfg.total, cfg.min_lr)


def build_single(cfg: LI.LoraConfig, layers: Sequence[int], proj_idx: Sequence[int],
                 tokens: Optional[int] = None, device="cuda", n_streams: int = 1,
                 overrides: Optional[dict] = None):
    """CUDA LoraStep and the oracle's problems/state from the same seeded inputs."""
    from bwd_adapter_adamw_gb300 import binding as L
    from bwd_adapter_adamw_gb300.step import Linear, LoraStep
    T = cfg.tokens if tokens is None else tokens
    linears, problems, state, init = [], {}, {}, {}
    for l in layers:
        for pi in proj_idx:
            pr = cfg.projs[pi]
            X = LI.make_x(cfg, l, pr, tokens=T)
            W = LI.make_w(cfg, l, pr)
            dY = LI.make_dy(cfg, l, pr, tokens=T)
            A = LI.make_a(cfg, l, pr)
            B = LI.make_b(cfg, l, pr)
            linears.append(Linear(l, pi, X.to(device), W.to(device), dY.to(device)))
            problems[(l, pi)] = dict(X=X, W=W, dY=dY, layer=l, proj=pi)
            init[(l, pi)] = (A, B, W)
    s = O.lora_scale(cfg.alpha, cfg.rank, cfg.rslora)
    hp = L.make_hp(cfg.beta1, cfg.beta2, cfg.eps, cfg.wd, cfg.plus_ratio)
    step = LoraStep(linears, rank=cfg.rank, scale=s, dtype=cfg.dtype, tokens=T, chunks=cfg.chunks,
                    dropout_p=cfg.dropout_p, seed=cfg.dropout_seed, dora=cfg.dora,
                    max_norm=cfg.max_norm, hp=hp, n_streams=n_streams, device=device)
    mA, vA = LI.make_adam_state(cfg, step.n_a, "A")
    mB, vB = LI.make_adam_state(cfg, step.n_b, "B")
    na, nb = step.n_a, step.n_b
    step.arena.m[:na].copy_(mA)
    step.arena.v[:na].copy_(vA)
    step.arena.m[na:na + nb].copy_(mB)
    step.arena.v[na:na + nb].copy_(vB)
    oa, ob = 0, 0
    for lin in step.linears:
        A, B, W = init[(lin.layer, lin.proj_id)]
        lin.A.copy_(A)
        lin.B.copy_(B)
        st = O.AdapterState(A.numpy().copy(), B.numpy().copy(),
                            mA[oa:oa + A.numel()].numpy().reshape(A.shape).copy(),
                            vA[oa:oa + A.numel()].numpy().reshape(A.shape).copy(),
                            mB[ob:ob + B.numel()].numpy().reshape(B.shape).copy(),
                            vB[ob:ob + B.numel()].numpy().reshape(B.shape).copy())
        oa += A.numel()
        ob += B.numel()
        if cfg.dora:
            mag = LI.dora_magnitude_init(W)
            lin.mag.copy_(mag)
            st.mag = mag.numpy().copy()
            st.mM = np.zeros_like(st.mag)
            st.vM = np.zeros_like(st.mag)
        state[(lin.layer, lin.proj_id)] = st
    step.prepare_weights()
    torch.cuda.synchronize()
    hp_o = O.AdamHP(lr=lr_for(cfg), beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps, wd=cfg.wd,
                    plus_ratio=cfg.plus_ratio, step=cfg.opt_step)
    return step, problems, state, s, hp_o
