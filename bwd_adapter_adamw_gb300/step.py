"""Host orchestration of one optimizer step through the C ABI.

This module allocates device buffers with torch (flat fp32 arenas for parameters, gradients and
Adam moments; per-stream workspaces) and sequences the library calls: per adapted linear a
forward and a backward over all accumulation chunks, then one grad-prepare and one AdamW launch
over the arena. It computes nothing itself: every number of the step comes from the library's
kernels.

Arena layout (one per adapter set): [A of every linear | B of every linear | DoRA magnitudes],
so a single lora_group describes the global clip ("4.3. Training Guide", Gradient clipping:
clipped globally by L2 norm) and the AdamW kinds. Multi-LoRA uses one group per slot
("Multi-LoRA Training Example (fully-async)", Design: per-slot state, step counts and clipping).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import torch

from . import binding as L

_DT = {"f32": L.LORA_F32, "bf16": L.LORA_BF16, "bf16fp8": L.LORA_BF16_FP8}


def _ws(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _streams_in_use(step):
    """(k, streams): the first k = min(active_streams, n_streams) side streams, or none for k = 1
    (everything on the caller's current stream)."""
    k = max(1, min(step.active_streams, step.n_streams))
    return k, (step.streams[:k] if (step.streams and k > 1) else [])


def _fork(main, use):
    if use:
        ev = torch.cuda.Event()
        ev.record(main)
        for s in use:
            s.wait_event(ev)


def _join(main, use):
    for s in use:
        ev = torch.cuda.Event()
        ev.record(s)
        main.wait_event(ev)


@dataclass
class Linear:
    """One adapted linear with its activations (device tensors)."""
    layer: int
    proj_id: int
    X: torch.Tensor          # [T, in]
    W: torch.Tensor          # [out, in]
    dY: torch.Tensor         # [T, out]
    Wp: Optional[torch.Tensor] = None   # prepared copy of W (bytes), filled by prepare_weights
    Y: Optional[torch.Tensor] = None
    dX: Optional[torch.Tensor] = None
    H: Optional[torch.Tensor] = None
    # views into the arenas
    A: Optional[torch.Tensor] = None
    B: Optional[torch.Tensor] = None
    gA: Optional[torch.Tensor] = None
    gB: Optional[torch.Tensor] = None
    mag: Optional[torch.Tensor] = None
    gmag: Optional[torch.Tensor] = None
    norm: Optional[torch.Tensor] = None

    @property
    def in_dim(self) -> int:
        return self.W.shape[1]

    @property
    def out_dim(self) -> int:
        return self.W.shape[0]


class Arena:
    """Flat fp32 parameter / gradient / moment arenas with named views."""

    def __init__(self, n: int, device):
        self.n = n
        self.params = torch.zeros(n, dtype=torch.float32, device=device)
        self.grads = torch.zeros(n, dtype=torch.float32, device=device)
        self.m = torch.zeros(n, dtype=torch.float32, device=device)
        self.v = torch.zeros(n, dtype=torch.float32, device=device)

    def view(self, which: str, offset: int, shape) -> torch.Tensor:
        numel = 1
        for s in shape:
            numel *= s
        return getattr(self, which)[offset:offset + numel].view(*shape)


class LoraStep:
    """One optimizer step over a set of independent adapted linears sharing rank/scale/dtype."""

    def __init__(self, linears: Sequence[Linear], *, rank: int, scale: float, dtype: str,
                 tokens: int, chunks: int, dropout_p: float = 0.0, seed: int = 0,
                 dora: bool = False, max_norm: float = 1.0, hp: Optional[L.lora_adamw_hp] = None,
                 n_streams: int = 1, device="cuda"):
        self.linears = list(linears)
        self.rank, self.scale, self.dtype = rank, scale, _DT[dtype]
        self.T, self.chunks = tokens, chunks
        self.dropout_p, self.seed, self.dora = dropout_p, seed, dora
        self.max_norm = max_norm
        self.hp = hp if hp is not None else L.make_hp()
        self.device = torch.device(device)
        # arena: [A ... | B ... | MAG ...]
        na = sum(rank * l.in_dim for l in self.linears)
        nb = sum(l.out_dim * rank for l in self.linears)
        nm = sum(l.out_dim for l in self.linears) if dora else 0
        self.n_a, self.n_b, self.n_mag = na, nb, nm
        self.arena = Arena(na + nb + nm, self.device)
        oa, ob, om = 0, na, na + nb
        for l in self.linears:
            l.A = self.arena.view("params", oa, (rank, l.in_dim))
            l.gA = self.arena.view("grads", oa, (rank, l.in_dim))
            oa += rank * l.in_dim
            l.B = self.arena.view("params", ob, (l.out_dim, rank))
            l.gB = self.arena.view("grads", ob, (l.out_dim, rank))
            ob += l.out_dim * rank
            if dora:
                l.mag = self.arena.view("params", om, (l.out_dim,))
                l.gmag = self.arena.view("grads", om, (l.out_dim,))
                om += l.out_dim
                l.norm = torch.empty(l.out_dim, dtype=torch.float32, device=self.device)
            act = l.X.dtype
            if l.Y is None:
                l.Y = torch.empty((self.T, l.out_dim), dtype=act, device=self.device)
            if l.dX is None:
                l.dX = torch.empty((self.T, l.in_dim), dtype=act, device=self.device)
            if l.H is None:
                l.H = torch.empty((self.T, rank), dtype=torch.float32, device=self.device)
        self.n_streams = max(1, n_streams)
        self.streams = [torch.cuda.Stream(device=self.device) for _ in range(self.n_streams)] \
            if self.n_streams > 1 else []
        self.active_streams = self.n_streams   # streams used by the next enqueue (<= n_streams)
        ws_need = max(L.lora_workspace_size(self.desc(l), self.T) for l in self.linears)
        if self.dora:   # the norm refresh shares the stream's workspace
            ws_need = max(ws_need, max(L.lora_dora_norm_workspace_size(self.desc(l))
                                       for l in self.linears))
        if ws_need == 0:
            raise L.LoraError(L.LORA_ERR_INVALID, "lora_workspace_size")
        self.ws = [_ws(ws_need, self.device) for _ in range(self.n_streams)]
        self.scale_norm = torch.zeros(2, dtype=torch.float64, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._groups_cache = None

    # ------------------------------------------------------------------------------------------
    def desc(self, l: Linear) -> L.lora_desc:
        return L.make_desc(l.in_dim, l.out_dim, self.rank, self.scale, self.dtype, self.dropout_p,
                           self.seed, l.layer, l.proj_id, self.dora)

    def prepare_weights(self, stream=None):
        for l in self.linears:
            if l.Wp is None:
                l.Wp = torch.empty(L.lora_prepared_weight_size(self.desc(l)), dtype=torch.uint8,
                                   device=self.device)
            L.lora_prepare_weight(self.desc(l), l.W, l.Wp, stream)

    def groups(self, lr: float, step: int):
        return L.make_groups([dict(offset=0, n_a=self.n_a, n_b=self.n_b, n_mag=self.n_mag,
                                   grad_scale=1.0 / self.T, max_norm=self.max_norm, lr=lr,
                                   step=step)])

    def prepare_ws(self) -> torch.Tensor:
        g = self.groups(0.0, 0)
        if not hasattr(self, "_prep_ws"):
            self._prep_ws = _ws(L.lora_grad_prepare_workspace_size(g), self.device)
        return self._prep_ws

    # ------------------------------------------------------------------------------------------
    def forward_backward(self, opt_step: int, per_chunk_calls: bool = False):
        """Enqueue forward + backward of every linear over all chunks (gradients accumulate)."""
        main = torch.cuda.current_stream(self.device)
        k, use = _streams_in_use(self)
        _fork(main, use)
        ct = self.T // self.chunks
        for i, l in enumerate(self.linears):
            st = use[i % k] if use else main
            ws = self.ws[i % k]
            d = self.desc(l)
            if self.dora:
                L.lora_dora_norm(d, l.W, l.A, l.B, l.norm, ws, stream=st)
            if per_chunk_calls:
                spans = [(c, c * ct, ct) for c in range(self.chunks)]
            else:
                spans = [(0, 0, self.T)]
            for (ordinal, t0, n) in spans:
                ctx = L.make_ctx(opt_step, ordinal, ct)
                sl = slice(t0, t0 + n)
                X, dY, Y, dX, H = l.X[sl], l.dY[sl], l.Y[sl], l.dX[sl], l.H[sl]
                L.lora_forward(d, ctx, n, X, l.W, l.Wp, l.A, l.B, l.mag, l.norm, Y, H, ws, stream=st)
                L.lora_backward(d, ctx, n, X, l.Wp, l.A, l.B, dY, H, l.mag, l.norm, Y, dX, l.gA,
                                l.gB, l.gmag, ws, stream=st)
        _join(main, use)

    def optimizer_step(self, lr: float, step: int, zero_grads: bool = True):
        g = self.groups(lr, step)
        ws = self.prepare_ws()
        L.lora_grad_prepare(self.arena.grads, g, self.scale_norm, self.status, ws)
        L.lora_adamw_step(self.arena.params, self.arena.grads, self.arena.m, self.arena.v, g,
                          self.hp, self.scale_norm, self.status, zero_grads)

    def run(self, opt_step: int, lr: float, per_chunk_calls: bool = False, zero_grads: bool = True):
        self.forward_backward(opt_step, per_chunk_calls)
        self.optimizer_step(lr, opt_step, zero_grads)

    def snapshot(self, snap: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Device copy of every adapter's parameters (the best-weights snapshot)."""
        if snap is None:
            snap = torch.empty_like(self.arena.params)
        L.lora_snapshot(self.arena.params, snap, self.groups(0.0, 0))
        return snap

    def restore(self, snap: torch.Tensor, zero_grads: bool = True):
        """Restore a snapshot and reset the optimizer (moments zeroed); the caller's next update
        passes step 0 again."""
        L.lora_restore(self.arena.params, snap, self.arena.grads, self.arena.m, self.arena.v,
                       self.groups(0.0, 0), zero_grads)


@dataclass
class FusedGroup:
    """Projections that read one input, run as one fused linear: the stacked frozen weight
    W [sum out_k, in] and output gradient dY [T, sum out_k], projection k in columns
    [off_k, off_k + out_k)."""
    layer: int
    proj_id: int                 # dropout key of the group (one mask for its projections)
    X: torch.Tensor              # [T, in]
    W: torch.Tensor              # [sum out_k, in]
    dY: torch.Tensor             # [T, sum out_k]
    outs: Tuple[int, ...]        # out_k
    Wp: Optional[torch.Tensor] = None
    Y: Optional[torch.Tensor] = None
    dX: Optional[torch.Tensor] = None
    H: Optional[torch.Tensor] = None            # [T, n rank]
    A: Optional[List[torch.Tensor]] = None      # arena views per projection
    B: Optional[List[torch.Tensor]] = None
    gA: Optional[List[torch.Tensor]] = None
    gB: Optional[List[torch.Tensor]] = None

    @property
    def in_dim(self) -> int:
        return self.W.shape[1]

    @property
    def out_dim(self) -> int:
        return self.W.shape[0]


class FusedLoraStep:
    """One optimizer step over groups of fused projections ("LoRA Training and Serving",
    --lora-type: fused projections, one adapter per projection): each group is one fused
    forward and one fused backward call (one frozen product over the stacked weight each, and
    one input gradient summed over the group's projections); the arena, the global clip and
    AdamW are LoraStep's."""

    def __init__(self, groups: Sequence[FusedGroup], *, rank: int, scale: float, dtype: str,
                 tokens: int, chunks: int, dropout_p: float = 0.0, seed: int = 0,
                 max_norm: float = 1.0, hp: Optional[L.lora_adamw_hp] = None,
                 n_streams: int = 1, device="cuda"):
        self.fgroups = list(groups)
        self.rank, self.scale, self.dtype = rank, scale, _DT[dtype]
        self.T, self.chunks = tokens, chunks
        self.dropout_p, self.seed, self.dora = dropout_p, seed, False
        self.max_norm = max_norm
        self.hp = hp if hp is not None else L.make_hp()
        self.device = torch.device(device)
        na = sum(rank * g.in_dim * len(g.outs) for g in self.fgroups)
        nb = sum(g.out_dim * rank for g in self.fgroups)
        self.n_a, self.n_b, self.n_mag = na, nb, 0
        self.arena = Arena(na + nb, self.device)
        oa, ob = 0, na
        for g in self.fgroups:
            if sum(g.outs) != g.out_dim:
                raise ValueError("the projections' widths must add up to the stacked weight's rows")
            g.A, g.gA, g.B, g.gB = [], [], [], []
            for o in g.outs:
                g.A.append(self.arena.view("params", oa, (rank, g.in_dim)))
                g.gA.append(self.arena.view("grads", oa, (rank, g.in_dim)))
                oa += rank * g.in_dim
                g.B.append(self.arena.view("params", ob, (o, rank)))
                g.gB.append(self.arena.view("grads", ob, (o, rank)))
                ob += o * rank
            act = g.X.dtype
            if g.Y is None:
                g.Y = torch.empty((self.T, g.out_dim), dtype=act, device=self.device)
            if g.dX is None:
                g.dX = torch.empty((self.T, g.in_dim), dtype=act, device=self.device)
            if g.H is None:
                g.H = torch.empty((self.T, rank * len(g.outs)), dtype=torch.float32,
                                  device=self.device)
        self.n_streams = max(1, n_streams)
        self.streams = [torch.cuda.Stream(device=self.device) for _ in range(self.n_streams)] \
            if self.n_streams > 1 else []
        self.active_streams = self.n_streams
        need = max(L.lora_fused_workspace_size(self.desc(g), self.T, self.projs(g))
                   for g in self.fgroups)
        if need == 0:
            raise L.LoraError(L.LORA_ERR_INVALID, "lora_fused_workspace_size")
        self.ws = [_ws(need, self.device) for _ in range(self.n_streams)]
        self.scale_norm = torch.zeros(2, dtype=torch.float64, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    def desc(self, g: FusedGroup) -> L.lora_desc:
        return L.make_desc(g.in_dim, g.out_dim, self.rank, self.scale, self.dtype, self.dropout_p,
                           self.seed, g.layer, g.proj_id, False)

    def projs(self, g: FusedGroup):
        return L.make_projs([dict(A=a, B=b, dA=ga, dB=gb, out=o)
                             for a, b, ga, gb, o in zip(g.A, g.B, g.gA, g.gB, g.outs)])

    def prepare_weights(self, stream=None):
        for g in self.fgroups:
            if g.Wp is None:
                g.Wp = torch.empty(L.lora_prepared_weight_size(self.desc(g)), dtype=torch.uint8,
                                   device=self.device)
            L.lora_prepare_weight(self.desc(g), g.W, g.Wp, stream)

    def forward_backward(self, opt_step: int, per_chunk_calls: bool = False):
        main = torch.cuda.current_stream(self.device)
        k, use = _streams_in_use(self)
        _fork(main, use)
        ct = self.T // self.chunks
        for i, g in enumerate(self.fgroups):
            st = use[i % k] if use else main
            ws = self.ws[i % k]
            d, pj = self.desc(g), self.projs(g)
            ctx = L.make_ctx(opt_step, 0, ct)
            L.lora_fused_forward(d, ctx, self.T, g.X, g.W, g.Wp, pj, g.Y, g.H, ws, stream=st)
            L.lora_fused_backward(d, ctx, self.T, g.X, g.Wp, pj, g.dY, g.H, g.dX, ws, stream=st)
        _join(main, use)

    groups = LoraStep.groups
    prepare_ws = LoraStep.prepare_ws
    optimizer_step = LoraStep.optimizer_step
    run = LoraStep.run
    snapshot = LoraStep.snapshot
    restore = LoraStep.restore


class ChainStep(LoraStep):
    """One optimizer step over a stack of adapted linears in which layer l's output is layer
    l + 1's input ("4.3. Training Guide", Truncated BPTT: the backward window is one chunk of
    tokens; Gradient accumulation: raw sums over the chunks in order). Each chunk runs forward
    through every layer and then backward through them in reverse, layer l's output gradient
    being layer l + 1's input gradient, all on one stream (each launch depends on the one
    before). The layers share the adapter rank, scale and dtype; W_l is [d_{l+1}, d_l]."""

    def __init__(self, Ws: Sequence[torch.Tensor], X0: torch.Tensor, dY_top: torch.Tensor, *,
                 layer_ids: Optional[Sequence[int]] = None, proj_id: int = 0, **kw):
        if kw.get("dora"):
            raise ValueError("the chained step has no DoRA mode")
        T, act, dev = X0.shape[0], X0.dtype, X0.device
        for l in range(1, len(Ws)):
            if Ws[l].shape[1] != Ws[l - 1].shape[0]:
                raise ValueError("layer widths do not chain")
        ids = list(layer_ids) if layer_ids is not None else list(range(len(Ws)))
        lins = [Linear(ids[l], proj_id, None, W, None) for l, W in enumerate(Ws)]
        for lin in lins:
            lin.Y = torch.empty((T, lin.out_dim), dtype=act, device=dev)
            lin.dX = torch.empty((T, lin.in_dim), dtype=act, device=dev)
        for l, lin in enumerate(lins):
            lin.X = X0 if l == 0 else lins[l - 1].Y          # the previous layer's output
            lin.dY = dY_top if l == len(lins) - 1 else lins[l + 1].dX
        kw["n_streams"] = 1
        super().__init__(lins, tokens=T, **kw)

    def forward_backward(self, opt_step: int, per_chunk_calls: bool = True):
        """Enqueue the chunked forward / reverse backward of the whole stack (gradients
        accumulate into the arena)."""
        st = torch.cuda.current_stream(self.device)
        ws = self.ws[0]
        ct = self.T // self.chunks
        for c in range(self.chunks):
            ctx = L.make_ctx(opt_step, c, ct)
            sl = slice(c * ct, (c + 1) * ct)
            for l in self.linears:
                L.lora_forward(self.desc(l), ctx, ct, l.X[sl], l.W, l.Wp, l.A, l.B, None, None,
                               l.Y[sl], l.H[sl], ws, stream=st)
            for l in reversed(self.linears):
                L.lora_backward(self.desc(l), ctx, ct, l.X[sl], l.Wp, l.A, l.B, l.dY[sl],
                                l.H[sl], None, None, None, l.dX[sl], l.gA, l.gB, None, ws,
                                stream=st)


# ----------------------------------------------------------------------------------------------
@dataclass
class MultiLinear:
    proj_id: int
    X: torch.Tensor
    W: torch.Tensor
    dY: torch.Tensor
    Wp: Optional[torch.Tensor] = None
    Y: Optional[torch.Tensor] = None
    dX: Optional[torch.Tensor] = None
    H: Optional[torch.Tensor] = None
    A: List[torch.Tensor] = field(default_factory=list)    # per slot, views into the arena
    B: List[torch.Tensor] = field(default_factory=list)
    gA: List[torch.Tensor] = field(default_factory=list)
    gB: List[torch.Tensor] = field(default_factory=list)

    @property
    def in_dim(self) -> int:
        return self.W.shape[1]

    @property
    def out_dim(self) -> int:
        return self.W.shape[0]


class MultiLoraStep:
    """Slot-keyed multi-LoRA over a shared frozen base: every linear has one adapter per slot;
    one arena group per slot = [A of the slot over all linears | B of the slot]."""

    def __init__(self, linears: Sequence[MultiLinear], *, slot_ranks: Sequence[int],
                 slot_scales: Sequence[float], dtype: str, tokens: int, seg_start: torch.Tensor,
                 seg_slot: torch.Tensor, dropout_p: float = 0.0, seed: int = 0,
                 max_norm: float = 1.0, hp: Optional[L.lora_adamw_hp] = None, n_streams: int = 1,
                 planned: bool = True, device="cuda"):
        self.linears = list(linears)
        self.ranks, self.scales = list(slot_ranks), list(slot_scales)
        self.n_slots = len(self.ranks)
        self.rmax = max(self.ranks)
        self.dtype = _DT[dtype]
        self.T = tokens
        self.seg_start, self.seg_slot = seg_start, seg_slot
        self.n_seg = int(seg_slot.numel())
        self.dropout_p, self.seed = dropout_p, seed
        self.max_norm = max_norm
        self.hp = hp if hp is not None else L.make_hp()
        self.device = torch.device(device)
        self.slot_off, self.slot_na, self.slot_nb = [], [], []
        off = 0
        for r in self.ranks:
            na = sum(r * l.in_dim for l in self.linears)
            nb = sum(l.out_dim * r for l in self.linears)
            self.slot_off.append(off)
            self.slot_na.append(na)
            self.slot_nb.append(nb)
            off += na + nb
        self.arena = Arena(off, self.device)
        for s, r in enumerate(self.ranks):
            oa, ob = self.slot_off[s], self.slot_off[s] + self.slot_na[s]
            for l in self.linears:
                l.A.append(self.arena.view("params", oa, (r, l.in_dim)))
                l.gA.append(self.arena.view("grads", oa, (r, l.in_dim)))
                oa += r * l.in_dim
                l.B.append(self.arena.view("params", ob, (l.out_dim, r)))
                l.gB.append(self.arena.view("grads", ob, (l.out_dim, r)))
                ob += l.out_dim * r
        for l in self.linears:
            act = l.X.dtype
            if l.Y is None:
                l.Y = torch.empty((self.T, l.out_dim), dtype=act, device=self.device)
            if l.dX is None:
                l.dX = torch.empty((self.T, l.in_dim), dtype=act, device=self.device)
            if l.H is None:
                l.H = torch.empty((self.T, self.rmax), dtype=torch.float32, device=self.device)
        self.n_streams = max(1, n_streams)
        self.streams = [torch.cuda.Stream(device=self.device) for _ in range(self.n_streams)] \
            if self.n_streams > 1 else []
        self.active_streams = self.n_streams   # streams used by the next enqueue (<= n_streams)
        need = max(L.multi_lora_workspace_size(self.desc(l), self.T, self.n_seg, self.slots(l))
                   for l in self.linears)
        if need == 0:
            raise L.LoraError(L.LORA_ERR_INVALID, "multi_lora_workspace_size")
        self.ws = [_ws(need, self.device) for _ in range(self.n_streams)]
        # the routing plan: the batch's token work tables, built once per forward_backward and
        # read by every linear's calls
        self.plan = None
        if planned and self.n_seg >= 1:
            nbytes = L.multi_lora_plan_size(self.T, self.n_seg, self.n_slots)
            if nbytes == 0:
                raise L.LoraError(L.LORA_ERR_INVALID, "multi_lora_plan_size")
            self.plan = _ws(nbytes, self.device)
        self.scale_norm = torch.zeros(2 * self.n_slots, dtype=torch.float64, device=self.device)
        self.status = torch.zeros(self.n_slots, dtype=torch.int32, device=self.device)

    def desc(self, l: MultiLinear) -> L.lora_desc:
        return L.make_desc(l.in_dim, l.out_dim, self.rmax, 0.0, self.dtype, self.dropout_p,
                           self.seed, 0, l.proj_id, False)

    def slots(self, l: MultiLinear):
        return L.make_slots([dict(A=l.A[s], B=l.B[s], dA=l.gA[s], dB=l.gB[s], rank=self.ranks[s],
                                  scale=self.scales[s]) for s in range(self.n_slots)])

    def prepare_weights(self, stream=None):
        for l in self.linears:
            if l.Wp is None:
                l.Wp = torch.empty(L.lora_prepared_weight_size(self.desc(l)), dtype=torch.uint8,
                                   device=self.device)
            L.lora_prepare_weight(self.desc(l), l.W, l.Wp, stream)

    def forward_backward(self, opt_step: int = 0):
        main = torch.cuda.current_stream(self.device)
        if self.plan is not None:
            L.multi_lora_plan_build(self.T, self.n_seg, self.seg_start, self.seg_slot,
                                    self.n_slots, self.plan, stream=main)
        k, use = _streams_in_use(self)
        _fork(main, use)
        for i, l in enumerate(self.linears):
            st = use[i % k] if use else main
            ws = self.ws[i % k]
            d = self.desc(l)
            ctx = L.make_ctx(opt_step, 0, 0)
            sl = self.slots(l)
            if self.plan is not None:
                L.multi_lora_forward_planned(d, ctx, self.T, self.n_seg, self.plan, l.X, l.W, l.Wp,
                                             sl, l.Y, l.H, ws, stream=st)
                L.multi_lora_backward_planned(d, ctx, self.T, self.n_seg, self.plan, l.X, l.Wp, sl,
                                              l.dY, l.H, l.dX, ws, stream=st)
            else:
                L.multi_lora_forward(d, ctx, self.T, l.X, l.W, l.Wp, self.n_seg, self.seg_start,
                                     self.seg_slot, sl, l.Y, l.H, ws, stream=st)
                L.multi_lora_backward(d, ctx, self.T, l.X, l.Wp, self.n_seg, self.seg_start,
                                      self.seg_slot, sl, l.dY, l.H, l.dX, ws, stream=st)
        _join(main, use)

    def groups(self, ready: Sequence[int], gbs: Sequence[int], lrs: Sequence[float],
               steps: Sequence[int]):
        return L.make_groups([dict(offset=self.slot_off[s], n_a=self.slot_na[s],
                                   n_b=self.slot_nb[s], grad_scale=1.0 / gbs[s],
                                   max_norm=self.max_norm, lr=lrs[s], step=steps[s])
                              for s in ready])

    def retire(self, slots: Sequence[int], clear_params: bool = True):
        """Retire finished adapter slots: their gradients (the partial accumulation), moments and,
        with clear_params, weights are zeroed. The caller resets the slots' accumulated sample
        counts and update counts."""
        if not slots:
            return
        g = L.make_groups([dict(offset=self.slot_off[s], n_a=self.slot_na[s],
                                n_b=self.slot_nb[s], grad_scale=1.0) for s in slots])
        L.lora_retire(self.arena.params, self.arena.grads, self.arena.m, self.arena.v, g,
                      clear_params)

    def optimizer_step(self, ready: Sequence[int], gbs, lrs, steps, zero_grads: bool = True):
        """Prepare + AdamW for the slots whose adapter batch is full (one group each); group i of
        the call reports in scale_norm[2i:2i+2] and status[i]."""
        if not ready:
            return
        g = self.groups(ready, gbs, lrs, steps)
        if not hasattr(self, "_prep_ws"):
            full = self.groups(range(self.n_slots), gbs, lrs, steps)
            self._prep_ws = _ws(L.lora_grad_prepare_workspace_size(full), self.device)
        L.lora_grad_prepare(self.arena.grads, g, self.scale_norm, self.status, self._prep_ws)
        L.lora_adamw_step(self.arena.params, self.arena.grads, self.arena.m, self.arena.v, g,
                          self.hp, self.scale_norm, self.status, zero_grads)
