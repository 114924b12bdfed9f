"""ctypes binding of liblora_gb300.so: argument marshalling only.

Every function here has the name of the C entry point it calls, converts torch tensors to device
pointers and Python values to the C structs, and raises LoraError on a nonzero status. All
computation happens in the library's kernels; there is no fallback of any kind. If the library
is missing the import fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "liblora_gb300.so")

LORA_OK = 0
LORA_ERR_INVALID = 1
LORA_ERR_ALIGN = 2
LORA_ERR_UNSUPPORTED = 3
LORA_ERR_WORKSPACE = 4
LORA_ERR_CUDA = 5
LORA_ERR_NONFINITE = 6
LORA_ERR_TIMEOUT = 7

LORA_F32 = 0
LORA_BF16 = 1
LORA_BF16_FP8 = 2
LORA_SCHED_CONSTANT = 0
LORA_SCHED_WARMUP_COSINE = 1
LORA_MAX_RANK = 64
LORA_MAX_SLOTS = 32
LORA_MAX_GROUPS = 64


class LoraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class lora_desc(C.Structure):
    _fields_ = [("in_dim", C.c_int64), ("out_dim", C.c_int64), ("rank", C.c_int32),
                ("scale", C.c_float), ("dtype", C.c_int32), ("dropout_p", C.c_float),
                ("seed", C.c_uint64), ("layer_id", C.c_uint32), ("proj_id", C.c_uint32),
                ("dora", C.c_int32)]


class lora_ctx(C.Structure):
    _fields_ = [("opt_step", C.c_uint64), ("accum_ordinal", C.c_uint32),
                ("chunk_tokens", C.c_int64)]


class lora_slot(C.Structure):
    _fields_ = [("A", C.c_void_p), ("B", C.c_void_p), ("dA", C.c_void_p), ("dB", C.c_void_p),
                ("rank", C.c_int32), ("scale", C.c_float)]


class lora_proj(C.Structure):
    _fields_ = [("A", C.c_void_p), ("B", C.c_void_p), ("dA", C.c_void_p), ("dB", C.c_void_p),
                ("out_dim", C.c_int64)]


class lora_group(C.Structure):
    _fields_ = [("offset", C.c_int64), ("n_a", C.c_int64), ("n_b", C.c_int64),
                ("n_mag", C.c_int64), ("grad_scale", C.c_double), ("max_norm", C.c_float),
                ("lr", C.c_float), ("step", C.c_int64)]


class lora_adamw_hp(C.Structure):
    _fields_ = [("beta1", C.c_double), ("beta2", C.c_double), ("eps", C.c_double),
                ("weight_decay", C.c_double), ("plus_ratio", C.c_double)]


def _load() -> C.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run bwd_adapter_adamw_gb300.build.build() (nvcc, sm_103a)")
    lib = C.CDLL(LIB_PATH)
    P, I32, I64, U64, SZ, F, D = (C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_size_t,
                                  C.c_float, C.c_double)
    DP, CP = C.POINTER(lora_desc), C.POINTER(lora_ctx)
    sig = {
        "lora_status_string": (C.c_char_p, [C.c_int]),
        "lora_scale": (F, [F, I32, I32]),
        "lora_lr_at": (D, [I32, D, U64, U64, U64, D]),
        "lora_workspace_size": (SZ, [DP, I64]),
        "lora_prepared_weight_size": (SZ, [DP]),
        "lora_prepare_weight": (C.c_int, [DP, P, P, P]),
        "lora_dora_norm_workspace_size": (SZ, [DP]),
        "lora_dora_norm": (C.c_int, [DP, P, P, P, P, P, SZ, P]),
        "lora_forward": (C.c_int, [DP, CP, I64, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "lora_backward": (C.c_int, [DP, CP, I64, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "lora_grad_prepare_workspace_size": (SZ, [I32, C.POINTER(lora_group)]),
        "lora_grad_prepare": (C.c_int, [P, I32, C.POINTER(lora_group), P, P, P, SZ, P]),
        "lora_grad_prepare_noalloc": (C.c_int, [P, I32, C.POINTER(lora_group), P, P, P]),
        "lora_adamw_step": (C.c_int, [P, P, P, P, I32, C.POINTER(lora_group),
                                      C.POINTER(lora_adamw_hp), P, P, I32, P]),
        "lora_snapshot": (C.c_int, [P, P, I32, C.POINTER(lora_group), P]),
        "lora_restore": (C.c_int, [P, P, P, P, P, I32, C.POINTER(lora_group), I32, P]),
        "lora_retire": (C.c_int, [P, P, P, P, I32, C.POINTER(lora_group), I32, P]),
        "multi_lora_workspace_size": (SZ, [DP, I64, I32, I32, C.POINTER(lora_slot)]),
        "lora_fused_workspace_size": (SZ, [DP, I64, I32, C.POINTER(lora_proj)]),
        "lora_fused_forward": (C.c_int, [DP, CP, I64, P, P, P, I32, C.POINTER(lora_proj), P, P,
                                         P, SZ, P]),
        "lora_fused_backward": (C.c_int, [DP, CP, I64, P, P, I32, C.POINTER(lora_proj), P, P, P,
                                          P, SZ, P]),
        "multi_lora_forward": (C.c_int, [DP, CP, I64, P, P, P, I32, P, P, I32,
                                         C.POINTER(lora_slot), P, P, P, SZ, P]),
        "multi_lora_backward": (C.c_int, [DP, CP, I64, P, P, I32, P, P, I32,
                                          C.POINTER(lora_slot), P, P, P, P, SZ, P]),
        "multi_lora_plan_size": (SZ, [I64, I32, I32]),
        "multi_lora_plan_build": (C.c_int, [I64, I32, P, P, I32, P, SZ, P]),
        "multi_lora_forward_planned": (C.c_int, [DP, CP, I64, I32, P, P, P, P, I32,
                                                 C.POINTER(lora_slot), P, P, P, SZ, P]),
        "multi_lora_backward_planned": (C.c_int, [DP, CP, I64, I32, P, P, P, I32,
                                                  C.POINTER(lora_slot), P, P, P, P, SZ, P]),
        "lora_dropout_mask": (C.c_int, [DP, CP, I64, P, P]),
        "lora_quantize_e4m3": (C.c_int, [P, I64, I64, P, P, P]),
        "multi_lora_token_slots": (C.c_int, [I64, I32, P, P, I32, P, P]),
        "lora_profile_arm": (C.c_int, [I32, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), I32]),
        "lora_profile_used": (I32, []),
        "lora_launch_counter": (U64, []),
        "lora_last_cuda_error": (C.c_char_p, []),
        "lora_device_error": (C.c_int, [C.POINTER(C.c_uint32), I32]),
        "lora_device_check": (C.c_int, [P]),
        "lora_set_wait_limit": (C.c_int, [U64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
EXPORTED = ("lora_status_string", "lora_scale", "lora_lr_at", "lora_workspace_size",
            "lora_prepared_weight_size", "lora_prepare_weight", "lora_dora_norm_workspace_size",
            "lora_dora_norm", "lora_forward", "lora_backward",
            "lora_grad_prepare_workspace_size", "lora_grad_prepare", "lora_grad_prepare_noalloc",
            "lora_adamw_step", "lora_snapshot", "lora_restore", "lora_retire",
            "multi_lora_workspace_size", "multi_lora_forward", "multi_lora_backward",
            "multi_lora_plan_size", "multi_lora_plan_build", "multi_lora_forward_planned",
            "multi_lora_backward_planned",
            "lora_fused_workspace_size", "lora_fused_forward", "lora_fused_backward",
            "lora_dropout_mask", "lora_quantize_e4m3", "multi_lora_token_slots", "lora_profile_arm",
            "lora_profile_used", "lora_launch_counter", "lora_last_cuda_error",
            "lora_device_error", "lora_device_check", "lora_set_wait_limit")

LORA_PROF_NONE = 0
LORA_PROF_FROZEN_FWD = 1
LORA_PROF_FROZEN_DX = 2
LORA_PROF_SHRINK = 3
LORA_PROF_G = 4
LORA_PROF_RED_DB = 5
LORA_PROF_RED_DA = 6
LORA_PROF_PREPARE = 7
LORA_PROF_ADAMW = 8
LORA_PROF_RED = 9


def library_path() -> str:
    return LIB_PATH


# ------------------------------------------------------------------------------------ marshalling
def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> int:
    if status == LORA_ERR_CUDA:
        raise LoraError(status, f"{where} [{_lib.lora_last_cuda_error().decode()}]")
    if status != LORA_OK:
        raise LoraError(status, where)
    return status


def status_string(status: int) -> str:
    return _lib.lora_status_string(status).decode()


def make_desc(in_dim, out_dim, rank, scale, dtype, dropout_p=0.0, seed=0, layer_id=0, proj_id=0,
              dora=False) -> lora_desc:
    return lora_desc(in_dim, out_dim, rank, scale, dtype, dropout_p, seed, layer_id, proj_id,
                     1 if dora else 0)


def make_ctx(opt_step=0, accum_ordinal=0, chunk_tokens=0) -> lora_ctx:
    return lora_ctx(opt_step, accum_ordinal, chunk_tokens)


def lora_scale(alpha: float, rank: int, rslora: bool) -> float:
    return _lib.lora_scale(alpha, rank, 1 if rslora else 0)


def lora_lr_at(kind: int, base: float, step: int, warmup: int, total: int, min_lr: float) -> float:
    return _lib.lora_lr_at(kind, base, step, warmup, total, min_lr)


def lora_workspace_size(d: lora_desc, T: int) -> int:
    return _lib.lora_workspace_size(C.byref(d), T)


def lora_prepared_weight_size(d: lora_desc) -> int:
    return _lib.lora_prepared_weight_size(C.byref(d))


def lora_prepare_weight(d: lora_desc, W, W_prep, stream=None):
    return _check(_lib.lora_prepare_weight(C.byref(d), _ptr(W), _ptr(W_prep), _stream(stream)),
                  "lora_prepare_weight")


def lora_dora_norm_workspace_size(d: lora_desc) -> int:
    return _lib.lora_dora_norm_workspace_size(C.byref(d))


def lora_dora_norm(d: lora_desc, W, A, B, norm_out, ws, ws_bytes: Optional[int] = None,
                   stream=None):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    return _check(_lib.lora_dora_norm(C.byref(d), _ptr(W), _ptr(A), _ptr(B), _ptr(norm_out),
                                      _ptr(ws), nbytes, _stream(stream)), "lora_dora_norm")


def lora_forward(d: lora_desc, c: Optional[lora_ctx], T: int, X, W, W_prep, A, B, dora_m, dora_n,
                 Y, H_save, ws, ws_bytes: Optional[int] = None, stream=None, check=True):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    st = _lib.lora_forward(C.byref(d), C.byref(c) if c is not None else None, T, _ptr(X), _ptr(W),
                           _ptr(W_prep), _ptr(A), _ptr(B), _ptr(dora_m), _ptr(dora_n), _ptr(Y), _ptr(H_save),
                           _ptr(ws), nbytes, _stream(stream))
    return _check(st, "lora_forward") if check else st


def lora_backward(d: lora_desc, c: Optional[lora_ctx], T: int, X, W_prep, A, B, dY, H_save, dora_m,
                  dora_n, Y_save, dX, dA, dB, dm, ws, ws_bytes: Optional[int] = None, stream=None,
                  check=True):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    st = _lib.lora_backward(C.byref(d), C.byref(c) if c is not None else None, T, _ptr(X),
                            _ptr(W_prep), _ptr(A), _ptr(B), _ptr(dY), _ptr(H_save), _ptr(dora_m),
                            _ptr(dora_n), _ptr(Y_save), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(dm),
                            _ptr(ws), nbytes, _stream(stream))
    return _check(st, "lora_backward") if check else st


def make_groups(groups: Sequence[dict]):
    arr = (lora_group * len(groups))()
    for i, g in enumerate(groups):
        arr[i] = lora_group(g["offset"], g.get("n_a", 0), g.get("n_b", 0), g.get("n_mag", 0),
                            g["grad_scale"], g.get("max_norm", 0.0), g.get("lr", 0.0),
                            g.get("step", 0))
    return arr


def lora_grad_prepare_workspace_size(groups) -> int:
    return _lib.lora_grad_prepare_workspace_size(len(groups), groups)


def lora_grad_prepare(grads, groups, d_scale_norm, d_status, ws, ws_bytes=None, stream=None,
                      check=True):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    st = _lib.lora_grad_prepare(_ptr(grads), len(groups), groups, _ptr(d_scale_norm),
                                _ptr(d_status), _ptr(ws), nbytes, _stream(stream))
    return _check(st, "lora_grad_prepare") if check else st


def lora_grad_prepare_noalloc(grads, groups, d_scale_norm, d_status, stream=None, check=True):
    """lora_grad_prepare without a workspace, for callers that cannot allocate device memory (its
    scratch is a fixed device array inside the library; calls must not overlap on the GPU)."""
    st = _lib.lora_grad_prepare_noalloc(_ptr(grads), len(groups), groups, _ptr(d_scale_norm),
                                        _ptr(d_status), _stream(stream))
    return _check(st, "lora_grad_prepare_noalloc") if check else st


def make_hp(beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, plus_ratio=1.0) -> lora_adamw_hp:
    return lora_adamw_hp(beta1, beta2, eps, weight_decay, plus_ratio)


def lora_adamw_step(params, grads, m, v, groups, hp: lora_adamw_hp, d_scale_norm, d_status,
                    zero_grads=False, stream=None, check=True):
    st = _lib.lora_adamw_step(_ptr(params), _ptr(grads), _ptr(m), _ptr(v), len(groups), groups,
                              C.byref(hp), _ptr(d_scale_norm), _ptr(d_status),
                              1 if zero_grads else 0, _stream(stream))
    return _check(st, "lora_adamw_step") if check else st


def lora_snapshot(params, snap, groups, stream=None, check=True):
    """snap = params over the groups' ranges (best-weights snapshot)."""
    st = _lib.lora_snapshot(_ptr(params), _ptr(snap), len(groups), groups, _stream(stream))
    return _check(st, "lora_snapshot") if check else st


def lora_restore(params, snap, grads, m, v, groups, zero_grads=False, stream=None, check=True):
    """params = snap and m = v = 0 (optimizer reset) over the groups' ranges; grads = 0 too when
    zero_grads. The caller restarts the groups' step counts."""
    st = _lib.lora_restore(_ptr(params), _ptr(snap), _ptr(grads), _ptr(m), _ptr(v), len(groups),
                           groups, 1 if zero_grads else 0, _stream(stream))
    return _check(st, "lora_restore") if check else st


def lora_retire(params, grads, m, v, groups, clear_params=False, stream=None, check=True):
    """grads = m = v = 0 over the groups' ranges (retired slots); params = 0 too when
    clear_params."""
    st = _lib.lora_retire(_ptr(params), _ptr(grads), _ptr(m), _ptr(v), len(groups), groups,
                          1 if clear_params else 0, _stream(stream))
    return _check(st, "lora_retire") if check else st


def lora_quantize_e4m3(src, codes, scales, stream=None, check=True):
    """Test hook: per-row E4M3 codes and scales of a bf16 [rows, K] matrix."""
    rows, K = src.shape
    st = _lib.lora_quantize_e4m3(_ptr(src), rows, K, _ptr(codes), _ptr(scales), _stream(stream))
    return _check(st, "lora_quantize_e4m3") if check else st


def make_slots(slots: Sequence[dict]):
    arr = (lora_slot * len(slots))()
    for i, s in enumerate(slots):
        arr[i] = lora_slot(_ptr(s["A"]), _ptr(s["B"]), _ptr(s.get("dA")), _ptr(s.get("dB")),
                           s["rank"], s["scale"])
    return arr


def multi_lora_workspace_size(d: lora_desc, T: int, n_seg: int, slots) -> int:
    return _lib.multi_lora_workspace_size(C.byref(d), T, n_seg, len(slots), slots)


def make_projs(projs: Sequence[dict]):
    arr = (lora_proj * len(projs))()
    for i, p in enumerate(projs):
        arr[i] = lora_proj(_ptr(p["A"]), _ptr(p["B"]), _ptr(p.get("dA")), _ptr(p.get("dB")),
                           p["out"])
    return arr


def lora_fused_workspace_size(d: lora_desc, T: int, projs) -> int:
    return _lib.lora_fused_workspace_size(C.byref(d), T, len(projs), projs)


def lora_fused_forward(d, c, T, X, W, W_prep, projs, Y, H_save, ws, ws_bytes=None, stream=None,
                       check=True):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    st = _lib.lora_fused_forward(C.byref(d), C.byref(c) if c is not None else None, T, _ptr(X),
                                 _ptr(W), _ptr(W_prep), len(projs), projs, _ptr(Y), _ptr(H_save),
                                 _ptr(ws), nbytes, _stream(stream))
    return _check(st, "lora_fused_forward") if check else st


def lora_fused_backward(d, c, T, X, W_prep, projs, dY, H_save, dX, ws, ws_bytes=None,
                        stream=None, check=True):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    st = _lib.lora_fused_backward(C.byref(d), C.byref(c) if c is not None else None, T,
                                  _ptr(X), _ptr(W_prep), len(projs), projs, _ptr(dY),
                                  _ptr(H_save), _ptr(dX), _ptr(ws), nbytes, _stream(stream))
    return _check(st, "lora_fused_backward") if check else st


def multi_lora_forward(d, c, T, X, W, W_prep, n_seg, seg_start, seg_slot, slots, Y, H_save, ws,
                       ws_bytes=None, stream=None, check=True):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    st = _lib.multi_lora_forward(C.byref(d), C.byref(c) if c is not None else None, T, _ptr(X),
                                 _ptr(W), _ptr(W_prep), n_seg, _ptr(seg_start), _ptr(seg_slot), len(slots),
                                 slots, _ptr(Y), _ptr(H_save), _ptr(ws), nbytes, _stream(stream))
    return _check(st, "multi_lora_forward") if check else st


def multi_lora_backward(d, c, T, X, W_prep, n_seg, seg_start, seg_slot, slots, dY, H_save, dX, ws,
                        ws_bytes=None, stream=None, check=True):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    st = _lib.multi_lora_backward(C.byref(d), C.byref(c) if c is not None else None, T, _ptr(X),
                                  _ptr(W_prep), n_seg, _ptr(seg_start), _ptr(seg_slot), len(slots),
                                  slots, _ptr(dY), _ptr(H_save), _ptr(dX), _ptr(ws), nbytes,
                                  _stream(stream))
    return _check(st, "multi_lora_backward") if check else st


def multi_lora_plan_size(T: int, n_seg: int, n_slots: int) -> int:
    return _lib.multi_lora_plan_size(T, n_seg, n_slots)


def multi_lora_plan_build(T, n_seg, seg_start, seg_slot, n_slots, plan, plan_bytes=None,
                          stream=None, check=True):
    nbytes = plan_bytes if plan_bytes is not None else plan.numel() * plan.element_size()
    st = _lib.multi_lora_plan_build(T, n_seg, _ptr(seg_start), _ptr(seg_slot), n_slots,
                                    _ptr(plan), nbytes, _stream(stream))
    return _check(st, "multi_lora_plan_build") if check else st


def multi_lora_forward_planned(d, c, T, n_seg, plan, X, W, W_prep, slots, Y, H_save, ws,
                               ws_bytes=None, stream=None, check=True):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    st = _lib.multi_lora_forward_planned(C.byref(d), C.byref(c) if c is not None else None, T,
                                         n_seg, _ptr(plan), _ptr(X), _ptr(W), _ptr(W_prep),
                                         len(slots), slots, _ptr(Y), _ptr(H_save), _ptr(ws),
                                         nbytes, _stream(stream))
    return _check(st, "multi_lora_forward_planned") if check else st


def multi_lora_backward_planned(d, c, T, n_seg, plan, X, W_prep, slots, dY, H_save, dX, ws,
                                ws_bytes=None, stream=None, check=True):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    st = _lib.multi_lora_backward_planned(C.byref(d), C.byref(c) if c is not None else None, T,
                                          n_seg, _ptr(plan), _ptr(X), _ptr(W_prep), len(slots),
                                          slots, _ptr(dY), _ptr(H_save), _ptr(dX), _ptr(ws),
                                          nbytes, _stream(stream))
    return _check(st, "multi_lora_backward_planned") if check else st


def lora_dropout_mask(d: lora_desc, c: Optional[lora_ctx], T: int, mask, stream=None, check=True):
    st = _lib.lora_dropout_mask(C.byref(d), C.byref(c) if c is not None else None, T, _ptr(mask),
                                _stream(stream))
    return _check(st, "lora_dropout_mask") if check else st


def multi_lora_token_slots(T, n_seg, seg_start, seg_slot, n_slots, token_slot, stream=None,
                           check=True):
    st = _lib.multi_lora_token_slots(T, n_seg, _ptr(seg_start), _ptr(seg_slot), n_slots,
                                     _ptr(token_slot), _stream(stream))
    return _check(st, "multi_lora_token_slots") if check else st


def lora_profile_arm(kernel_class: int, start_events: Sequence, stop_events: Sequence):
    """Bracket the next len(start_events) launches of one kernel class with torch.cuda.Event
    pairs (recorded on the launching stream)."""
    n = len(start_events)
    if any(not e.cuda_event for e in list(start_events) + list(stop_events)):
        raise ValueError("lora_profile_arm: record each event once first (torch creates the "
                         "CUDA event lazily)")
    starts = (C.c_void_p * max(n, 1))(*[e.cuda_event for e in start_events])
    stops = (C.c_void_p * max(n, 1))(*[e.cuda_event for e in stop_events])
    return _check(_lib.lora_profile_arm(kernel_class, starts, stops, n), "lora_profile_arm")


def lora_profile_used() -> int:
    return _lib.lora_profile_used()


def lora_launch_counter() -> int:
    return _lib.lora_launch_counter()


def lora_device_check(stream=None) -> int:
    """Synchronise the stream and return the device status (LORA_OK, or LORA_ERR_TIMEOUT when a
    kernel's pipeline wait ran out of its bound) without raising."""
    return _lib.lora_device_check(_stream(stream))


def lora_set_wait_limit(cycles: int) -> None:
    """Test hook: bound of the frozen products' pipeline waits (0 = the default)."""
    _check(_lib.lora_set_wait_limit(int(cycles)), "lora_set_wait_limit")


def lora_device_error(reset: bool = False) -> int:
    """Device error bits of the tensor-core products (0 = none); synchronous."""
    v = C.c_uint32(0)
    _check(_lib.lora_device_error(C.byref(v), 1 if reset else 0), "lora_device_error")
    return v.value
