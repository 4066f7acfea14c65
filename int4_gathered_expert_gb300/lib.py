"""ctypes binding of libe0moe (include/e0moe.h): same names, argument
marshalling only.  Every computation runs in the CUDA library; there is no
fallback.  Loading fails loudly when the library has not been built.

Arguments that are device buffers accept a torch tensor (its data_ptr() is
passed) or a raw integer address; ``None`` passes NULL.  Streams accept a
torch.cuda.Stream, an integer handle or None (the current torch stream).
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libe0moe.so")

E0_OK, E0_ERR_ARG, E0_ERR_NULL, E0_ERR_UNSUPPORTED, E0_ERR_CUDA = 0, -1, -2, -3, -4
E0_ST_SLOT_MISS, E0_ST_BAD_EXPERT, E0_ST_NONFINITE, E0_ST_TIMEOUT, E0_ST_POOL_FULL, E0_ST_INTERNAL = 1, 2, 4, 8, 16, 32
E0_ROUTE_SOFTMAX_TOPK, E0_ROUTE_SIGMOID_GROUP = 0, 1
E0_MAX_E, E0_MAX_K, E0_MAX_T_DECODE, E0_MAX_LORA_RANK = 1024, 32, 64, 64

vp = C.c_void_p
i32 = C.c_int32


class QTensor(C.Structure):
    _fields_ = [("codes", vp), ("scale", vp), ("bias", vp)]


class ExpertQ(C.Structure):
    _fields_ = [("gate", QTensor), ("up", QTensor), ("down", QTensor)]


class SlotPool(C.Structure):
    _fields_ = [("data", vp), ("slot_table", vp), ("occupant", vp),
                ("n_slots", i32), ("H", i32), ("I", i32), ("E", i32)]


class RouteParams(C.Structure):
    _fields_ = [("mode", i32), ("K", i32), ("n_groups", i32), ("topk_groups", i32),
                ("scale", C.c_float), ("logit_bias", vp)]


class SharedExpert(C.Structure):
    _fields_ = [("data", vp), ("A_gate", vp), ("B_gate", vp), ("A_up", vp), ("B_up", vp),
                ("A_down", vp), ("B_down", vp), ("rank", i32), ("alpha", C.c_float)]


class Prerouter(C.Structure):
    _fields_ = [("fc1", vp), ("b1", vp), ("fc2", vp), ("b2", vp), ("lres", vp),
                ("H", i32), ("E", i32), ("hidden", i32)]


class ExpertCache(C.Structure):
    _fields_ = [("data", C.c_void_p), ("key", C.c_void_p), ("stamp", C.c_void_p), ("map", C.c_void_p),
                ("counters", C.c_void_p), ("scratch", C.c_void_p), ("capacity", C.c_int32), ("n_keys", C.c_int32)]


class StackLayer(C.Structure):
    _fields_ = [("pool", SlotPool), ("W_router", vp), ("shared", C.POINTER(SharedExpert)),
                ("head", C.POINTER(Prerouter)), ("consumer", i32)]


class StackTrace(C.Structure):
    _fields_ = [("r", vp), ("inds", vp), ("w", vp), ("head_logits", vp), ("pred_inds", vp)]


_lib = None


def load() -> C.CDLL:
    """Load libe0moe.so; raises if it is missing (no CPU fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libe0moe.so is not built ({LIB_PATH}); run int4_gathered_expert_gb300.build")
    lib = C.CDLL(LIB_PATH)
    sz = C.c_size_t
    P = C.POINTER
    sig = {
        "e0_slot_bytes": (sz, [C.c_int, C.c_int]),
        "e0_workspace_size": (sz, [C.c_int] * 6),
        "e0_pack_experts": (C.c_int, [P(ExpertQ), C.c_int, P(SlotPool), P(i32), P(i32), vp]),
        "e0_slot_update": (C.c_int, [P(SlotPool), vp, C.c_int, vp, C.c_int, vp, vp, vp]),
        "e0_route_softmax_topk": (C.c_int, [vp, C.c_int, C.c_int, C.c_int, vp, vp, vp, vp]),
        "e0_route_sigmoid_group": (C.c_int, [vp, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_float,
                                             vp, vp, vp, vp]),
        "e0_rmsnorm": (C.c_int, [vp, C.c_int, C.c_int, C.c_float, vp, vp]),
        "e0_moe_block_forward": (C.c_int, [vp, C.c_int, P(SlotPool), vp, P(RouteParams), vp, vp,
                                           P(SharedExpert), vp, vp, vp, vp, sz, vp, vp]),
        "e0_moe_block_forward_noalloc": (C.c_int, [vp, C.c_int, P(SlotPool), vp, P(RouteParams), vp, vp,
                                                   P(SharedExpert), vp, vp, vp, vp, vp]),
        "e0_prerouter_forward": (C.c_int, [vp, C.c_int, vp, vp, P(Prerouter), P(RouteParams), vp, vp, vp,
                                           vp, sz, vp, vp]),
        "e0_stack_workspace_size": (sz, [C.c_int] * 6),
        "e0_stack_prepare": (C.c_int, [P(StackLayer), C.c_int, C.c_int, C.c_int, C.c_int, P(RouteParams),
                                       vp, sz, vp]),
        "e0_stack_step": (C.c_int, [vp, vp, vp, P(StackTrace), C.c_int, vp, vp]),
        "e0_stack_step_range": (C.c_int, [vp, vp, vp, C.c_int, C.c_int, P(StackTrace), vp, vp]),
        "e0_stack_update_layers": (C.c_int, [vp, P(StackLayer), C.c_int, vp]),
        "e0_stack_prefetch_experts": (C.c_int, [vp, C.c_int, C.c_int, P(SlotPool), vp, vp, vp]),
        "e0_stack_prefetch_experts_batch": (C.c_int, [vp, P(i32), C.c_int, C.c_int, P(SlotPool), P(vp), vp, vp]),
        "e0_stack_prefetch_experts_cached": (C.c_int, [vp, C.c_int, C.c_int, P(SlotPool), vp, P(ExpertCache), vp,
                                                       vp]),
        "e0_stack_prefetch_experts_cached_batch": (C.c_int, [vp, P(i32), C.c_int, C.c_int, P(SlotPool), P(vp),
                                                             P(ExpertCache), vp, vp]),
        "e0_prefill_sort": (C.c_int, [vp, C.c_int, C.c_int, C.c_int, vp, vp, vp, vp, sz, vp]),
        "e0_moe_prefill_forward": (C.c_int, [vp, C.c_int, P(SlotPool), vp, P(RouteParams), vp, vp, vp,
                                             vp, sz, vp, vp]),
        "e0_selftest_bounded_wait": (C.c_int, [vp, C.c_uint32, vp, vp]),
        "e0_read_status": (C.c_int, [vp, P(C.c_uint32), vp]),
        "e0_status_string": (C.c_char_p, [C.c_int]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def exported_symbols():
    """Names of the C entry points this binding declares."""
    return ["e0_slot_bytes", "e0_workspace_size", "e0_pack_experts", "e0_slot_update", "e0_route_softmax_topk",
            "e0_route_sigmoid_group", "e0_rmsnorm", "e0_moe_block_forward", "e0_moe_block_forward_noalloc",
            "e0_prerouter_forward",
            "e0_stack_workspace_size", "e0_stack_prepare", "e0_stack_step", "e0_stack_step_range",
            "e0_stack_update_layers", "e0_stack_prefetch_experts", "e0_stack_prefetch_experts_batch",
            "e0_stack_prefetch_experts_cached", "e0_stack_prefetch_experts_cached_batch",
            "e0_prefill_sort",
            "e0_moe_prefill_forward", "e0_selftest_bounded_wait", "e0_read_status", "e0_status_string"]


# ---------------------------------------------------------------- marshalling


def ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def stream_handle(s=None) -> Optional[int]:
    import torch
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


class E0Error(RuntimeError):
    def __init__(self, name, code):
        lib = load()
        super().__init__(f"{name} returned {code}: {lib.e0_status_string(code).decode()}")
        self.code = code


def _check(name, rc, raise_on_error):
    if raise_on_error and rc != E0_OK:
        raise E0Error(name, rc)
    return rc


def route_params(mode=E0_ROUTE_SOFTMAX_TOPK, K=4, n_groups=1, topk_groups=1, scale=1.0, logit_bias=None):
    """The routing parameters as the C ABI takes them.  The struct holds only
    the device address of ``logit_bias``, so it also keeps a reference to the
    tensor: a temporary passed here stays allocated as long as the struct."""
    rp = RouteParams(mode, K, n_groups, topk_groups, scale, ptr(logit_bias))
    rp._logit_bias = logit_bias
    return rp


# ---------------------------------------------------------------- entry points (same names)


def e0_slot_bytes(H, I):
    return load().e0_slot_bytes(H, I)


def e0_workspace_size(op, T, H, I, E, K):
    return load().e0_workspace_size(op, T, H, I, E, K)


def e0_pack_experts(src_list, pool: SlotPool, dst_slots, expert_ids=None, stream=None, raise_on_error=True):
    n = len(src_list)
    arr = (ExpertQ * n)(*src_list)
    slots = (i32 * n)(*[int(s) for s in dst_slots])
    ids = (i32 * n)(*[int(e) for e in expert_ids]) if expert_ids is not None else None
    rc = load().e0_pack_experts(arr, n, C.byref(pool), slots, ids, stream_handle(stream))
    return _check("e0_pack_experts", rc, raise_on_error)


def e0_slot_update(pool: SlotPool, inds_next, n_next, inds_cur, n_cur, bank, status=None, stream=None,
                   raise_on_error=True):
    rc = load().e0_slot_update(C.byref(pool), ptr(inds_next), n_next, ptr(inds_cur), n_cur, ptr(bank),
                               ptr(status), stream_handle(stream))
    return _check("e0_slot_update", rc, raise_on_error)


def e0_route_softmax_topk(logits, T, E, K, inds, w, status=None, stream=None, raise_on_error=True):
    rc = load().e0_route_softmax_topk(ptr(logits), T, E, K, ptr(inds), ptr(w), ptr(status), stream_handle(stream))
    return _check("e0_route_softmax_topk", rc, raise_on_error)


def e0_route_sigmoid_group(logits, T, E, n_groups, topk_groups, K, s, inds, w, status=None, stream=None,
                           raise_on_error=True):
    rc = load().e0_route_sigmoid_group(ptr(logits), T, E, n_groups, topk_groups, K, s, ptr(inds), ptr(w),
                                       ptr(status), stream_handle(stream))
    return _check("e0_route_sigmoid_group", rc, raise_on_error)


def e0_rmsnorm(r, T, H, eps, h, stream=None, raise_on_error=True):
    rc = load().e0_rmsnorm(ptr(r), T, H, eps, ptr(h), stream_handle(stream))
    return _check("e0_rmsnorm", rc, raise_on_error)


def e0_moe_block_forward(x, T, pool: SlotPool, W_router, rp: RouteParams, inds_in, w_in, shared, y, inds_out,
                         w_out, ws, ws_bytes, status=None, stream=None, raise_on_error=True):
    sh = C.byref(shared) if shared is not None else None
    rc = load().e0_moe_block_forward(ptr(x), T, C.byref(pool), ptr(W_router), C.byref(rp), ptr(inds_in),
                                     ptr(w_in), sh, ptr(y), ptr(inds_out), ptr(w_out), ptr(ws), ws_bytes,
                                     ptr(status), stream_handle(stream))
    return _check("e0_moe_block_forward", rc, raise_on_error)


def e0_moe_block_forward_noalloc(x, T, pool: SlotPool, W_router, rp: RouteParams, inds_in, w_in, shared, y,
                                 inds_out, w_out, status=None, stream=None, raise_on_error=True):
    """e0_moe_block_forward without a workspace: the library's fixed scratch
    array is used instead (see the header for its size and sharing rules)."""
    sh = C.byref(shared) if shared is not None else None
    rc = load().e0_moe_block_forward_noalloc(ptr(x), T, C.byref(pool), ptr(W_router), C.byref(rp), ptr(inds_in),
                                             ptr(w_in), sh, ptr(y), ptr(inds_out), ptr(w_out), ptr(status),
                                             stream_handle(stream))
    return _check("e0_moe_block_forward_noalloc", rc, raise_on_error)


def e0_prerouter_forward(h, T, inds_cur, inds_prev, head: Prerouter, rp: RouteParams, logits_out, inds_next,
                         w_next, ws, ws_bytes, status=None, stream=None, raise_on_error=True):
    rc = load().e0_prerouter_forward(ptr(h), T, ptr(inds_cur), ptr(inds_prev), C.byref(head), C.byref(rp),
                                     ptr(logits_out), ptr(inds_next), ptr(w_next), ptr(ws), ws_bytes,
                                     ptr(status), stream_handle(stream))
    return _check("e0_prerouter_forward", rc, raise_on_error)


def e0_stack_workspace_size(L, H, I, E, K, head_hidden):
    return load().e0_stack_workspace_size(L, H, I, E, K, head_hidden)


def e0_stack_prepare(layers, H, I, E, rp: RouteParams, ws, ws_bytes, stream=None, raise_on_error=True):
    arr = (StackLayer * len(layers))(*layers)
    rc = load().e0_stack_prepare(arr, len(layers), H, I, E, C.byref(rp), ptr(ws), ws_bytes, stream_handle(stream))
    return _check("e0_stack_prepare", rc, raise_on_error)


def e0_stack_step(x, r_out, ws, trace: Optional[StackTrace] = None, impl=0, status=None, stream=None,
                  raise_on_error=True):
    tr = C.byref(trace) if trace is not None else None
    rc = load().e0_stack_step(ptr(x), ptr(r_out), ptr(ws), tr, impl, ptr(status), stream_handle(stream))
    return _check("e0_stack_step", rc, raise_on_error)


def e0_stack_step_range(x, r_out, ws, layer_begin, layer_end, trace: Optional[StackTrace] = None, status=None,
                        stream=None, raise_on_error=True):
    tr = C.byref(trace) if trace is not None else None
    rc = load().e0_stack_step_range(ptr(x), ptr(r_out), ptr(ws), int(layer_begin), int(layer_end), tr, ptr(status),
                                    stream_handle(stream))
    return _check("e0_stack_step_range", rc, raise_on_error)


def e0_stack_update_layers(ws, layers, stream=None, raise_on_error=True):
    arr = (StackLayer * len(layers))(*layers)
    rc = load().e0_stack_update_layers(ptr(ws), arr, len(layers), stream_handle(stream))
    return _check("e0_stack_update_layers", rc, raise_on_error)


def e0_stack_prefetch_experts_batch(ws, layers, t_next, pools, banks, status=None, stream=None, raise_on_error=True):
    n = len(layers)
    la = (i32 * max(n, 1))(*[int(l) for l in layers])
    pa = (SlotPool * max(n, 1))(*pools)
    ba = (vp * max(n, 1))(*[ptr(b) for b in banks])
    rc = load().e0_stack_prefetch_experts_batch(ptr(ws), la, n, int(t_next), pa, ba, ptr(status), stream_handle(stream))
    return _check("e0_stack_prefetch_experts_batch", rc, raise_on_error)


def e0_stack_prefetch_experts_cached_batch(ws, layers, t_next, pools, banks, cache, status=None, stream=None,
                                           raise_on_error=True):
    n = len(layers)
    la = (i32 * max(n, 1))(*[int(l) for l in layers])
    pa = (SlotPool * max(n, 1))(*pools)
    ba = (vp * max(n, 1))(*[ptr(b) for b in banks])
    rc = load().e0_stack_prefetch_experts_cached_batch(ptr(ws), la, n, int(t_next), pa, ba, C.byref(cache), ptr(status),
                                                       stream_handle(stream))
    return _check("e0_stack_prefetch_experts_cached_batch", rc, raise_on_error)


def e0_stack_prefetch_experts(ws, layer, t_next, pool: SlotPool, bank, status=None, stream=None, raise_on_error=True):
    rc = load().e0_stack_prefetch_experts(ptr(ws), int(layer), int(t_next), C.byref(pool), ptr(bank), ptr(status),
                                          stream_handle(stream))
    return _check("e0_stack_prefetch_experts", rc, raise_on_error)


def e0_stack_prefetch_experts_cached(ws, layer, t_next, pool: SlotPool, bank, cache: ExpertCache, status=None,
                                     stream=None, raise_on_error=True):
    rc = load().e0_stack_prefetch_experts_cached(ptr(ws), int(layer), int(t_next), C.byref(pool), ptr(bank),
                                                 C.byref(cache), ptr(status), stream_handle(stream))
    return _check("e0_stack_prefetch_experts_cached", rc, raise_on_error)


def e0_prefill_sort(inds, T, K, E, counts, offsets, perm, ws, ws_bytes, stream=None, raise_on_error=True):
    rc = load().e0_prefill_sort(ptr(inds), T, K, E, ptr(counts), ptr(offsets), ptr(perm), ptr(ws), ws_bytes,
                                stream_handle(stream))
    return _check("e0_prefill_sort", rc, raise_on_error)


def e0_moe_prefill_forward(X, T, bank: SlotPool, W_router, rp: RouteParams, Y, inds_out, w_out, ws, ws_bytes,
                           status=None, stream=None, raise_on_error=True):
    rc = load().e0_moe_prefill_forward(ptr(X), T, C.byref(bank), ptr(W_router), C.byref(rp), ptr(Y),
                                       ptr(inds_out), ptr(w_out), ptr(ws), ws_bytes, ptr(status),
                                       stream_handle(stream))
    return _check("e0_moe_prefill_forward", rc, raise_on_error)


E0_SELFTEST_MAX_WAIT_US = 2000000


def e0_selftest_bounded_wait(flag, limit_us, status, stream=None, raise_on_error=True):
    rc = load().e0_selftest_bounded_wait(ptr(flag), int(limit_us), ptr(status), stream_handle(stream))
    return _check("e0_selftest_bounded_wait", rc, raise_on_error)


def e0_read_status(status, stream=None) -> int:
    out = C.c_uint32(0)
    rc = load().e0_read_status(ptr(status), C.byref(out), stream_handle(stream))
    if rc != E0_OK:
        raise E0Error("e0_read_status", rc)
    return int(out.value)


def e0_status_string(code) -> str:
    return load().e0_status_string(code).decode()
