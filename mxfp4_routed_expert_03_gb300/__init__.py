"""Python binding of libmoe.so, the GB300 routed-expert FFN library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/moe.h``. The functions keep the
C names (``moe_create``, ``moe_plan``, ``moe_forward``, ``moe_decode``, ...);
tensors are passed as device pointers and PyTorch only provides device memory
and streams. Importing this module fails loudly if the library is missing;
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE_TIMEOUT = -5
MOE_ERR_NAN_LOGIT = -6
MOE_ERR_BAD_INDEX = -7
MOE_ERR_NOT_PREPARED = -8
MOE_ERR_CORRUPT_TILE = -9

MOE_ROUTER_LOGITS = 0
MOE_ROUTER_XWR = 1

MOE_OP_PLAN = 0
MOE_OP_FORWARD = 1
MOE_OP_DECODE = 2

# Every symbol include/moe.h declares.
EXPORTS = ("moe_create", "moe_destroy", "moe_expert_bytes", "moe_prepared_bytes", "moe_prepare",
           "moe_workspace_bytes", "moe_plan", "moe_router_logits", "moe_forward", "moe_decode",
           "moe_decode_noalloc", "moe_stream_state_bytes", "moe_create_streaming",
           "moe_stream_stats", "moe_store_tiles_per_expert", "moe_store_blob_bound",
           "moe_store_encode", "moe_store_decode", "moe_create_streaming_store",
           "moe_profile_kernel", "moe_set_fault_injection", "moe_status", "moe_strerror")

MOE_INJECT_NONE = 0
MOE_INJECT_GEMM_STALL = 1

MOE_PROF_NONE = 0
MOE_PROF_DECODE_GATEUP = 1
MOE_PROF_DECODE_DOWN = 2
MOE_PROF_FORWARD_GEMM1 = 3
MOE_PROF_FORWARD_GEMM2 = 4
MOE_PROF_ROUTER = 5
MOE_PROF_SHARED_GATEUP = 6
MOE_PROF_SHARED_DOWN = 7
MOE_PROF_STREAM_COPY = 8


MOE_ACT_EXACT = 0
MOE_ACT_MXFP4 = 1

MOE_W_MXFP4 = 0
MOE_W_FP8 = 1


class moe_desc(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("router_mode", ctypes.c_int32), ("has_shared", ctypes.c_int32),
                ("act_mode", ctypes.c_int32), ("weight_format", ctypes.c_int32)]


class moe_tile_rec(ctypes.Structure):
    _fields_ = [("offset_lo", ctypes.c_uint32), ("offset_hi", ctypes.c_uint32),
                ("n_bytes", ctypes.c_uint32), ("n_words", ctypes.c_uint32),
                ("adler", ctypes.c_uint32), ("flags", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32 * 2)]


class moe_store(ctypes.Structure):
    _fields_ = [("blob", ctypes.c_void_p), ("blob_bytes", ctypes.c_int64),
                ("tiles", ctypes.c_void_p), ("tables", ctypes.c_void_p)]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q",
                                                "down_s", "w_router", "sh_gate", "sh_up",
                                                "sh_down")]


class moe_plan_buf(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("topk_idx", "topk_w", "counts", "offsets", "perm",
                                                "inv", "active")]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        super().__init__(f"{where}: {moe_strerror(code)} ({code})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe.so (raises OSError if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with "
                          "mxfp4_routed_expert_03_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        L.moe_create.argtypes = [ctypes.POINTER(moe_desc), ctypes.POINTER(moe_weights),
                                 ctypes.POINTER(p)]
        L.moe_create.restype = ctypes.c_int
        L.moe_destroy.argtypes = [p]
        L.moe_destroy.restype = None
        L.moe_expert_bytes.argtypes = [i32, i32]
        L.moe_expert_bytes.restype = i64
        L.moe_prepared_bytes.argtypes = [p]
        L.moe_prepared_bytes.restype = sz
        L.moe_prepare.argtypes = [p, p, sz, p]
        L.moe_prepare.restype = ctypes.c_int
        L.moe_workspace_bytes.argtypes = [p, i32, i32]
        L.moe_workspace_bytes.restype = sz
        L.moe_plan.argtypes = [p, i32, p, p, ctypes.POINTER(moe_plan_buf), p, sz, p]
        L.moe_plan.restype = ctypes.c_int
        L.moe_router_logits.argtypes = [p, i32, p, p, p]
        L.moe_router_logits.restype = ctypes.c_int
        for fn in (L.moe_forward, L.moe_decode):
            fn.argtypes = [p, i32, p, ctypes.POINTER(moe_plan_buf), p, p, sz, p]
            fn.restype = ctypes.c_int
        L.moe_decode_noalloc.argtypes = [p, i32, p, ctypes.POINTER(moe_plan_buf), p, p]
        L.moe_decode_noalloc.restype = ctypes.c_int
        L.moe_profile_kernel.argtypes = [p, i32, p, p]
        L.moe_profile_kernel.restype = ctypes.c_int
        L.moe_set_fault_injection.argtypes = [p, i32, i64]
        L.moe_set_fault_injection.restype = ctypes.c_int
        L.moe_status.argtypes = [p, p]
        L.moe_status.restype = ctypes.c_int
        L.moe_strerror.argtypes = [ctypes.c_int]
        L.moe_strerror.restype = ctypes.c_char_p
        L.moe_stream_state_bytes.argtypes = [i32, i32]
        L.moe_stream_state_bytes.restype = sz
        L.moe_create_streaming.argtypes = [ctypes.POINTER(moe_desc), ctypes.POINTER(moe_weights),
                                           ctypes.POINTER(moe_weights), i32, p, ctypes.POINTER(p)]
        L.moe_create_streaming.restype = ctypes.c_int
        L.moe_stream_stats.argtypes = [p, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                       ctypes.POINTER(i32), p]
        L.moe_stream_stats.restype = ctypes.c_int
        L.moe_store_tiles_per_expert.argtypes = [i32, i32]
        L.moe_store_tiles_per_expert.restype = i32
        L.moe_store_blob_bound.argtypes = [i32, i32, i32]
        L.moe_store_blob_bound.restype = i64
        L.moe_store_encode.argtypes = [i32, i32, i32, ctypes.POINTER(moe_weights), p, i64,
                                       ctypes.POINTER(i64), p, p, i32]
        L.moe_store_encode.restype = ctypes.c_int
        L.moe_store_decode.argtypes = [i32, i32, i32, ctypes.POINTER(moe_store), p, p, i32,
                                       ctypes.POINTER(moe_weights), i32, p, p]
        L.moe_store_decode.restype = ctypes.c_int
        L.moe_create_streaming_store.argtypes = [ctypes.POINTER(moe_desc),
                                                 ctypes.POINTER(moe_store),
                                                 ctypes.POINTER(moe_weights), i32, p,
                                                 ctypes.POINTER(p)]
        L.moe_create_streaming_store.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(t) -> int | None:
    """Device pointer of a tensor (or an int pointer, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def moe_strerror(code: int) -> str:
    return lib().moe_strerror(code).decode()


def moe_expert_bytes(d_model: int, d_ff: int) -> int:
    return lib().moe_expert_bytes(d_model, d_ff)


def moe_create(desc: moe_desc, weights: moe_weights) -> int:
    h = ctypes.c_void_p()
    rc = lib().moe_create(ctypes.byref(desc), ctypes.byref(weights), ctypes.byref(h))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_create")
    return h.value


def moe_stream_state_bytes(n_experts: int, n_slots: int) -> int:
    return lib().moe_stream_state_bytes(n_experts, n_slots)


def moe_create_streaming(desc: moe_desc, host_weights: moe_weights, slot_weights: moe_weights,
                         n_slots: int, state) -> int:
    """host_weights: pinned host arrays of all experts; slot_weights: device cache arrays."""
    h = ctypes.c_void_p()
    rc = lib().moe_create_streaming(ctypes.byref(desc), ctypes.byref(host_weights),
                                    ctypes.byref(slot_weights), n_slots, _ptr(state),
                                    ctypes.byref(h))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_create_streaming")
    return h.value


def moe_store_tiles_per_expert(d_model: int, d_ff: int) -> int:
    return lib().moe_store_tiles_per_expert(d_model, d_ff)


def moe_store_blob_bound(n_experts: int, d_model: int, d_ff: int) -> int:
    return lib().moe_store_blob_bound(n_experts, d_model, d_ff)


def moe_store_encode(n_experts: int, d_model: int, d_ff: int, host_weights: moe_weights,
                     blob, blob_cap: int, tiles, tables, n_threads: int = 0) -> int:
    """Host encoder; blob, tiles, tables are host buffers (pointers or tensors).
    Returns the packed blob size."""
    nbytes = ctypes.c_int64(0)
    rc = lib().moe_store_encode(n_experts, d_model, d_ff, ctypes.byref(host_weights), _ptr(blob),
                                blob_cap, ctypes.byref(nbytes), _ptr(tiles), _ptr(tables),
                                n_threads)
    if rc != MOE_OK:
        raise MoeError(rc, "moe_store_encode")
    return nbytes.value


def moe_store_decode(n_experts: int, d_model: int, d_ff: int, store: moe_store, experts, slots,
                     n: int, slot_weights: moe_weights, n_slots: int, status, stream=None) -> int:
    return lib().moe_store_decode(n_experts, d_model, d_ff, ctypes.byref(store), _ptr(experts),
                                  _ptr(slots), n, ctypes.byref(slot_weights), n_slots,
                                  _ptr(status), _stream(stream))


def moe_create_streaming_store(desc: moe_desc, store: moe_store, slot_weights: moe_weights,
                               n_slots: int, state) -> int:
    """store: the compressed store (blob in pinned host memory, records and tables on the
    device); slot_weights: device cache arrays."""
    h = ctypes.c_void_p()
    rc = lib().moe_create_streaming_store(ctypes.byref(desc), ctypes.byref(store),
                                          ctypes.byref(slot_weights), n_slots, _ptr(state),
                                          ctypes.byref(h))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_create_streaming_store")
    return h.value


def moe_stream_stats(h, stream=None) -> tuple:
    """(hits, misses, last_misses) of a streaming handle; synchronises the stream."""
    hits, misses, last = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    rc = lib().moe_stream_stats(h, ctypes.byref(hits), ctypes.byref(misses), ctypes.byref(last),
                                _stream(stream))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_stream_stats")
    return hits.value, misses.value, last.value


def moe_destroy(h: int) -> None:
    lib().moe_destroy(h)


def moe_prepared_bytes(h: int) -> int:
    return lib().moe_prepared_bytes(h)


def moe_prepare(h, buf, nbytes, stream=None) -> int:
    return lib().moe_prepare(h, _ptr(buf), nbytes, _stream(stream))


def moe_workspace_bytes(h: int, T: int, op: int) -> int:
    return lib().moe_workspace_bytes(h, T, op)


def moe_plan(h, T, logits, x, plan: moe_plan_buf, ws, ws_bytes, stream=None) -> int:
    return lib().moe_plan(h, T, _ptr(logits), _ptr(x), ctypes.byref(plan), _ptr(ws), ws_bytes,
                          _stream(stream))


def moe_router_logits(h, T, x, logits, stream=None) -> int:
    return lib().moe_router_logits(h, T, _ptr(x), _ptr(logits), _stream(stream))


def moe_forward(h, T, x, plan: moe_plan_buf, out, ws, ws_bytes, stream=None) -> int:
    return lib().moe_forward(h, T, _ptr(x), ctypes.byref(plan), _ptr(out), _ptr(ws), ws_bytes,
                             _stream(stream))


def moe_decode(h, T, x, plan: moe_plan_buf, out, ws, ws_bytes, stream=None) -> int:
    return lib().moe_decode(h, T, _ptr(x), ctypes.byref(plan), _ptr(out), _ptr(ws), ws_bytes,
                            _stream(stream))


def moe_profile_kernel(h, which: int, ev_start=None, ev_stop=None) -> int:
    """ev_start/ev_stop: torch.cuda.Event (already recorded once) or raw cudaEvent_t."""
    def raw(e):
        if e is None or isinstance(e, int):
            return e
        return e.cuda_event
    return lib().moe_profile_kernel(h, which, raw(ev_start), raw(ev_stop))


def moe_decode_noalloc(h, T, x, plan: moe_plan_buf, out, stream=None) -> int:
    """moe_decode with the library's fixed scratch (no workspace argument)."""
    return lib().moe_decode_noalloc(h, T, _ptr(x), ctypes.byref(plan), _ptr(out), _stream(stream))


def moe_set_fault_injection(h, mode: int, timeout_cycles: int = 0) -> int:
    """Test hook: injection mode (MOE_INJECT_*) and device-wait limit in SM cycles (0: default)."""
    return lib().moe_set_fault_injection(h, mode, timeout_cycles)


def moe_status(h, stream=None) -> int:
    return lib().moe_status(h, _stream(stream))


def check(rc: int, where: str = "") -> None:
    if rc != MOE_OK:
        raise MoeError(rc, where)
