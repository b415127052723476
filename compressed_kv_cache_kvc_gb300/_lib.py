"""ctypes declarations of the C ABI in ``include/kvc.h`` (argument marshalling
only).  Loading fails loudly when ``libkvc.so`` has not been built: there is
no fallback implementation."""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvc.so")

KVC_OK = 0
KVC_ERR_INVALID_ARG = 1
KVC_ERR_UNSUPPORTED = 2
KVC_ERR_CAPACITY = 3
KVC_ERR_CUDA = 4
KVC_ERR_DEVICE = 5
KVC_ERR_STATE = 6

KVC_VERSION = 400  # the header this binding's structures and signatures follow
KVC_ATTN_ACCUM_H2O = 0x1
KVC_CODES_INT = 0
KVC_CODES_E4M3 = 1
KVC_EVICT_H2O = 0
KVC_EVICT_STREAMING = 1
KVC_EVICT_BLOCK = 2
KVC_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

BUF = dict(K_CODES=0, V_CODES=1, K_SCALE=2, V_SCALE=3, SLOT_POS=4, SCORE=5, SINK_K=6, SINK_V=7,
           SINK_SCORE=8, BLOCK_TABLE=9, SEQ_SLOTS=10, SEQ_POS=11, FREE_STACK=12, COUNTERS=13, PLAN=14,
           RING_K=15, RING_V=16, RING_SCORE=17)


class KvcConfig(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("bf16_window", ctypes.c_int32), ("codes", ctypes.c_int32)]


class KvcEvictParams(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("budget", ctypes.c_int32), ("recent", ctypes.c_int32),
                ("window", ctypes.c_int32), ("retention", ctypes.c_double)]


class KvcError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int32
_SZ = ctypes.c_size_t

_SIGS = {
    "kvc_version": (_I, []),
    "kvc_status_string": (ctypes.c_char_p, [_I]),
    "kvc_state_bytes": (_SZ, [ctypes.POINTER(KvcConfig)]),
    "kvc_cache_create": (_I, [ctypes.POINTER(KvcConfig), _P, _SZ, ctypes.POINTER(_P)]),
    "kvc_cache_destroy": (None, [_P]),
    "kvc_cache_reset": (_I, [_P, _P, _P]),
    "kvc_cache_buffer": (_I, [_P, _I, ctypes.POINTER(_P), ctypes.POINTER(_SZ)]),
    "kvc_cache_lengths": (_I, [_P, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "kvc_cache_sync_host": (_I, [_P, _P]),
    "kvc_release_sequences": (_I, [_P, _I, _I, _P]),
    "kvc_workspace_bytes": (_SZ, [_P, _I]),
    "kvc_quantize_append": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "kvc_decode_attention": (_I, [_P, _I, _I, _P, _P, ctypes.c_float, _I, _P, _SZ, _P]),
    "kvc_h2o_select_evict": (_I, [_P, _I, _I, ctypes.POINTER(KvcEvictParams), _P, _P, _SZ, _P]),
    "kvc_compact_blocks": (_I, [_P, _I, _I, _P, _P, _SZ, _P]),
    "kvc_decode_step": (_I, [_P, _I, _I, _P, _P, _P, _P, ctypes.c_float, ctypes.POINTER(KvcEvictParams), _P, _SZ, _P]),
    "kvc_decode_step_overlap": (_I, [_P, _I, _I, _P, _P, _P, _P, ctypes.c_float, ctypes.POINTER(KvcEvictParams), _P,
                                     _SZ, _P, _P]),
    "kvc_decode_attention_noalloc": (_I, [_P, _I, _I, _P, _P, ctypes.c_float, _I, _P]),
    "kvc_prefill_workspace_bytes": (_SZ, [_P, _I, _I]),
    "kvc_prefill_attention": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, ctypes.c_float, _I, _P, _SZ, _P]),
    "kvc_prefill_context_workspace_bytes": (_SZ, [_P, _I, _I]),
    "kvc_prefill_context": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, ctypes.c_float, _I, _P, _SZ, _P]),
    "kvc_read_status": (_I, [_P, ctypes.POINTER(_I), _P]),
    "kvc_set_trace_events": (_I, [_P, _P, _P]),
    "kvc_last_launch_count": (_I, [_P]),
}


def lib() -> ctypes.CDLL:
    """The loaded library (raises when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        if L.kvc_version() != KVC_VERSION:
            raise RuntimeError(f"{LIB_PATH} is version {L.kvc_version()}, the binding expects {KVC_VERSION}: rebuild it")
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().kvc_status_string(status).decode()
    except Exception:  # library unavailable while formatting an error
        return "status"


def check(status: int, what: str) -> None:
    if status != KVC_OK:
        raise KvcError(status, what)
