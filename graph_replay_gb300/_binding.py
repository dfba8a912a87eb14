"""ctypes binding of libgraphdec.so (include/graphdec.h): argument marshalling
only.  Every step of the decode path runs in the library's CUDA kernels; there
is no fallback.  If the library has not been built, importing this module
raises ImportError."""
from __future__ import annotations

import ctypes
import os

from . import build as _build

DEC_OK = 0
DEC_E_INVALID = 1
DEC_E_UNSUPPORTED = 2
DEC_E_RANGE = 3
DEC_E_STATE = 4
DEC_E_CUDA = 5
DEC_E_OOM = 6
DEC_E_DEVICE_FAULT = 7
DEC_E_NEEDS_RESET = 8
DEC_E_POISONED = 9
DEC_E_TIMEOUT = 10

DEC_FAULT_TOKEN = 0x1
DEC_FAULT_POS = 0x2
DEC_FAULT_WRITE_MAP = 0x4
DEC_FAULT_SLOT_MAP = 0x8
DEC_FAULT_WAIT = 0x10

DEC_DTYPE_F32 = 0
DEC_DTYPE_BF16 = 1
DEC_KV_CONTIGUOUS = 0
DEC_KV_PAGED = 1
DEC_STRATEGY_GRAPH = 0
DEC_STRATEGY_PERSISTENT = 1
DEC_SWEEP_CAP = 0
DEC_SWEEP_POS = 1

(DEC_W_EMBED, DEC_W_ATTN_NORM, DEC_W_Q, DEC_W_K, DEC_W_V, DEC_W_O, DEC_W_FFN_NORM, DEC_W_GATE, DEC_W_UP,
 DEC_W_DOWN, DEC_W_FINAL_NORM, DEC_W_LM_HEAD) = range(12)


class dec_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn_hidden", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("weight_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("device", ctypes.c_int32), ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
                ("wait_timeout_ms", ctypes.c_int64)]


class dec_weight(ctypes.Structure):
    _fields_ = [("role", ctypes.c_int32), ("layer", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("data", ctypes.c_void_p)]


class dec_stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("replays", ctypes.c_int64), ("eager_steps", ctypes.c_int64),
                ("kernels_per_step", ctypes.c_int32), ("graph_nodes", ctypes.c_int32),
                ("attn_splits", ctypes.c_int32), ("attn_split_len", ctypes.c_int32),
                ("last_fault", ctypes.c_uint32), ("state", ctypes.c_int32), ("captured", ctypes.c_int32),
                ("rows", ctypes.c_int32), ("cap", ctypes.c_int32), ("kv_layout", ctypes.c_int32),
                ("strategy", ctypes.c_int32), ("reserved", ctypes.c_int32), ("last_step_us", ctypes.c_double), ("workspace_bytes", ctypes.c_int64),
                ("kv_bytes", ctypes.c_int64)]


# every symbol the header declares: (name, restype, argtypes)
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SIG = [
    ("dec_init", ctypes.c_int, [ctypes.POINTER(dec_config), ctypes.POINTER(_P)]),
    ("dec_load_weights", ctypes.c_int, [_P, ctypes.POINTER(dec_weight), ctypes.c_size_t]),
    ("dec_workspace_size", ctypes.c_int, [ctypes.POINTER(dec_config), _I32, _I32, _I32, _I32, _I32,
                                          ctypes.POINTER(ctypes.c_size_t)]),
    ("dec_capture", ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _I32, _P, ctypes.c_size_t, _P]),
    ("dec_set_slot_map", ctypes.c_int, [_P, _P]),
    ("dec_step", ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P]),
    ("dec_launch", ctypes.c_int, [_P, _P]),
    ("dec_wait", ctypes.c_int, [_P, _P, _P, _P]),
    ("dec_chain", ctypes.c_int, [_P, _I32, _P, _P, _P, _P]),
    ("dec_prefill", ctypes.c_int, [_P, _P, _P, _I32, _I32, _P, _P]),
    ("dec_prefill_block", ctypes.c_int, [_P, _I32, _P, _P, _I32, _I32, _P, _P]),
    ("dec_set_sampler", ctypes.c_int, [_P, _P]),
    ("dec_logprobs", ctypes.c_int, [_P, _I32, _P, _P]),
    ("dec_set_strategy", ctypes.c_int, [_P, _I32]),
    ("dec_set_kv_sweep", ctypes.c_int, [_P, _I32]),
    ("dec_set_eager", ctypes.c_int, [_P, _I32]),
    ("dec_reset_state", ctypes.c_int, [_P]),
    ("dec_kv_ptr", ctypes.c_int, [_P, _I32, _I32, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)]),
    ("dec_attention", ctypes.c_int, [_P, _I32, _P, _P, _P]),
    ("dec_attention_static", ctypes.c_int, [_P, _I32, _P, _P, _P]),
    ("dec_logits_ptr", ctypes.c_int, [_P, ctypes.POINTER(_P)]),
    ("dec_stream", ctypes.c_int, [_P, ctypes.POINTER(_P)]),
    ("dec_stats_get", ctypes.c_int, [_P, ctypes.POINTER(dec_stats)]),
    ("dec_slot_map_ptr", ctypes.c_int, [_P, ctypes.POINTER(_P)]),
    ("dec_launch_kernel", ctypes.c_int, [_P, _I32, _I32, ctypes.POINTER(_I64)]),
    ("dec_trace", ctypes.c_int, [_P, _I32]),
    ("dec_trace_read", ctypes.c_int, [_P, _P, ctypes.c_size_t]),
    ("dec_debug_busy", ctypes.c_int, [_P, _I64]),
    ("dec_set_timeout", ctypes.c_int, [_P, _I64]),
    ("dec_debug_wait", ctypes.c_int, [_P, ctypes.c_uint32, ctypes.c_uint32, _I32, _I32]),
    ("dec_last_error", ctypes.c_char_p, [_P]),
    ("dec_status_str", ctypes.c_char_p, [ctypes.c_int]),
    ("dec_destroy", ctypes.c_int, [_P]),
]
SYMBOLS = [s[0] for s in _SIG]


def library_path() -> str:
    return _build.LIB


def load_library(path: str | None = None) -> ctypes.CDLL:
    path = path or _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libgraphdec.so is not built ({path}); run graph_replay_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, res, args in _SIG:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


class DecError(RuntimeError):
    def __init__(self, status: int, msg: str):
        self.status = status
        super().__init__(f"{status_str(status)}: {msg}")


def status_str(s: int) -> str:
    return lib().dec_status_str(s).decode()


def last_error(h) -> str:
    m = lib().dec_last_error(h)
    return m.decode() if m else ""


def check(h, status: int) -> int:
    if status != DEC_OK:
        raise DecError(status, last_error(h))
    return status


# ---- one Python function per C entry point, same names ----

def dec_init(cfg: dec_config) -> int:
    h = ctypes.c_void_p()
    rc = lib().dec_init(ctypes.byref(cfg), ctypes.byref(h))
    if rc != DEC_OK:
        raise DecError(rc, last_error(None))
    return h.value


def dec_load_weights(h, bindings) -> None:
    arr = (dec_weight * len(bindings))(*bindings)
    check(h, lib().dec_load_weights(h, arr, len(bindings)))


def dec_workspace_size(cfg: dec_config, cap, rows, kv_layout, page_size=0, num_pages=0) -> int:
    n = ctypes.c_size_t()
    rc = lib().dec_workspace_size(ctypes.byref(cfg), cap, rows, kv_layout, page_size, num_pages, ctypes.byref(n))
    if rc != DEC_OK:
        raise DecError(rc, "dec_workspace_size")
    return n.value


def dec_capture(h, cap, rows, kv_layout, page_size=0, num_pages=0, workspace=None, workspace_bytes=0,
                stream=None) -> None:
    check(h, lib().dec_capture(h, cap, rows, kv_layout, page_size, num_pages, workspace, workspace_bytes, stream))


def dec_set_slot_map(h, map_ptr) -> int:
    return lib().dec_set_slot_map(h, map_ptr)


def dec_step(h, tokens_ptr, pos_ptr, write_map_ptr, logits_ptr, ids_ptr, nonfinite_ptr) -> int:
    return lib().dec_step(h, tokens_ptr, pos_ptr, write_map_ptr, logits_ptr, ids_ptr, nonfinite_ptr)


def dec_launch(h, dev_slots_ptr) -> int:
    return lib().dec_launch(h, dev_slots_ptr)


def dec_wait(h, logits_ptr, ids_ptr, nonfinite_ptr) -> int:
    return lib().dec_wait(h, logits_ptr, ids_ptr, nonfinite_ptr)


def dec_chain(h, n_steps: int, tokens_ptr, pos_ptr, ids_ptr, nonfinite_ptr) -> int:
    return lib().dec_chain(h, n_steps, tokens_ptr, pos_ptr, ids_ptr, nonfinite_ptr)


DEC_CHAIN_MAX_STEPS = 4096


class dec_sampler(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float),
                ("min_p", ctypes.c_float), ("seed", ctypes.c_uint64), ("n_logprobs", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


DEC_SAMPLER_MAX_TOP_K = 1024
DEC_LOGPROBS_MAX = 8


def dec_set_sampler(h, sampler) -> int:
    return lib().dec_set_sampler(h, None if sampler is None else ctypes.byref(sampler))


def dec_logprobs(h, n: int, ids_ptr, vals_ptr) -> int:
    return lib().dec_logprobs(h, n, ids_ptr, vals_ptr)


def dec_prefill(h, pages_ptr, tokens_ptr, n: int, pos0: int, logits_ptr, id_ptr) -> int:
    return lib().dec_prefill(h, pages_ptr, tokens_ptr, n, pos0, logits_ptr, id_ptr)


def dec_prefill_block(h, row: int, pages_ptr, tokens_ptr, n: int, pos0: int, logits_ptr, id_ptr) -> int:
    return lib().dec_prefill_block(h, row, pages_ptr, tokens_ptr, n, pos0, logits_ptr, id_ptr)


def dec_set_strategy(h, strategy: int) -> None:
    check(h, lib().dec_set_strategy(h, strategy))


def dec_set_kv_sweep(h, sweep: int) -> None:
    check(h, lib().dec_set_kv_sweep(h, sweep))


def dec_set_eager(h, eager: bool) -> None:
    check(h, lib().dec_set_eager(h, 1 if eager else 0))


def dec_reset_state(h) -> int:
    return lib().dec_reset_state(h)


def dec_kv_ptr(h, layer, which):
    p = ctypes.c_void_p()
    n = ctypes.c_size_t()
    check(h, lib().dec_kv_ptr(h, layer, which, ctypes.byref(p), ctypes.byref(n)))
    return p.value, n.value


def dec_attention(h, layer: int, qkv_ptr, pos_ptr, out_ptr) -> int:
    return lib().dec_attention(h, layer, qkv_ptr, pos_ptr, out_ptr)


def dec_attention_static(h, layer: int, qkv_ptr, pos_ptr, out_ptr) -> int:
    return lib().dec_attention_static(h, layer, qkv_ptr, pos_ptr, out_ptr)


def dec_logits_ptr(h) -> int:
    p = ctypes.c_void_p()
    check(h, lib().dec_logits_ptr(h, ctypes.byref(p)))
    return p.value


def dec_stream(h) -> int:
    p = ctypes.c_void_p()
    check(h, lib().dec_stream(h, ctypes.byref(p)))
    return p.value or 0


def dec_stats_get(h) -> dec_stats:
    st = dec_stats()
    check(h, lib().dec_stats_get(h, ctypes.byref(st)))
    return st


def dec_slot_map_ptr(h) -> int:
    p = ctypes.c_void_p()
    check(h, lib().dec_slot_map_ptr(h, ctypes.byref(p)))
    return p.value


def dec_launch_kernel(h, index: int, pdl: bool = False) -> int:
    n = ctypes.c_int64()
    check(h, lib().dec_launch_kernel(h, index, 1 if pdl else 0, ctypes.byref(n)))
    return n.value


def dec_trace(h, enable: bool) -> None:
    check(h, lib().dec_trace(h, 1 if enable else 0))


def dec_trace_read(h, n_kernels: int):
    import numpy as np
    out = np.zeros(4 * n_kernels, dtype=np.uint64)
    check(h, lib().dec_trace_read(h, out.ctypes.data, n_kernels))
    return out.reshape(n_kernels, 4)


def dec_debug_busy(h, microseconds: int) -> None:
    check(h, lib().dec_debug_busy(h, microseconds))


def dec_set_timeout(h, ms: int) -> None:
    check(h, lib().dec_set_timeout(h, ms))


def dec_debug_wait(h, grid_polls: int = 0, ring_polls: int = 0, hold_phase: int = -1, drop_stage: int = -1) -> None:
    check(h, lib().dec_debug_wait(h, grid_polls, ring_polls, hold_phase, drop_stage))


def dec_destroy(h) -> int:
    return lib().dec_destroy(h)
