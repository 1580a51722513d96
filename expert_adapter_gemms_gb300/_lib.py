"""ctypes binding of libmoe_lora.so (the C ABI declared in include/moe_lora.h).

Argument marshalling only: tensors are checked (device, dtype, layout) and their
device pointers passed with the current CUDA stream. Every computation runs in
the library's kernels; there is no fallback path. If the library has not been
built, every call raises :class:`MoeLoraUnavailable`.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch  # loads the CUDA runtime the library links against

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_lora.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE_TOO_SMALL, ERR_TIMEOUT = range(6)
DEVERR_EXPERT_RANGE, DEVERR_ADAPTER_RANGE, DEVERR_TIMEOUT = 1, 2, 4
ALIGN_NFIELDS = 12
(AF_HEADER, AF_SORTED_SLOTS, AF_SLOT_ROW, AF_ROW_EXPERT, AF_ROW_ADAPTER, AF_EXPERT_BEGIN,
 AF_TILES, AF_LORA_BLOCKS, AF_MAX_TILES, AF_MAX_LORA_BLOCKS, AF_SCRATCH, AF_TOTAL_BYTES) = range(12)
LAYER_NUM_STAGES = 9
LAYER_STAGE_NAMES = ["route", "align", "gather", "gate_up_gemm", "gate_up_shrink",
                     "gate_up_expand_swiglu", "down_gemm", "down_shrink", "down_expand_combine"]


class MoeLoraUnavailable(RuntimeError):
    """The compiled library is missing; build it first (no fallback exists)."""


class MoeLoraError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


class AlignDesc(ctypes.Structure):
    _fields_ = [("buf", ctypes.c_void_p), ("T", ctypes.c_int32), ("k", ctypes.c_int32),
                ("E", ctypes.c_int32), ("L", ctypes.c_int32), ("bm_base", ctypes.c_int32),
                ("bm_lora", ctypes.c_int32), ("adapter_ranks", ctypes.c_void_p)]


class LayerOpts(ctypes.Structure):
    _fields_ = [("bm_base", ctypes.c_int32), ("bm_lora", ctypes.c_int32),
                ("disable_pdl", ctypes.c_int32), ("num_events", ctypes.c_int32),
                ("events", ctypes.POINTER(ctypes.c_void_p)), ("adapter_ranks", ctypes.c_void_p),
                ("gate_up_slices", ctypes.c_int32), ("expand_mode", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_int64), ("mma_pairs", ctypes.c_int32)]


class LayerPlan(ctypes.Structure):
    _fields_ = [("bm_base", ctypes.c_int32), ("bm_lora", ctypes.c_int32),
                ("expert_major_rows", ctypes.c_int32), ("fused_expand", ctypes.c_int32),
                ("launches", ctypes.c_int32), ("early_reads", ctypes.c_int32),
                ("route_in_align", ctypes.c_int32)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_AP = ctypes.POINTER(AlignDesc)

# name -> (restype, argtypes)
SIGNATURES = {
    "moe_lora_status_string": (ctypes.c_char_p, [_I]),
    "moe_topk_softmax": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_lora_align_buffer_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_lora_align_layout": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int64)]),
    "moe_lora_align": (_I, [_P, _P, _AP, _P]),
    "moe_lora_get_error": (_I, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_lora_clear_error": (_I, [_P, _P]),
    "moe_gather_rows": (_I, [_P, _AP, _I, _P, _P]),
    "moe_grouped_gemm": (_I, [_P, _P, _AP, _I, _I, _P, _P]),
    "lora_shrink": (_I, [_P, _I, _P, _AP, _I, _I, _P, _P]),
    "lora_expand_add": (_I, [_P, _P, _AP, _I, _I, _I, _P, _P, _I, _P, _P]),
    "moe_lora_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_lora_layer": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I,
                            _I, _P, _I, _P, _SZ, _P]),
    "moe_lora_layer_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                               _I, _I, _P, _I, _P, _SZ, ctypes.POINTER(LayerOpts), _P]),
    "moe_lora_layer_tiles": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int32),
                                  ctypes.POINTER(ctypes.c_int32)]),
    "moe_lora_layer_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(LayerOpts),
                                 ctypes.POINTER(LayerPlan)]),
    "moe_lora_host_io_layout": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int64),
                                     ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "moe_lora_layer_host": (_I, [_P, _P, _P, _SZ, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                                 _P, _I, _I, _I, _P, _SZ, ctypes.POINTER(LayerOpts), _P]),
}

_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise MoeLoraUnavailable(
                        f"{LIB_PATH} is not built; run expert_adapter_gemms_gb300.build.build()")
                h = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(h, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = h
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().moe_lora_status_string(status).decode()
    except MoeLoraUnavailable:
        return "library not built"


def check(status: int, what: str) -> None:
    if status != OK:
        raise MoeLoraError(status, what)


def stream_handle(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def ptr(t) -> int:
    return 0 if t is None else t.data_ptr()
