"""ctypes view of libdflash.so (include/dflash.h).  Argument marshalling only.

Loading fails loudly when the library has not been built: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash.so")

DFLASH_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "pool exhausted",
                4: "CUDA error", 5: "device status set", 6: "workspace too small",
                7: "too large for the fixed scratch", 8: "not allowed while capturing"}
ROUND_DEVICE = (1 << 64) - 1   # dflash_accept: take the round from the device counter
DEV_POOL_EXHAUSTED, DEV_SEQ_TOO_LONG, DEV_WAIT_TIMEOUT, DEV_BAD_TOKEN, DEV_BAD_ROWS, DEV_BAD_BLOCK = 1, 2, 4, 8, 16, 32
DTYPE_F32, DTYPE_BF16, DTYPE_BF16_W8 = 0, 1, 2

EXPORTED = ("dflash_workspace_size", "dflash_kv_pool_size", "dflash_create", "dflash_destroy",
            "dflash_reset", "dflash_release", "dflash_inject_kv", "dflash_draft_block",
            "dflash_accept", "dflash_get_status", "dflash_status_string", "dflash_gemm_bf16",
            "dflash_profile_enable", "dflash_profile_read", "dflash_truncate", "dflash_gemm_bf16_noalloc",
            "dflash_graph_begin", "dflash_graph_end", "dflash_graph_launch", "dflash_graph_destroy",
            "dflash_gemm_w8", "dflash_block_attention")
PROF_CLASSES = ("proj", "lm_head", "inject", "attention", "rowwise", "accept")


class DflashConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "mask_id",
        "n_taps", "tap_width", "block_k", "page_size", "max_batch", "max_pages_per_seq", "n_pages",
        "max_rows", "max_inject_rows")] + [("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                                           ("dtype", ctypes.c_int)]


_VP = ctypes.c_void_p
_PVP = ctypes.POINTER(ctypes.c_void_p)


class DflashWeights(ctypes.Structure):
    _fields_ = [("w_fc", _VP), ("g_fc", _VP), ("embed", _VP), ("g_final", _VP), ("w_lm", _VP),
                ("w_kv_inject", _VP), ("key_offset", _VP),
                ("w_qkv", _PVP), ("w_o", _PVP), ("w_gu", _PVP), ("w_down", _PVP),
                ("g_in", _PVP), ("g_post", _PVP),
                ("s_fc", _VP), ("s_lm", _VP), ("s_kv_inject", _VP),
                ("s_qkv", _PVP), ("s_o", _PVP), ("s_gu", _PVP), ("s_down", _PVP)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libdflash (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdflash.so not built at {LIB_PATH}; run "
                               "python -m block_diffusion_speculative_hidden_gb300.build_lib")
        L = ctypes.CDLL(LIB_PATH)
        sz = ctypes.c_size_t
        i32p = ctypes.c_void_p
        L.dflash_workspace_size.restype = sz
        L.dflash_workspace_size.argtypes = [ctypes.POINTER(DflashConfig)]
        L.dflash_kv_pool_size.restype = sz
        L.dflash_kv_pool_size.argtypes = [ctypes.POINTER(DflashConfig)]
        L.dflash_create.restype = ctypes.c_int
        L.dflash_create.argtypes = [ctypes.POINTER(DflashConfig), ctypes.POINTER(DflashWeights), _VP, sz,
                                    i32p, i32p, _VP, sz, ctypes.POINTER(ctypes.c_void_p)]
        L.dflash_destroy.restype = ctypes.c_int
        L.dflash_destroy.argtypes = [_VP]
        L.dflash_reset.restype = ctypes.c_int
        L.dflash_reset.argtypes = [_VP, _VP]
        L.dflash_release.restype = ctypes.c_int
        L.dflash_release.argtypes = [_VP, ctypes.c_int, _VP]
        L.dflash_truncate.restype = ctypes.c_int
        L.dflash_truncate.argtypes = [_VP, ctypes.c_int, ctypes.c_int, _VP]
        L.dflash_inject_kv.restype = ctypes.c_int
        L.dflash_inject_kv.argtypes = [_VP, _VP, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _VP]
        L.dflash_draft_block.restype = ctypes.c_int
        L.dflash_draft_block.argtypes = [_VP, ctypes.c_int, ctypes.c_int, i32p, _VP, _VP, i32p, _VP]
        L.dflash_accept.restype = ctypes.c_int
        L.dflash_accept.argtypes = [_VP, ctypes.c_int, ctypes.c_int, i32p, i32p, _VP, _VP, ctypes.c_float,
                                    ctypes.c_uint64, ctypes.c_uint64, i32p, i32p, i32p, _VP]
        L.dflash_get_status.restype = ctypes.c_int
        L.dflash_get_status.argtypes = [_VP, ctypes.POINTER(ctypes.c_int), _VP]
        L.dflash_gemm_bf16.restype = ctypes.c_int
        L.dflash_gemm_bf16.argtypes = [_VP, ctypes.c_int, ctypes.c_int, _VP, _VP, ctypes.c_int, _VP, ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_int), _VP, _VP]
        L.dflash_block_attention.restype = ctypes.c_int
        L.dflash_block_attention.argtypes = [_VP, ctypes.c_int, ctypes.c_int, i32p, i32p, _VP, _VP, _VP, _VP, _VP]
        L.dflash_gemm_w8.restype = ctypes.c_int
        L.dflash_gemm_w8.argtypes = [_VP, _VP, ctypes.c_int, ctypes.c_int, _VP, _VP, ctypes.c_int, _VP, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_int), _VP, _VP]
        L.dflash_gemm_bf16_noalloc.restype = ctypes.c_int
        L.dflash_gemm_bf16_noalloc.argtypes = [_VP, ctypes.c_int, ctypes.c_int, _VP, _VP, ctypes.c_int, _VP,
                                               ctypes.c_int, ctypes.POINTER(ctypes.c_int), _VP, _VP]
        L.dflash_profile_enable.restype = ctypes.c_int
        L.dflash_profile_enable.argtypes = [_VP, ctypes.c_int]
        L.dflash_profile_read.restype = ctypes.c_int
        L.dflash_profile_read.argtypes = [_VP, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int), _VP]
        L.dflash_graph_begin.restype = ctypes.c_int
        L.dflash_graph_begin.argtypes = [_VP, _VP]
        L.dflash_graph_end.restype = ctypes.c_int
        L.dflash_graph_end.argtypes = [_VP, _VP, ctypes.POINTER(ctypes.c_void_p)]
        L.dflash_graph_launch.restype = ctypes.c_int
        L.dflash_graph_launch.argtypes = [_VP, _VP]
        L.dflash_graph_destroy.restype = ctypes.c_int
        L.dflash_graph_destroy.argtypes = [_VP]
        L.dflash_status_string.restype = ctypes.c_char_p
        L.dflash_status_string.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


class DflashError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)} ({code})")
        self.code = code


def check(code: int, what: str) -> None:
    if code != DFLASH_OK:
        raise DflashError(code, what)
