"""GB300-native hot path of DFlash block-diffusion speculative drafting.

libdflash (csrc/, C ABI in include/dflash.h) holds the CUDA kernels; this
package is the thin Python binding over it.
"""
from ._lib import ROUND_DEVICE, DflashError, lib  # noqa: F401
from .drafter import Drafter, RoundGraph, gemm_bf16, gemm_w8, weights_to_device  # noqa: F401

__all__ = ["Drafter", "RoundGraph", "DflashError", "ROUND_DEVICE", "lib", "gemm_bf16", "gemm_w8", "weights_to_device"]
