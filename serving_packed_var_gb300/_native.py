"""ctypes view of libadaflash.so (the C ABI declared in include/adaflash.h).

Loading fails loudly when the library has not been built: there is no other
implementation to fall back to.
"""

from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libadaflash.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "adaflash.h")

ADAFLASH_OK = 0
ADAFLASH_ERR_INVALID_ARG = 1
ADAFLASH_ERR_UNSUPPORTED = 2
ADAFLASH_ERR_CUDA = 3
ADAFLASH_ERR_TIMEOUT = 4
ADAFLASH_ERR_BAD_OFFSETS = 5
ADAFLASH_ERR_BAD_TOKEN = 6

ADAFLASH_FP32 = 0
ADAFLASH_BF16 = 1
ADAFLASH_MAX_VOCAB = 524288

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_f64 = ctypes.c_double

SIGNATURES = {
    "adaflash_verify_packed": [_vp, _i32, _i64, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp],
    "adaflash_opd_loss_fwd": [_vp, _i32, _i64, _vp, _i32, _i64, _vp, _vp, _i32, _i32, _i32, _f32, _f32,
                              _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "adaflash_opd_loss_bwd": [_vp, _i32, _i64, _vp, _i32, _i64, _vp, _i32, _i32, _i32, _f32, _f32,
                              _vp, _vp, _vp, _f32, _vp, _i64, _vp, _vp],
    "adaflash_opd_loss_fwd_bwd": [_vp, _i32, _i64, _vp, _i32, _i64, _vp, _vp, _i32, _i32, _i32, _f32, _f32,
                                  _vp, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp],
    "adaflash_verify_sampled": [_vp, _i32, _i64, _vp, _i32, _i64, _vp, _vp, _i32, _i32, _i32, _f32,
                                _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "adaflash_selftest_bounded_wait": [_vp, _i32, _vp],
    "adaflash_lmhead_workspace_bytes": [_i32, _i32, _i32, _i32],
    "adaflash_lmhead_logits": [_vp, _i64, _i32, _vp, _i64, _i32, _i32, _vp, _i64, _vp, _vp],
    "adaflash_lmhead_opd_fwd": [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp, _vp, _i32, _i32, _i32,
                                _f32, _f32, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "adaflash_lmhead_opd_fwd_static": [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp, _vp, _i32, _i32, _i32,
                                       _f32, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "adaflash_packer_create": [_i32, _f64, _f64, _vp],
    "adaflash_packer_destroy": [_vp],
    "adaflash_packer_plan": [_vp, _vp, _i32, _vp, _vp, _vp, _vp],
    "adaflash_packer_observe": [_vp, _i32, _i32],
    "adaflash_packer_estimate": [_vp, _vp],
    "adaflash_status_string": [_i32],
    "adaflash_kernel_launches": [],
}

_lib = None


class LibraryMissing(RuntimeError):
    pass


def lib() -> ctypes.CDLL:
    """The loaded library with argument and result types set."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise LibraryMissing(
            f"{LIB_PATH} is missing: build it with serving_packed_var_gb300.build.build() "
            "(nvcc, sm_103a); the package has no other implementation")
    L = ctypes.CDLL(LIB_PATH)
    for name, args in SIGNATURES.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = {"adaflash_status_string": ctypes.c_char_p,
                      "adaflash_kernel_launches": ctypes.c_uint64,
                      "adaflash_lmhead_workspace_bytes": ctypes.c_int64}.get(name, ctypes.c_int)
    _lib = L
    return L


def declared_functions(header: str = HEADER):
    """Names of the functions include/adaflash.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(adaflash_[a-z_]+)\s*\(", text)))


def status_string(code: int) -> str:
    return lib().adaflash_status_string(code).decode()
