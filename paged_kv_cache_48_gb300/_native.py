"""ctypes view of ``libpagedkv.so`` (the C ABI declared in include/pagedkv.h).

Argument marshalling only.  Loading fails loudly when the library has not
been built: there is no fallback implementation anywhere in the package.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

PKG = Path(__file__).resolve().parent
LIBRARY = PKG / "libpagedkv.so"
HEADER = PKG.parent / "include" / "pagedkv.h"
HEADERS = sorted((PKG.parent / "include").glob("*.h"))

PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_ARG", 2: "PKV_ERR_DTYPE",
                3: "PKV_ERR_SHAPE", 4: "PKV_ERR_CUDA", 5: "PKV_ERR_RANGE",
                6: "PKV_ERR_TIMEOUT", 7: "PKV_ERR_WORKSPACE"}
PKV_BF16 = 0
PKV_FP8_E4M3 = 1
PKV_NOALLOC_SCRATCH_BYTES = 16 << 20


class PkvCache(ctypes.Structure):
    """Mirror of ``pkv_cache``."""
    _fields_ = [
        ("key_cache", ctypes.c_void_p),
        ("value_cache", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
    ]


_P = ctypes.c_void_p
_SIGNATURES = {
    "paged_kv_write": (ctypes.c_int, [_P, _P, _P, ctypes.c_int64,
                                      ctypes.POINTER(PkvCache), _P]),
    "paged_kv_zero_blocks": (ctypes.c_int, [ctypes.POINTER(PkvCache), _P,
                                            ctypes.c_int64, ctypes.c_int, _P]),
    "paged_kv_zero_and_write": (ctypes.c_int, [_P, _P, _P, ctypes.c_int64,
                                               ctypes.POINTER(PkvCache), _P,
                                               ctypes.c_int64, ctypes.c_int, _P]),
    "paged_kv_copy_blocks": (ctypes.c_int, [ctypes.POINTER(PkvCache), _P, _P,
                                            ctypes.c_int64, ctypes.c_int, _P]),
    "paged_kv_swap_out": (ctypes.c_int, [ctypes.POINTER(PkvCache), _P,
                                         ctypes.c_int64, ctypes.c_int, _P, _P,
                                         _P]),
    "paged_kv_swap_in": (ctypes.c_int, [ctypes.POINTER(PkvCache), _P,
                                        ctypes.c_int64, ctypes.c_int, _P, _P,
                                        _P]),
    "paged_prepare_inputs": (ctypes.c_int, [
        _P, _P, ctypes.c_int32, _P, ctypes.c_int32, _P, _P, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int64, _P, _P, _P, _P, _P, _P, _P]),
    "paged_attention_decode": (ctypes.c_int, [
        _P, ctypes.POINTER(PkvCache), _P, ctypes.c_int32, _P, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_float, _P, ctypes.c_int32, ctypes.c_int32,
        _P, ctypes.c_size_t, _P]),
    "paged_attention_decode_step": (ctypes.c_int, [
        _P, _P, _P, _P, ctypes.c_int64, ctypes.POINTER(PkvCache), _P,
        ctypes.c_int32, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _P,
        ctypes.c_int32, ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "paged_attention_prefill": (ctypes.c_int, [
        _P, ctypes.POINTER(PkvCache), _P, ctypes.c_int32, _P, _P,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, _P,
        ctypes.c_int32, _P]),
    "paged_attention_decode_cascade": (ctypes.c_int, [
        _P, ctypes.POINTER(PkvCache), _P, ctypes.c_int32, _P, ctypes.c_int32,
        ctypes.c_int32, _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_float, _P, ctypes.c_int32, ctypes.c_int32, _P, ctypes.c_size_t,
        _P]),
    "paged_attention_cascade_workspace_bytes": (ctypes.c_size_t, [
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    "paged_attention_decode_noalloc": (ctypes.c_int, [
        _P, ctypes.POINTER(PkvCache), _P, ctypes.c_int32, _P, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_float, _P, ctypes.c_int32, ctypes.c_int32,
        _P]),
    "paged_attention_workspace_bytes": (ctypes.c_size_t, [
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32]),
    "paged_attention_partition_tokens": (ctypes.c_int32, [
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int32]),
    "pkv_check": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int64)]),
    "pkv_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_version": (ctypes.c_int32, []),
    "pkv_testing_fail_decode_sequence": (None, [ctypes.c_int32]),
}

_LIB = None


class PagedKVError(RuntimeError):
    def __init__(self, call: str, status: int, detail: int = -1):
        self.status = status
        self.detail = detail
        name = STATUS_NAMES.get(status, str(status))
        msg = f"{call} failed: {name}"
        if _LIB is not None:
            msg += f" ({_LIB.pkv_status_str(status).decode()})"
        if detail >= 0:
            msg += f", index {detail}"
        super().__init__(msg)


def declared_functions() -> list:
    """Names of the functions the headers under include/ declare."""
    text = "\n".join(h.read_text() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    keywords = {"if", "sizeof", "defined"}
    return sorted({n for n in names if n not in keywords and
                   (n.startswith("paged_") or n.startswith("pkv_"))})


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not LIBRARY.exists():
            raise RuntimeError(
                f"{LIBRARY} is missing: build it with "
                "`python -m paged_kv_cache_48_gb300.build` (needs nvcc); the "
                "package has no CPU or PyTorch fallback")
        handle = ctypes.CDLL(str(LIBRARY))
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def check(call: str, status: int) -> None:
    if status != PKV_OK:
        raise PagedKVError(call, status)
