"""Plain fp64 CPU oracle for the paged KV-cache decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (``paged_kv_cache_48_gb300``) never imports it and shares no code with
it: the arithmetic lives in ``pagedkv_oracle.c`` and this module only
marshals numpy arrays into that C library through ctypes.

What each function restates is documented in the C file; the sources are the
vLLM concept page (compassingai.com, "技术原理" pseudocode), the vLLM v0.17.1
notes (admirer.cn, "修复方案") and the vLLM internals post
(naphjohn.github.io, §1.1 and Figure 1).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, library special cases, invariants and format-definition
values); no function is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "pagedkv_oracle.c"
LIBRARY = _HERE / "liboracle.so"

DTYPE_BF16 = 0
DTYPE_FP8_E4M3 = 1


def compile_library(source: Path = SOURCE, output: Path = LIBRARY,
                    extra_flags: tuple = ()) -> Path:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math)."""
    output = Path(output)
    tmp = output.with_name(output.name + f".tmp{os.getpid()}")
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", *extra_flags,
           str(source), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


def _needs_build(lib: Path, src: Path) -> bool:
    return (not lib.exists()) or lib.stat().st_mtime < src.stat().st_mtime


_P = ctypes.c_void_p


class Oracle:
    """ctypes view of one compiled oracle library (the real one, or a
    deliberately mutated copy built by the mutation tests)."""

    def __init__(self, path: Path):
        self.path = Path(path)
        lib = ctypes.CDLL(str(self.path))
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.oracle_quantize_e4m3.argtypes = [ctypes.c_uint16, ctypes.c_float]
        lib.oracle_quantize_e4m3.restype = ctypes.c_uint8
        lib.oracle_kv_write.argtypes = [
            _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_float, ctypes.c_float, _P, _P, _P,
            ctypes.c_long]
        lib.oracle_kv_write.restype = ctypes.c_long
        lib.oracle_zero_blocks.argtypes = [_P, _P, ctypes.c_size_t,
                                           ctypes.c_int, _P, ctypes.c_long]
        lib.oracle_zero_blocks.restype = ctypes.c_long
        lib.oracle_attention_decode.argtypes = [
            _P, _P, _P, ctypes.c_int, ctypes.c_double, ctypes.c_double,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P,
            ctypes.c_int, _P, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            _P, _P, ctypes.c_long, ctypes.c_int]
        lib.oracle_attention_decode.restype = ctypes.c_long
        lib.oracle_attention_prefill.argtypes = [
            _P, _P, _P, ctypes.c_int, ctypes.c_double, ctypes.c_double,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P,
            ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            _P, _P, ctypes.c_long, ctypes.c_int]
        lib.oracle_attention_prefill.restype = ctypes.c_long
        for name in ("oracle_copy_blocks",):
            fn = getattr(lib, name)
            fn.argtypes = [_P, _P, ctypes.c_size_t, ctypes.c_int, _P, _P,
                           ctypes.c_long]
            fn.restype = ctypes.c_long
        for name in ("oracle_swap_out", "oracle_swap_in"):
            fn = getattr(lib, name)
            fn.argtypes = [_P, _P, ctypes.c_size_t, ctypes.c_int, _P,
                           ctypes.c_long, _P, _P]
            fn.restype = ctypes.c_long
        lib.oracle_prepare_inputs.argtypes = [
            _P, _P, ctypes.c_int, _P, ctypes.c_int, _P, _P, ctypes.c_int,
            ctypes.c_int, ctypes.c_long, _P, _P, _P, _P, _P, _P]
        lib.oracle_prepare_inputs.restype = ctypes.c_long
        lib.oracle_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_num_threads.restype = ctypes.c_int
        self.lib = lib

    # -- number formats -------------------------------------------------
    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(int(bits))

    def e4m3_to_double(self, code: int) -> float:
        return self.lib.oracle_e4m3_to_double(int(code))

    def e4m3_from_float(self, x: float) -> int:
        return self.lib.oracle_e4m3_from_float(float(np.float32(x)))

    def quantize_e4m3(self, x_bf16_bits: int, scale: float) -> int:
        return self.lib.oracle_quantize_e4m3(int(x_bf16_bits),
                                             float(np.float32(scale)))

    def num_threads(self, n_threads: int = 0) -> int:
        return self.lib.oracle_num_threads(int(n_threads))

    # -- path steps -----------------------------------------------------
    def kv_write(self, key_cache: np.ndarray, value_cache: np.ndarray,
                 dtype: int, block_size: int, num_kv_heads: int,
                 head_dim: int, k_scale: float, v_scale: float,
                 k: np.ndarray, v: np.ndarray,
                 slot_mapping: np.ndarray) -> int:
        """In-place slot-mapped write into host caches (uint8 byte views).
        k, v: uint16 bf16 bits [T, Hkv, d]; slot_mapping int64 [T]."""
        _check_c(key_cache, np.uint8)
        _check_c(value_cache, np.uint8)
        k = np.ascontiguousarray(k, dtype=np.uint16)
        v = np.ascontiguousarray(v, dtype=np.uint16)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        eb = 2 if dtype == DTYPE_BF16 else 1
        block_bytes = block_size * num_kv_heads * head_dim * eb
        num_blocks = key_cache.size // block_bytes
        return self.lib.oracle_kv_write(
            key_cache.ctypes.data, value_cache.ctypes.data, dtype, num_blocks,
            block_size, num_kv_heads, head_dim, float(np.float32(k_scale)),
            float(np.float32(v_scale)), k.ctypes.data, v.ctypes.data,
            slots.ctypes.data, slots.size)

    def zero_blocks(self, key_cache: np.ndarray, value_cache: np.ndarray,
                    block_bytes: int, block_ids: np.ndarray) -> int:
        _check_c(key_cache, np.uint8)
        _check_c(value_cache, np.uint8)
        ids = np.ascontiguousarray(block_ids, dtype=np.int32)
        num_blocks = key_cache.size // block_bytes
        return self.lib.oracle_zero_blocks(
            key_cache.ctypes.data, value_cache.ctypes.data, block_bytes,
            num_blocks, ids.ctypes.data, ids.size)

    def copy_blocks(self, key_cache, value_cache, block_bytes, src, dst):
        """In-place copy of blocks src[i] -> dst[i] (in order)."""
        _check_c(key_cache, np.uint8)
        _check_c(value_cache, np.uint8)
        s = np.ascontiguousarray(src, dtype=np.int32)
        d = np.ascontiguousarray(dst, dtype=np.int32)
        assert s.shape == d.shape
        return self.lib.oracle_copy_blocks(
            key_cache.ctypes.data, value_cache.ctypes.data, block_bytes,
            key_cache.size // block_bytes, s.ctypes.data, d.ctypes.data,
            s.size)

    def swap_out(self, key_cache, value_cache, block_bytes, ids):
        """Returns (out_k, out_v, errors): the blocks packed in id order."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        out_k = np.zeros(ids.size * block_bytes, np.uint8)
        out_v = np.zeros(ids.size * block_bytes, np.uint8)
        err = self.lib.oracle_swap_out(
            key_cache.ctypes.data, value_cache.ctypes.data, block_bytes,
            key_cache.size // block_bytes, ids.ctypes.data, ids.size,
            out_k.ctypes.data, out_v.ctypes.data)
        return out_k, out_v, err

    def swap_in(self, key_cache, value_cache, block_bytes, ids, in_k, in_v):
        _check_c(key_cache, np.uint8)
        _check_c(value_cache, np.uint8)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        in_k = np.ascontiguousarray(in_k, dtype=np.uint8)
        in_v = np.ascontiguousarray(in_v, dtype=np.uint8)
        return self.lib.oracle_swap_in(
            key_cache.ctypes.data, value_cache.ctypes.data, block_bytes,
            key_cache.size // block_bytes, ids.ctypes.data, ids.size,
            in_k.ctypes.data, in_v.ctypes.data)

    def prepare_inputs(self, idx_mapping, num_scheduled, state_block_table,
                       state_num_computed, state_token_ids, total_tokens):
        """Step inputs gathered from the request state table.  Returns a
        dict of arrays and the error count."""
        idx = np.ascontiguousarray(idx_mapping, dtype=np.int32)
        ns = np.ascontiguousarray(num_scheduled, dtype=np.int32)
        sbt = np.ascontiguousarray(state_block_table, dtype=np.int32)
        snc = np.ascontiguousarray(state_num_computed, dtype=np.int32)
        tok = np.ascontiguousarray(state_token_ids, dtype=np.int32)
        B = idx.size
        R, MB = sbt.shape
        ML = tok.shape[1]
        T = int(total_tokens)
        out = {"block_tables": np.full((B, MB), -7, np.int32),
               "seq_lens": np.full(B, -7, np.int32),
               "query_start_loc": np.full(B + 1, -7, np.int32),
               "positions": np.full(T, -7, np.int32),
               "input_ids": np.full(T, -7, np.int32),
               "slot_mapping": np.full(T, -7, np.int64)}
        err = self.lib.oracle_prepare_inputs(
            idx.ctypes.data, ns.ctypes.data, B, sbt.ctypes.data, MB,
            snc.ctypes.data, tok.ctypes.data, ML, R, T,
            out["block_tables"].ctypes.data, out["seq_lens"].ctypes.data,
            out["query_start_loc"].ctypes.data, out["positions"].ctypes.data,
            out["input_ids"].ctypes.data, out["slot_mapping"].ctypes.data)
        return out, err

    def attention_decode(self, q: np.ndarray, key_cache: np.ndarray,
                         value_cache: np.ndarray, dtype: int,
                         k_scale: float, v_scale: float, block_size: int,
                         num_kv_heads: int, head_dim: int,
                         block_tables: np.ndarray, seq_lens: np.ndarray,
                         scale: float, pairs=None, n_threads: int = 0):
        """fp64 decode attention.  q: uint16 bf16 bits [B, Hq, d].
        Returns (out float64 [B, Hq, d], error_count).  With ``pairs``
        (int array [n, 2] of (b, h)) only those rows are computed; the other
        rows of ``out`` stay 0."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        B, Hq, d = q.shape
        assert d == head_dim
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        assert tables.shape[0] == B and lens.shape == (B,)
        _check_c(key_cache, np.uint8)
        _check_c(value_cache, np.uint8)
        eb = 2 if dtype == DTYPE_BF16 else 1
        num_blocks = key_cache.size // (block_size * num_kv_heads * head_dim * eb)
        out = np.zeros((B, Hq, d), dtype=np.float64)
        if pairs is None:
            pp, n_pairs = None, 0
        else:
            pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
            pp, n_pairs = pairs.ctypes.data, pairs.shape[0]
        err = self.lib.oracle_attention_decode(
            q.ctypes.data, key_cache.ctypes.data, value_cache.ctypes.data,
            dtype, float(k_scale), float(v_scale), num_blocks, block_size,
            num_kv_heads, head_dim, tables.ctypes.data, tables.shape[1],
            lens.ctypes.data, B, Hq, float(scale), out.ctypes.data, pp,
            n_pairs, int(n_threads))
        return out, err

    def attention_prefill(self, q: np.ndarray, key_cache: np.ndarray,
                          value_cache: np.ndarray, dtype: int,
                          k_scale: float, v_scale: float, block_size: int,
                          num_kv_heads: int, head_dim: int,
                          block_tables: np.ndarray, seq_lens: np.ndarray,
                          query_start_loc: np.ndarray, scale: float,
                          rows=None, n_threads: int = 0):
        """fp64 prefill / chunked-prefill attention (causal within each
        sequence's chunk).  q: uint16 bf16 bits [T, Hq, d]; query_start_loc
        int [B+1].  Returns (out float64 [T, Hq, d], error_count).  With
        ``rows`` (int array [n, 2] of (token, head)) only those rows are
        computed; the others stay 0."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        T, Hq, d = q.shape
        assert d == head_dim
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
        B = lens.shape[0]
        assert tables.shape[0] == B and qsl.shape == (B + 1,)
        assert B == 0 or qsl[B] == T
        _check_c(key_cache, np.uint8)
        _check_c(value_cache, np.uint8)
        eb = 2 if dtype == DTYPE_BF16 else 1
        num_blocks = key_cache.size // (block_size * num_kv_heads * head_dim * eb)
        out = np.zeros((T, Hq, d), dtype=np.float64)
        if rows is None:
            rp, n_rows = None, 0
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
            rp, n_rows = rows.ctypes.data, rows.shape[0]
        err = self.lib.oracle_attention_prefill(
            q.ctypes.data, key_cache.ctypes.data, value_cache.ctypes.data,
            dtype, float(k_scale), float(v_scale), num_blocks, block_size,
            num_kv_heads, head_dim, tables.ctypes.data,
            tables.shape[1] if tables.ndim == 2 else 0, lens.ctypes.data,
            qsl.ctypes.data, B, Hq, float(scale), out.ctypes.data, rp, n_rows,
            int(n_threads))
        return out, err


def _check_c(a: np.ndarray, dt) -> None:
    if a.dtype != dt or not a.flags["C_CONTIGUOUS"]:
        raise TypeError(f"expected C-contiguous {np.dtype(dt).name} array")


_DEFAULT = None


def load(rebuild: bool = False) -> Oracle:
    """The oracle built from ``pagedkv_oracle.c`` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None or rebuild:
        if rebuild or _needs_build(LIBRARY, SOURCE):
            compile_library()
        _DEFAULT = Oracle(LIBRARY)
    return _DEFAULT
