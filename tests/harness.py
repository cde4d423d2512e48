"""Runs one workload through the CUDA path (via the C ABI binding) and
through the CPU oracle, on the same seeded inputs, and compares them.

The oracle never sees a value the CUDA path produced: both start from the
workload's initial pool bytes and apply their own zeroing, writes and
attention.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import oracle
from paged_kv_cache_48_gb300 import (PagedKVCache, paged_attention_decode,
                                     paged_attention_prefill, paged_kv_write,
                                     paged_kv_zero_and_write, paged_kv_zero_blocks,
                                     pkv_check)
from paged_kv_cache_48_gb300.workload import PrefillWorkload, Workload

# Tolerances of the parity bar: |gpu - ref| <= ATOL + RTOL * |ref| per
# element, bf16 KV 1e-2 / 1e-2, fp8 KV 3e-2 / 3e-2.
TOL = {"bf16": (1e-2, 1e-2), "fp8_e4m3": (3e-2, 3e-2)}


def _cache_dtype(W: Workload):
    return torch.bfloat16 if W.kv_dtype == "bf16" else torch.uint8


def _u16_to_bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(device)


@dataclass
class GpuState:
    cache: PagedKVCache
    q: torch.Tensor
    tables: torch.Tensor
    seq_lens: torch.Tensor
    step_k: torch.Tensor
    step_v: torch.Tensor
    step_slots: torch.Tensor
    fresh: np.ndarray


def upload(W: Workload, device="cuda", write_history=True) -> GpuState:
    """Pool bytes to the device, then the history tokens written through
    paged_kv_write (in chunks)."""
    shape = (W.num_blocks, W.block_size, W.num_kv_heads, W.head_dim)
    dt = _cache_dtype(W)
    kc = torch.from_numpy(W.init_key).view(dt).reshape(shape).to(device)
    vc = torch.from_numpy(W.init_value).view(dt).reshape(shape).to(device)
    cache = PagedKVCache(kc, vc, W.kv_dtype, W.k_scale, W.v_scale)
    if write_history and W.hist_slots.size:
        chunk = 1 << 18
        for s in range(0, W.hist_slots.size, chunk):
            e = min(W.hist_slots.size, s + chunk)
            paged_kv_write(_u16_to_bf16(W.hist_k[s:e], device),
                           _u16_to_bf16(W.hist_v[s:e], device),
                           torch.from_numpy(W.hist_slots[s:e]).to(device), cache)
    return GpuState(
        cache=cache, q=_u16_to_bf16(W.q, device),
        tables=torch.from_numpy(W.block_tables).to(device),
        seq_lens=torch.from_numpy(W.seq_lens).to(device),
        step_k=_u16_to_bf16(W.step_k, device),
        step_v=_u16_to_bf16(W.step_v, device),
        step_slots=torch.from_numpy(W.step_slots).to(device),
        fresh=W.fresh_blocks.copy())


def gpu_step(W: Workload, G: GpuState, partition_tokens=0, skip_zero=False,
             out=None, fused=False, max_seq_len=None):
    """One decode step: zero fresh blocks, write the step's tokens, attend.
    fused: the zeroing and the write as one paged_kv_zero_and_write call.
    max_seq_len: the host bound given to attention (default: the longest
    sequence; bench.py gives the table width, max_blocks * 16)."""
    if fused and not skip_zero:
        paged_kv_zero_and_write(G.step_k, G.step_v, G.step_slots, G.cache, G.fresh)
    else:
        if not skip_zero and G.fresh.size:
            paged_kv_zero_blocks(G.cache, G.fresh)
        if G.step_slots.numel():
            paged_kv_write(G.step_k, G.step_v, G.step_slots, G.cache)
    return paged_attention_decode(G.q, G.cache, G.tables, G.seq_lens, W.scale,
                                  max_seq_len=W.max_seq_len if max_seq_len is None
                                  else max_seq_len, out=out,
                                  partition_tokens=partition_tokens)


def run_gpu(W: Workload, partition_tokens=0, skip_zero=False, device="cuda",
            want_cache=True, fused=False, max_seq_len=None):
    G = upload(W, device)
    out = gpu_step(W, G, partition_tokens, skip_zero, fused=fused,
                   max_seq_len=max_seq_len)
    status, detail = pkv_check()
    res = {"out": out.float().cpu().numpy(), "status": status,
           "detail": detail, "state": G}
    if want_cache:
        res["key"] = G.cache.key_cache.view(torch.uint8).cpu().numpy().reshape(-1)
        res["value"] = G.cache.value_cache.view(torch.uint8).cpu().numpy().reshape(-1)
    return res


def oracle_cache(W: Workload, skip_zero=False):
    """The pool after the oracle's own history write, zeroing and step
    write."""
    o = oracle.load()
    dt = oracle.DTYPE_BF16 if W.kv_dtype == "bf16" else oracle.DTYPE_FP8_E4M3
    kc = W.init_key.copy()
    vc = W.init_value.copy()
    e1 = o.kv_write(kc, vc, dt, W.block_size, W.num_kv_heads, W.head_dim,
                    W.k_scale, W.v_scale, W.hist_k, W.hist_v, W.hist_slots)
    e2 = 0 if skip_zero else o.zero_blocks(kc, vc, W.block_bytes,
                                          W.fresh_blocks)
    e3 = o.kv_write(kc, vc, dt, W.block_size, W.num_kv_heads, W.head_dim,
                    W.k_scale, W.v_scale, W.step_k, W.step_v, W.step_slots)
    assert e1 == e2 == e3 == 0
    return kc, vc


def oracle_out(W: Workload, kc, vc, pairs=None, n_threads=0):
    o = oracle.load()
    dt = oracle.DTYPE_BF16 if W.kv_dtype == "bf16" else oracle.DTYPE_FP8_E4M3
    out, err = o.attention_decode(W.q, kc, vc, dt, W.k_scale, W.v_scale,
                                  W.block_size, W.num_kv_heads, W.head_dim,
                                  W.block_tables, W.seq_lens, W.scale,
                                  pairs=pairs, n_threads=n_threads)
    assert err == 0
    return out


def assert_close(gpu: np.ndarray, ref: np.ndarray, kv_dtype: str, mask=None):
    atol, rtol = TOL[kv_dtype]
    g = gpu.astype(np.float64)
    if mask is not None:
        g, ref = g[mask], ref[mask]
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    err = np.abs(g - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), (
        f"{int(bad.sum())} of {bad.size} elements out of tolerance; "
        f"max abs err {err.max():.3e}")
    return float(err.max())


# ---------------------------------------------------------------------------
# chunked prefill
# ---------------------------------------------------------------------------

@dataclass
class PrefillGpuState:
    cache: PagedKVCache
    q: torch.Tensor
    tables: torch.Tensor
    seq_lens: torch.Tensor
    qsl: torch.Tensor
    step_k: torch.Tensor
    step_v: torch.Tensor
    step_slots: torch.Tensor


def upload_prefill(W: PrefillWorkload, device="cuda") -> PrefillGpuState:
    """Pool bytes to the device and the history written through
    paged_kv_write; the chunk's K/V stay pending for the step."""
    shape = (W.num_blocks, W.block_size, W.num_kv_heads, W.head_dim)
    dt = torch.bfloat16 if W.kv_dtype == "bf16" else torch.uint8
    kc = torch.from_numpy(W.init_key).view(dt).reshape(shape).to(device)
    vc = torch.from_numpy(W.init_value).view(dt).reshape(shape).to(device)
    cache = PagedKVCache(kc, vc, W.kv_dtype, W.k_scale, W.v_scale)
    if W.hist_slots.size:
        chunk = 1 << 18
        for s in range(0, W.hist_slots.size, chunk):
            e = min(W.hist_slots.size, s + chunk)
            paged_kv_write(_u16_to_bf16(W.hist_k[s:e], device),
                           _u16_to_bf16(W.hist_v[s:e], device),
                           torch.from_numpy(W.hist_slots[s:e]).to(device), cache)
    return PrefillGpuState(
        cache=cache, q=_u16_to_bf16(W.q, device),
        tables=torch.from_numpy(W.block_tables).to(device),
        seq_lens=torch.from_numpy(W.seq_lens).to(device),
        qsl=torch.from_numpy(W.query_start_loc).to(device),
        step_k=_u16_to_bf16(W.step_k, device),
        step_v=_u16_to_bf16(W.step_v, device),
        step_slots=torch.from_numpy(W.step_slots).to(device))


def gpu_prefill_step(W: PrefillWorkload, G: PrefillGpuState, out=None):
    """One chunked-prefill step: write the chunk's K/V, then attend."""
    if G.step_slots.numel():
        paged_kv_write(G.step_k, G.step_v, G.step_slots, G.cache)
    return paged_attention_prefill(G.q, G.cache, G.tables, G.seq_lens, G.qsl,
                                   W.scale, max_query_len=W.max_query_len,
                                   out=out)


def _oracle_dtype(W):
    return oracle.DTYPE_BF16 if W.kv_dtype == "bf16" else oracle.DTYPE_FP8_E4M3


def oracle_prefill_cache(W: PrefillWorkload):
    o = oracle.load()
    kc = W.init_key.copy()
    vc = W.init_value.copy()
    for k, v, sl in ((W.hist_k, W.hist_v, W.hist_slots),
                     (W.step_k, W.step_v, W.step_slots)):
        assert o.kv_write(kc, vc, _oracle_dtype(W), W.block_size,
                          W.num_kv_heads, W.head_dim, W.k_scale, W.v_scale,
                          k, v, sl) == 0
    return kc, vc


def oracle_prefill_out(W: PrefillWorkload, kc, vc, rows=None, n_threads=0):
    out, err = oracle.load().attention_prefill(
        W.q, kc, vc, _oracle_dtype(W), W.k_scale, W.v_scale, W.block_size,
        W.num_kv_heads, W.head_dim, W.block_tables, W.seq_lens,
        W.query_start_loc, W.scale, rows=rows, n_threads=n_threads)
    assert err == 0
    return out
