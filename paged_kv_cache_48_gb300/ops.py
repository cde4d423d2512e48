"""PyTorch-facing binding of the C ABI (include/pagedkv.h).

Marshalling only: tensors are checked for dtype, shape, device and
contiguity, their data pointers and torch's current CUDA stream are passed
to ``libpagedkv.so``, and a non-OK status raises ``PagedKVError``.  Every
step of the path (write, zeroing, gather, attention, reduce) runs in the
library's kernels; PyTorch only owns the device memory and the streams.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np
import torch

from . import _native
from ._native import PagedKVError, PkvCache

BLOCK_SIZE = 16
_DTYPES = {"bf16": _native.PKV_BF16, "fp8_e4m3": _native.PKV_FP8_E4M3}


def _stream_handle(stream: Optional[torch.cuda.Stream], device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _require(t: torch.Tensor, name: str, dtype, device=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class PagedKVCache:
    """Key and value caches of shape [num_blocks, 16, num_kv_heads,
    head_dim] on one CUDA device, bf16 or fp8 E4M3 (stored as uint8 with a
    per-tensor fp32 scale each)."""

    def __init__(self, key_cache: torch.Tensor, value_cache: torch.Tensor,
                 kv_dtype: str = "bf16", k_scale: float = 1.0,
                 v_scale: float = 1.0):
        if kv_dtype not in _DTYPES:
            raise ValueError(f"kv_dtype must be one of {list(_DTYPES)}")
        elt = torch.bfloat16 if kv_dtype == "bf16" else torch.uint8
        _require(key_cache, "key_cache", elt, ndim=4)
        _require(value_cache, "value_cache", elt, device=key_cache.device,
                 ndim=4)
        if key_cache.shape != value_cache.shape:
            raise ValueError("key_cache and value_cache shapes differ")
        if key_cache.shape[1] != BLOCK_SIZE:
            raise ValueError("block_size must be 16")
        if not key_cache.is_cuda:
            raise ValueError("caches must live on a CUDA device")
        self.key_cache = key_cache
        self.value_cache = value_cache
        self.kv_dtype = kv_dtype
        self.k_scale = float(k_scale)
        self.v_scale = float(v_scale)
        self._struct = PkvCache(
            key_cache.data_ptr(), value_cache.data_ptr(), key_cache.shape[0],
            BLOCK_SIZE, key_cache.shape[2], key_cache.shape[3],
            _DTYPES[kv_dtype], self.k_scale, self.v_scale)

    @classmethod
    def empty(cls, num_blocks: int, num_kv_heads: int, head_dim: int,
              kv_dtype: str = "bf16", k_scale: float = 1.0,
              v_scale: float = 1.0, device="cuda") -> "PagedKVCache":
        elt = torch.bfloat16 if kv_dtype == "bf16" else torch.uint8
        shape = (num_blocks, BLOCK_SIZE, num_kv_heads, head_dim)
        return cls(torch.empty(shape, dtype=elt, device=device),
                   torch.empty(shape, dtype=elt, device=device), kv_dtype,
                   k_scale, v_scale)

    @property
    def device(self) -> torch.device:
        return self.key_cache.device

    @property
    def num_blocks(self) -> int:
        return self.key_cache.shape[0]

    @property
    def num_kv_heads(self) -> int:
        return self.key_cache.shape[2]

    @property
    def head_dim(self) -> int:
        return self.key_cache.shape[3]

    @property
    def block_bytes(self) -> int:
        """Bytes of one block of one cache."""
        return BLOCK_SIZE * self.num_kv_heads * self.head_dim * \
            self.key_cache.element_size()

    def c_struct(self) -> PkvCache:
        return self._struct


def paged_kv_write(k: torch.Tensor, v: torch.Tensor,
                   slot_mapping: torch.Tensor, cache: PagedKVCache,
                   stream: Optional[torch.cuda.Stream] = None) -> None:
    """Write tokens' K/V rows ([T, num_kv_heads, head_dim] bf16) into
    their slots (int64 [T], negative = skip)."""
    dev = cache.device
    _require(k, "k", torch.bfloat16, dev, 3)
    _require(v, "v", torch.bfloat16, dev, 3)
    _require(slot_mapping, "slot_mapping", torch.int64, dev, 1)
    T = k.shape[0]
    if v.shape != k.shape or slot_mapping.shape[0] != T or \
            k.shape[1:] != (cache.num_kv_heads, cache.head_dim):
        raise ValueError("k, v, slot_mapping shapes do not match the cache")
    st = _native.lib().paged_kv_write(
        k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
        ctypes.byref(cache.c_struct()), _stream_handle(stream, dev))
    _native.check("paged_kv_write", st)


def paged_kv_zero_blocks(cache: PagedKVCache, block_ids,
                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """Zero every byte of the K and V segments of the given blocks.  Host
    ids (numpy array, list or CPU tensor) ride in the launch parameters;
    a CUDA int32 tensor is read by the kernel directly."""
    dev = cache.device
    if isinstance(block_ids, torch.Tensor) and block_ids.is_cuda:
        _require(block_ids, "block_ids", torch.int32, dev, 1)
        ptr, n, on_host, keep = block_ids.data_ptr(), block_ids.numel(), 0, None
    else:
        if isinstance(block_ids, torch.Tensor):
            block_ids = block_ids.numpy()
        keep = np.ascontiguousarray(block_ids, dtype=np.int32).reshape(-1)
        ptr, n, on_host = keep.ctypes.data, keep.size, 1
    st = _native.lib().paged_kv_zero_blocks(
        ctypes.byref(cache.c_struct()), ptr, n, on_host,
        _stream_handle(stream, dev))
    del keep
    _native.check("paged_kv_zero_blocks", st)


def paged_kv_zero_and_write(k: torch.Tensor, v: torch.Tensor,
                            slot_mapping: torch.Tensor, cache: PagedKVCache,
                            block_ids,
                            stream: Optional[torch.cuda.Stream] = None) -> None:
    """paged_kv_zero_blocks(cache, block_ids) then paged_kv_write(k, v,
    slot_mapping, cache), in one launch (more than 4096 host ids take
    several)."""
    dev = cache.device
    _require(k, "k", torch.bfloat16, dev, 3)
    _require(v, "v", torch.bfloat16, dev, 3)
    _require(slot_mapping, "slot_mapping", torch.int64, dev, 1)
    T = k.shape[0]
    if v.shape != k.shape or slot_mapping.shape[0] != T or \
            k.shape[1:] != (cache.num_kv_heads, cache.head_dim):
        raise ValueError("k, v, slot_mapping shapes do not match the cache")
    ptr, n, on_host, keep = _block_ids(block_ids, dev)
    st = _native.lib().paged_kv_zero_and_write(
        k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
        ctypes.byref(cache.c_struct()), ptr, n, on_host,
        _stream_handle(stream, dev))
    del keep
    _native.check("paged_kv_zero_and_write", st)


def _block_ids(ids, dev):
    """(pointer, count, ids_on_host, keep-alive) for a block-id list."""
    if isinstance(ids, torch.Tensor) and ids.is_cuda:
        _require(ids, "block ids", torch.int32, dev, 1)
        return ids.data_ptr(), ids.numel(), 0, ids
    if isinstance(ids, torch.Tensor):
        ids = ids.numpy()
    keep = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    return keep.ctypes.data, keep.size, 1, keep


def paged_kv_copy_blocks(cache: PagedKVCache, src_ids, dst_ids,
                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy blocks src_ids[i] -> dst_ids[i] in both caches (copy-on-write
    of shared blocks).  Ids: host arrays/lists or CUDA int32 tensors."""
    dev = cache.device
    sp, sn, s_host, s_keep = _block_ids(src_ids, dev)
    dp, dn, d_host, d_keep = _block_ids(dst_ids, dev)
    if sn != dn or s_host != d_host:
        raise ValueError("src_ids and dst_ids must match in length and place")
    st = _native.lib().paged_kv_copy_blocks(
        ctypes.byref(cache.c_struct()), sp, dp, sn, s_host,
        _stream_handle(stream, dev))
    del s_keep, d_keep
    _native.check("paged_kv_copy_blocks", st)


def _check_pinned(t: torch.Tensor, name: str, nbytes: int):
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned():
        raise ValueError(f"{name} must be a pinned CPU tensor")
    if not t.is_contiguous() or t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} must be contiguous with >= {nbytes} bytes")


def paged_kv_swap_out(cache: PagedKVCache, block_ids, host_k: torch.Tensor,
                      host_v: torch.Tensor,
                      stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy blocks to pinned host tensors (packed in id order)."""
    dev = cache.device
    p, n, on_host, keep = _block_ids(block_ids, dev)
    nbytes = n * cache.block_bytes
    _check_pinned(host_k, "host_k", nbytes)
    _check_pinned(host_v, "host_v", nbytes)
    st = _native.lib().paged_kv_swap_out(
        ctypes.byref(cache.c_struct()), p, n, on_host, host_k.data_ptr(),
        host_v.data_ptr(), _stream_handle(stream, dev))
    del keep
    _native.check("paged_kv_swap_out", st)


def paged_kv_swap_in(cache: PagedKVCache, block_ids, host_k: torch.Tensor,
                     host_v: torch.Tensor,
                     stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy packed blocks from pinned host tensors into the cache."""
    dev = cache.device
    p, n, on_host, keep = _block_ids(block_ids, dev)
    nbytes = n * cache.block_bytes
    _check_pinned(host_k, "host_k", nbytes)
    _check_pinned(host_v, "host_v", nbytes)
    st = _native.lib().paged_kv_swap_in(
        ctypes.byref(cache.c_struct()), p, n, on_host, host_k.data_ptr(),
        host_v.data_ptr(), _stream_handle(stream, dev))
    del keep
    _native.check("paged_kv_swap_in", st)


def paged_prepare_inputs(idx_mapping: torch.Tensor,
                         num_scheduled: torch.Tensor,
                         state_block_table: torch.Tensor,
                         state_num_computed: torch.Tensor,
                         state_token_ids: torch.Tensor, total_tokens: int,
                         out: Optional[dict] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> dict:
    """Gather one step's inputs from the persistent request state table
    (all int32 CUDA tensors).  Returns block_tables, seq_lens,
    query_start_loc, positions, input_ids and slot_mapping (written into
    ``out`` when given, e.g. a previous call's result)."""
    dev = state_block_table.device
    for t, n, nd in ((idx_mapping, "idx_mapping", 1),
                     (num_scheduled, "num_scheduled", 1),
                     (state_block_table, "state_block_table", 2),
                     (state_num_computed, "state_num_computed", 1),
                     (state_token_ids, "state_token_ids", 2)):
        _require(t, n, torch.int32, dev, nd)
    B = idx_mapping.shape[0]
    R, MB = state_block_table.shape
    if num_scheduled.shape[0] != B or state_num_computed.shape[0] != R or \
            state_token_ids.shape[0] != R:
        raise ValueError("state table and batch shapes do not match")
    T = int(total_tokens)
    shapes = {"block_tables": ((B, MB), torch.int32),
              "seq_lens": ((B,), torch.int32),
              "query_start_loc": ((B + 1,), torch.int32),
              "positions": ((T,), torch.int32),
              "input_ids": ((T,), torch.int32),
              "slot_mapping": ((T,), torch.int64)}
    if out is None:
        out = {k: torch.empty(sh, dtype=dt, device=dev)
               for k, (sh, dt) in shapes.items()}
    else:
        for k, (sh, dt) in shapes.items():
            _require(out[k], k, dt, dev, len(sh))
            if tuple(out[k].shape) != sh:
                raise ValueError(f"out[{k!r}] must have shape {sh}")
    st = _native.lib().paged_prepare_inputs(
        idx_mapping.data_ptr(), num_scheduled.data_ptr(), B,
        state_block_table.data_ptr(), MB, state_num_computed.data_ptr(),
        state_token_ids.data_ptr(), state_token_ids.shape[1], R, T,
        out["block_tables"].data_ptr(), out["seq_lens"].data_ptr(),
        out["query_start_loc"].data_ptr(), out["positions"].data_ptr(),
        out["input_ids"].data_ptr(), out["slot_mapping"].data_ptr(),
        _stream_handle(stream, dev))
    _native.check("paged_prepare_inputs", st)
    return out


def paged_attention_workspace_bytes(batch: int, num_heads: int,
                                    num_kv_heads: int, head_dim: int,
                                    max_seq_len: int,
                                    partition_tokens: int = 0) -> int:
    return int(_native.lib().paged_attention_workspace_bytes(
        batch, num_heads, num_kv_heads, head_dim, max_seq_len,
        partition_tokens))


def paged_attention_partition_tokens(batch: int, num_heads: int,
                                     num_kv_heads: int, max_seq_len: int,
                                     partition_tokens: int = 0) -> int:
    return int(_native.lib().paged_attention_partition_tokens(
        batch, num_heads, num_kv_heads, max_seq_len, partition_tokens))


def paged_attention_decode(q: torch.Tensor, cache: PagedKVCache,
                           block_tables: torch.Tensor,
                           seq_lens: torch.Tensor, scale: float,
                           max_seq_len: int, out: Optional[torch.Tensor] = None,
                           partition_tokens: int = 0,
                           workspace: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None
                           ) -> torch.Tensor:
    """Decode attention: q [B, Hq, d] bf16, block_tables int32 [B,
    max_blocks], seq_lens int32 [B] (device), max_seq_len a host bound of
    seq_lens.  Returns out [B, Hq, d] bf16."""
    return _decode("paged_attention_decode", q, None, None, cache,
                   block_tables, seq_lens, scale, max_seq_len, out,
                   partition_tokens, workspace, stream)


def paged_attention_decode_step(q: torch.Tensor, k_new: torch.Tensor,
                                v_new: torch.Tensor, cache: PagedKVCache,
                                block_tables: torch.Tensor,
                                seq_lens: torch.Tensor, scale: float,
                                max_seq_len: int,
                                out: Optional[torch.Tensor] = None,
                                partition_tokens: int = 0,
                                workspace: Optional[torch.Tensor] = None,
                                stream: Optional[torch.cuda.Stream] = None,
                                new_start_loc: Optional[torch.Tensor] = None
                                ) -> torch.Tensor:
    """One decode step: the new tokens' K and V (k_new / v_new [N, Hkv, d]
    bf16) are written into the cache, then attention as
    paged_attention_decode.  Without new_start_loc, N = B and row b is
    sequence b's token at position seq_lens[b] - 1; with it (int32 [B + 1],
    device), rows new_start_loc[b] .. new_start_loc[b+1] - 1 are sequence
    b's last positions.  Blocks whose first position is new have their
    rows past the sequence zeroed.  Returns out [B, Hq, d] bf16."""
    return _decode("paged_attention_decode_step", q, k_new, v_new, cache,
                   block_tables, seq_lens, scale, max_seq_len, out,
                   partition_tokens, workspace, stream, new_start_loc)


def _decode(name, q, k_new, v_new, cache, block_tables, seq_lens, scale,
            max_seq_len, out, partition_tokens, workspace, stream,
            new_start_loc=None):
    dev = cache.device
    _require(q, "q", torch.bfloat16, dev, 3)
    _require(block_tables, "block_tables", torch.int32, dev, 2)
    _require(seq_lens, "seq_lens", torch.int32, dev, 1)
    B, Hq, d = q.shape
    if d != cache.head_dim or block_tables.shape[0] != B or \
            seq_lens.shape[0] != B:
        raise ValueError("q, block_tables, seq_lens shapes do not match")
    if out is None:
        out = torch.empty_like(q)
    else:
        _require(out, "out", torch.bfloat16, dev, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    need = paged_attention_workspace_bytes(B, Hq, cache.num_kv_heads, d,
                                           max_seq_len, partition_tokens)
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _require(workspace, "workspace", torch.uint8, dev, 1)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    common = (ctypes.byref(cache.c_struct()), block_tables.data_ptr(),
              block_tables.shape[1], seq_lens.data_ptr(), B, Hq, float(scale),
              out.data_ptr(), int(max_seq_len), int(partition_tokens), ws_ptr,
              ws_bytes, _stream_handle(stream, dev))
    if k_new is None:
        st = _native.lib().paged_attention_decode(q.data_ptr(), *common)
    else:
        n_new = k_new.shape[0] if k_new.dim() == 3 else -1
        for t, n in ((k_new, "k_new"), (v_new, "v_new")):
            _require(t, n, torch.bfloat16, dev, 3)
            if t.shape != (n_new, cache.num_kv_heads, d):
                raise ValueError(f"{n} must be [num_new, num_kv_heads, head_dim]")
        nsl = None
        if new_start_loc is not None:
            _require(new_start_loc, "new_start_loc", torch.int32, dev, 1)
            if new_start_loc.shape[0] != B + 1:
                raise ValueError("new_start_loc must be [batch + 1]")
            nsl = new_start_loc.data_ptr()
        elif n_new != B:
            raise ValueError("without new_start_loc, k_new holds one row per sequence")
        st = _native.lib().paged_attention_decode_step(
            q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), nsl, n_new, *common)
    _native.check(name, st)
    return out


def paged_attention_cascade_workspace_bytes(batch: int, num_heads: int,
                                            num_kv_heads: int, head_dim: int,
                                            max_seq_len: int, max_prefix_len: int,
                                            partition_tokens: int = 0) -> int:
    """Device workspace bytes paged_attention_decode_cascade needs."""
    return int(_native.lib().paged_attention_cascade_workspace_bytes(
        batch, num_heads, num_kv_heads, head_dim, max_seq_len, max_prefix_len,
        partition_tokens))


def paged_attention_decode_cascade(q: torch.Tensor, cache: PagedKVCache,
                                   block_tables: torch.Tensor,
                                   seq_lens: torch.Tensor,
                                   group_start: torch.Tensor,
                                   prefix_len: torch.Tensor, scale: float,
                                   max_seq_len: int, max_group_size: int,
                                   max_prefix_len: int,
                                   out: Optional[torch.Tensor] = None,
                                   partition_tokens: int = 0,
                                   workspace: Optional[torch.Tensor] = None,
                                   stream: Optional[torch.cuda.Stream] = None
                                   ) -> torch.Tensor:
    """Decode attention with each group's shared prefix attended once for
    all its members: group_start int32 [G+1] (members are consecutive
    sequences), prefix_len int32 [G] (multiples of 16).  Same arguments and
    result as paged_attention_decode otherwise."""
    dev = cache.device
    _require(q, "q", torch.bfloat16, dev, 3)
    _require(block_tables, "block_tables", torch.int32, dev, 2)
    _require(seq_lens, "seq_lens", torch.int32, dev, 1)
    _require(group_start, "group_start", torch.int32, dev, 1)
    _require(prefix_len, "prefix_len", torch.int32, dev, 1)
    B, Hq, d = q.shape
    G = prefix_len.shape[0]
    if d != cache.head_dim or block_tables.shape[0] != B or \
            seq_lens.shape[0] != B or group_start.shape[0] != G + 1:
        raise ValueError("q, block_tables, seq_lens, group_start, prefix_len "
                         "shapes do not match")
    if out is None:
        out = torch.empty_like(q)
    else:
        _require(out, "out", torch.bfloat16, dev, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    need = paged_attention_cascade_workspace_bytes(
        B, Hq, cache.num_kv_heads, d, max_seq_len, max_prefix_len,
        partition_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _require(workspace, "workspace", torch.uint8, dev, 1)
    st = _native.lib().paged_attention_decode_cascade(
        q.data_ptr(), ctypes.byref(cache.c_struct()), block_tables.data_ptr(),
        block_tables.shape[1], seq_lens.data_ptr(), B, Hq,
        group_start.data_ptr(), prefix_len.data_ptr(), G, int(max_group_size),
        int(max_prefix_len), float(scale), out.data_ptr(), int(max_seq_len),
        int(partition_tokens), workspace.data_ptr(), workspace.numel(),
        _stream_handle(stream, dev))
    _native.check("paged_attention_decode_cascade", st)
    return out


def paged_attention_prefill(q: torch.Tensor, cache: PagedKVCache,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor,
                            query_start_loc: torch.Tensor, scale: float,
                            max_query_len: int,
                            out: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None
                            ) -> torch.Tensor:
    """Prefill / chunked-prefill attention, causal within each sequence:
    q [T, Hq, d] bf16 (all sequences' query tokens back to back),
    query_start_loc int32 [B+1], seq_lens int32 [B] (cached tokens
    including the chunk), max_query_len a host bound of the chunk lengths.
    Returns out [T, Hq, d] bf16."""
    dev = cache.device
    _require(q, "q", torch.bfloat16, dev, 3)
    _require(block_tables, "block_tables", torch.int32, dev, 2)
    _require(seq_lens, "seq_lens", torch.int32, dev, 1)
    _require(query_start_loc, "query_start_loc", torch.int32, dev, 1)
    T, Hq, d = q.shape
    B = seq_lens.shape[0]
    if d != cache.head_dim or block_tables.shape[0] != B or \
            query_start_loc.shape[0] != B + 1:
        raise ValueError("q, block_tables, seq_lens, query_start_loc shapes "
                         "do not match")
    if out is None:
        out = torch.empty_like(q)
    else:
        _require(out, "out", torch.bfloat16, dev, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    st = _native.lib().paged_attention_prefill(
        q.data_ptr(), ctypes.byref(cache.c_struct()), block_tables.data_ptr(),
        block_tables.shape[1], seq_lens.data_ptr(), query_start_loc.data_ptr(),
        B, Hq, T, float(scale), out.data_ptr(), int(max_query_len),
        _stream_handle(stream, dev))
    _native.check("paged_attention_prefill", st)
    return out


def pkv_check(stream: Optional[torch.cuda.Stream] = None, device=None):
    """Synchronise the stream and return (status, detail) from the device
    error word, clearing it."""
    detail = ctypes.c_int64(-1)
    st = _native.lib().pkv_check(_stream_handle(stream, device),
                                 ctypes.byref(detail))
    return int(st), int(detail.value)


def raise_on_device_error(stream: Optional[torch.cuda.Stream] = None,
                          device=None) -> None:
    st, detail = pkv_check(stream, device)
    if st != _native.PKV_OK:
        raise PagedKVError("device check", st, detail)
