"""paged_attention_decode_noalloc: decode attention for callers that cannot
allocate device memory (for example code running inside an allocator or
under a fully committed memory budget), using the library's fixed device
scratch array instead of a caller workspace.

Called through the C ABI and compared with paged_attention_decode (given a
workspace) within the parity tolerance, on two calls in a row, so that a
second call over the scratch the first one left behind is covered too.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import harness
from paged_kv_cache_48_gb300 import _native
from paged_kv_cache_48_gb300 import workload as wl
from paged_kv_cache_48_gb300.ops import paged_attention_workspace_bytes

pytestmark = pytest.mark.gpu
PKV_OK, PKV_ERR_ARG, PKV_ERR_WORKSPACE = 0, 1, 7


def _call_existing(W, G, pt):
    out = torch.empty_like(G.q)
    need = paged_attention_workspace_bytes(W.batch, W.num_heads,
                                           W.num_kv_heads, W.head_dim,
                                           W.max_seq_len, pt)
    assert need > 0  # the case must exercise the scratch
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = _native.lib().paged_attention_decode(
        G.q.data_ptr(), ctypes.byref(G.cache.c_struct()), G.tables.data_ptr(),
        G.tables.shape[1], G.seq_lens.data_ptr(), W.batch, W.num_heads,
        W.scale, out.data_ptr(), W.max_seq_len, pt, ws.data_ptr(), need,
        stream)
    assert st == PKV_OK
    torch.cuda.synchronize()
    return out


def _call_noalloc(W, G, pt, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return _native.lib().paged_attention_decode_noalloc(
        G.q.data_ptr(), ctypes.byref(G.cache.c_struct()), G.tables.data_ptr(),
        G.tables.shape[1], G.seq_lens.data_ptr(), W.batch, W.num_heads,
        W.scale, out.data_ptr(), W.max_seq_len, pt, stream)


@pytest.mark.parametrize("make,pt", [
    (lambda: wl.llama8b_gqa(small=True), 64),
    (lambda: wl.fp8_recycle(small=True), 32),
    (lambda: wl.long_context(small=True), 512),
], ids=["bf16_gqa", "fp8", "long_context"])
def test_noalloc_matches_workspace_entry_point_twice(make, pt):
    W = make()
    G = harness.upload(W)
    harness.gpu_step(W, G)  # zero + write the step's tokens
    ref = _call_existing(W, G, pt).float().cpu().numpy()
    for _ in range(2):
        out = torch.full_like(G.q, float("nan"))
        assert _call_noalloc(W, G, pt, out) == PKV_OK
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        atol, rtol = harness.TOL[W.kv_dtype]
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - ref) <= atol + rtol * np.abs(ref))
    assert harness.pkv_check()[0] == PKV_OK


def _call_noalloc_sized(W, G, out, max_seq_len, pt):
    return _native.lib().paged_attention_decode_noalloc(
        G.q.data_ptr(), ctypes.byref(G.cache.c_struct()), G.tables.data_ptr(),
        G.tables.shape[1], G.seq_lens.data_ptr(), W.batch, W.num_heads,
        W.scale, out.data_ptr(), max_seq_len, pt,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_rejects_needs_beyond_its_scratch():
    W = wl.tiny_mha()
    G = harness.upload(W)
    out = torch.empty_like(G.q)
    assert _call_noalloc(W, G, 16, out) == PKV_OK  # small need: fine
    # 65535 partitions of 16 tokens: a valid grid whose partials (4 x 8 x
    # 65535 rows) need far more than the fixed scratch; rejected on the
    # host, nothing launched.
    most = 16 * 65535
    need = paged_attention_workspace_bytes(W.batch, W.num_heads,
                                           W.num_kv_heads, W.head_dim, most, 16)
    assert need > _native.PKV_NOALLOC_SCRATCH_BYTES
    assert _call_noalloc_sized(W, G, out, most, 16) == PKV_ERR_WORKSPACE
    # one partition more is an invalid grid: the answer
    # paged_attention_decode gives, whatever the scratch size
    assert _call_noalloc_sized(W, G, out, most + 16, 16) == PKV_ERR_ARG
    torch.cuda.synchronize()


def test_noalloc_takes_no_device_memory_after_its_first_call():
    """The first call on a device may load the scratch array (and take its
    16 MiB then); every later call leaves the device's free memory as it
    was."""
    W = wl.llama8b_gqa(small=True)
    G = harness.upload(W)
    out = torch.empty_like(G.q)
    assert _call_noalloc(W, G, 64, out) == PKV_OK   # set-up call
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _call_noalloc(W, G, 64, out) == PKV_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert harness.pkv_check()[0] == PKV_OK
