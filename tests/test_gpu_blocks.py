"""Block copy (copy-on-write) and swap out/in against the oracle: bit-exact."""
import ctypes

import numpy as np
import pytest
import torch

import harness
import oracle
from paged_kv_cache_48_gb300 import (PagedKVCache, PagedKVError, _native,
                                     paged_attention_decode,
                                     paged_kv_copy_blocks, paged_kv_swap_in,
                                     paged_kv_swap_out, paged_kv_write,
                                     pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu
PKV_OK, PKV_ERR_ARG, PKV_ERR_RANGE = 0, 1, 5


def _random_cache(kv_dtype, NB=300, Hkv=8, d=128, seed=0):
    rng = np.random.default_rng(seed)
    elt = 2 if kv_dtype == "bf16" else 1
    nbytes = NB * 16 * Hkv * d * elt
    hk = rng.integers(0, 256, nbytes, dtype=np.uint8)
    hv = rng.integers(0, 256, nbytes, dtype=np.uint8)
    dt = torch.bfloat16 if kv_dtype == "bf16" else torch.uint8
    shape = (NB, 16, Hkv, d)
    kc = torch.from_numpy(hk.copy()).view(dt).reshape(shape).cuda()
    vc = torch.from_numpy(hv.copy()).view(dt).reshape(shape).cuda()
    return PagedKVCache(kc, vc, kv_dtype, 0.5, 0.25), hk, hv, rng


def _bytes(t):
    return t.view(torch.uint8).cpu().numpy().reshape(-1)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("on_host", [True, False])
def test_copy_blocks_matches_oracle(kv_dtype, on_host):
    cache, hk, hv, rng = _random_cache(kv_dtype)
    perm = rng.permutation(cache.num_blocks).astype(np.int32)
    src, dst = perm[:100], perm[100:200]  # disjoint pairs
    if on_host:
        paged_kv_copy_blocks(cache, src, dst)
    else:
        paged_kv_copy_blocks(cache, torch.from_numpy(src).cuda(),
                             torch.from_numpy(dst).cuda())
    assert pkv_check()[0] == PKV_OK
    oracle.load().copy_blocks(hk, hv, cache.block_bytes, src, dst)
    assert np.array_equal(_bytes(cache.key_cache), hk)
    assert np.array_equal(_bytes(cache.value_cache), hv)


def test_copy_blocks_many_ids_and_range_errors():
    cache, hk, hv, rng = _random_cache("fp8_e4m3", NB=5000, Hkv=1, d=64)
    perm = rng.permutation(cache.num_blocks).astype(np.int32)
    src, dst = perm[:2400], perm[2400:4800]  # two launches of host ids
    paged_kv_copy_blocks(cache, src, dst)
    assert pkv_check()[0] == PKV_OK
    oracle.load().copy_blocks(hk, hv, cache.block_bytes, src, dst)
    assert np.array_equal(_bytes(cache.key_cache), hk)
    paged_kv_copy_blocks(cache, np.array([1, cache.num_blocks], np.int32),
                         np.array([-1, 2], np.int32))
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail in (0, 1)
    assert np.array_equal(_bytes(cache.key_cache), hk)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("on_host", [True, False])
def test_swap_out_then_in_matches_oracle(kv_dtype, on_host):
    cache, hk, hv, rng = _random_cache(kv_dtype, seed=3)
    bb = cache.block_bytes
    perm = rng.permutation(cache.num_blocks).astype(np.int32)
    ids_out, ids_in = perm[:70], perm[70:140]
    host_k = torch.zeros(70 * bb, dtype=torch.uint8).pin_memory()
    host_v = torch.zeros(70 * bb, dtype=torch.uint8).pin_memory()
    arg = (lambda a: a) if on_host else (lambda a: torch.from_numpy(a).cuda())
    paged_kv_swap_out(cache, arg(ids_out), host_k, host_v)
    assert pkv_check()[0] == PKV_OK
    ok, ov, err = oracle.load().swap_out(hk, hv, bb, ids_out)
    assert err == 0
    assert np.array_equal(host_k.numpy(), ok)
    assert np.array_equal(host_v.numpy(), ov)
    paged_kv_swap_in(cache, arg(ids_in), host_k, host_v)
    assert pkv_check()[0] == PKV_OK
    oracle.load().swap_in(hk, hv, bb, ids_in, ok, ov)
    assert np.array_equal(_bytes(cache.key_cache), hk)
    assert np.array_equal(_bytes(cache.value_cache), hv)


def test_swap_rejects_pageable_host_memory():
    cache, hk, hv, rng = _random_cache("bf16", NB=8, seed=4)
    pageable = np.zeros(2 * cache.block_bytes, np.uint8)
    ids = np.array([1, 2], np.int32)
    st = _native.lib().paged_kv_swap_out(
        ctypes.byref(cache.c_struct()), ids.ctypes.data, 2, 1,
        pageable.ctypes.data, pageable.ctypes.data,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == PKV_ERR_ARG
    with pytest.raises(ValueError):
        paged_kv_swap_out(cache, ids, torch.zeros(2 * cache.block_bytes,
                                                  dtype=torch.uint8),
                          torch.zeros(2 * cache.block_bytes, dtype=torch.uint8))
    assert np.array_equal(_bytes(cache.key_cache), hk)


def test_copy_on_write_of_a_shared_prefix_block():
    """A group shares its prefix blocks (refcount > 1).  One member diverges
    inside the last prefix block: the block is copied to a fresh one, the
    member's table points at the copy, and its new token is written there.
    The other members still read the untouched original; every output
    matches the oracle on the same operations."""
    W = wl.prefix_shared(small=True)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    kc_o, vc_o = harness.oracle_cache(W)
    grp = W.groups[0]
    member = grp["members"][1]
    shared = grp["prefix_blocks"][-1]
    used = set(int(x) for x in W.block_tables[W.block_tables >= 0])
    fresh = next(b for b in range(W.num_blocks) if b not in used)
    # GPU: copy, re-point, overwrite token 5 of the copied block
    paged_kv_copy_blocks(G.cache, np.array([shared], np.int32),
                         np.array([fresh], np.int32))
    tables = W.block_tables.copy()
    j = len(grp["prefix_blocks"]) - 1
    tables[member, j] = fresh
    rng = np.random.default_rng(11)
    k_new = wl.bf16_bits(rng.standard_normal((1, W.num_kv_heads, W.head_dim)).astype(np.float32))
    v_new = wl.bf16_bits(rng.standard_normal((1, W.num_kv_heads, W.head_dim)).astype(np.float32))
    slot = np.array([fresh * 16 + 5], np.int64)
    paged_kv_write(harness._u16_to_bf16(k_new, "cuda"), harness._u16_to_bf16(v_new, "cuda"),
                   torch.from_numpy(slot).cuda(), G.cache)
    out = paged_attention_decode(G.q, G.cache, torch.from_numpy(tables).cuda(),
                                 G.seq_lens, W.scale, max_seq_len=W.max_seq_len)
    assert pkv_check()[0] == PKV_OK
    # oracle: the same three operations on its own cache
    o = oracle.load()
    assert o.copy_blocks(kc_o, vc_o, W.block_bytes, [shared], [fresh]) == 0
    assert o.kv_write(kc_o, vc_o, oracle.DTYPE_BF16, 16, W.num_kv_heads,
                      W.head_dim, 1.0, 1.0, k_new, v_new, slot) == 0
    assert np.array_equal(_bytes(G.cache.key_cache), kc_o)
    assert np.array_equal(_bytes(G.cache.value_cache), vc_o)
    W2 = wl.Workload(**{**W.__dict__})
    W2.block_tables = tables
    ref = harness.oracle_out(W2, kc_o, vc_o)
    harness.assert_close(out.float().cpu().numpy(), ref, "bf16")
    # the other members still see the original block
    other = grp["members"][0]
    assert W.block_tables[other, j] == shared
