"""paged_kv_zero_and_write (zeroing of fresh blocks and the slot-mapped
write in one launch) against the oracle's zeroing followed by its write:
byte-exact caches.  The cases put tokens in fresh blocks (the rows the
zeroing must leave to the write), in other blocks, and padding slots; they
repeat fresh ids, pass more host ids than one launch carries, and plant out
of range ids and slots."""
import numpy as np
import pytest
import torch

import harness
import oracle
from paged_kv_cache_48_gb300 import (PagedKVCache, paged_kv_zero_and_write,
                                     pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu
PKV_OK, PKV_ERR_RANGE = 0, 5
DT = {"bf16": oracle.DTYPE_BF16, "fp8_e4m3": oracle.DTYPE_FP8_E4M3}


@pytest.mark.parametrize("ids_on_device", [False, True], ids=["host_ids", "device_ids"])
@pytest.mark.parametrize("make", [
    wl.tiny_mha,
    lambda: wl.llama8b_gqa(small=True),
    lambda: wl.fp8_recycle(small=True),
], ids=["tiny", "llama_small", "fp8_small"])
def test_decode_step_matches_zero_then_write(make, ids_on_device):
    W = make()
    G = harness.upload(W)
    ids = torch.from_numpy(W.fresh_blocks).cuda() if ids_on_device else W.fresh_blocks
    paged_kv_zero_and_write(G.step_k, G.step_v, G.step_slots, G.cache, ids)
    assert pkv_check()[0] == PKV_OK
    kc, vc = harness.oracle_cache(W)
    assert np.array_equal(G.cache.key_cache.view(torch.uint8).cpu().numpy().reshape(-1), kc)
    assert np.array_equal(G.cache.value_cache.view(torch.uint8).cpu().numpy().reshape(-1), vc)


def _synthetic(kv_dtype, NB, Hkv, d, T, n_fresh, seed, pad_every=7):
    """A pool of stale bytes, fresh ids (one repeated), and T tokens of which
    about half land in fresh blocks (partial rows) and some are padding."""
    rng = np.random.default_rng(seed)
    elt = 1 if kv_dtype == "fp8_e4m3" else 2
    block_bytes = 16 * Hkv * d * elt
    init_k = rng.integers(0, 256, NB * block_bytes, dtype=np.uint8)
    init_v = rng.integers(0, 256, NB * block_bytes, dtype=np.uint8)
    fresh = rng.choice(NB, n_fresh, replace=False).astype(np.int32)
    fresh = np.concatenate([fresh, fresh[:1]])  # a repeated id
    in_fresh = fresh[rng.integers(0, n_fresh, T // 2)].astype(np.int64) * 16 + \
        rng.integers(0, 16, T // 2)
    others = np.setdiff1d(np.arange(NB * 16), np.concatenate(
        [np.arange(b * 16, b * 16 + 16) for b in fresh]))
    rest = rng.choice(others, T - T // 2, replace=False)
    slots = np.concatenate([np.unique(in_fresh), rest])
    slots = slots[rng.permutation(slots.size)].astype(np.int64)
    slots[::pad_every] = -1
    T = slots.size
    k = wl.bf16_bits(rng.standard_normal((T, Hkv, d)).astype(np.float32))
    v = wl.bf16_bits(rng.standard_normal((T, Hkv, d)).astype(np.float32))
    return init_k, init_v, block_bytes, fresh, slots, k, v


def _run(kv_dtype, NB, Hkv, d, init_k, init_v, fresh, slots, k, v, ids_on_device=False):
    shape = (NB, 16, Hkv, d)
    dt = torch.uint8 if kv_dtype == "fp8_e4m3" else torch.bfloat16
    kc = torch.from_numpy(init_k).view(dt).reshape(shape).cuda()
    vc = torch.from_numpy(init_v).view(dt).reshape(shape).cuda()
    scale = 0.25 if kv_dtype == "fp8_e4m3" else 1.0
    cache = PagedKVCache(kc, vc, kv_dtype, scale, scale)
    kt = torch.from_numpy(k).view(torch.bfloat16).cuda()
    vt = torch.from_numpy(v).view(torch.bfloat16).cuda()
    ids = torch.from_numpy(fresh).cuda() if ids_on_device else fresh
    paged_kv_zero_and_write(kt, vt, torch.from_numpy(slots).cuda(), cache, ids)
    st = pkv_check()
    return (kc.view(torch.uint8).cpu().numpy().reshape(-1),
            vc.view(torch.uint8).cpu().numpy().reshape(-1), st, scale)


def _oracle(kv_dtype, Hkv, d, init_k, init_v, block_bytes, fresh, slots, k, v, scale):
    o = oracle.load()
    ok, ov = init_k.copy(), init_v.copy()
    e1 = o.zero_blocks(ok, ov, block_bytes, fresh)
    e2 = o.kv_write(ok, ov, DT[kv_dtype], 16, Hkv, d, scale, scale, k, v, slots)
    return ok, ov, e1, e2


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("ids_on_device", [False, True], ids=["host_ids", "device_ids"])
def test_tokens_in_fresh_and_old_blocks(kv_dtype, ids_on_device):
    NB, Hkv, d = 96, 2, 128
    ik, iv, bb, fresh, slots, k, v = _synthetic(kv_dtype, NB, Hkv, d, 300, 20, seed=11)
    gk, gv, st, scale = _run(kv_dtype, NB, Hkv, d, ik, iv, fresh, slots, k, v, ids_on_device)
    ok, ov, e1, e2 = _oracle(kv_dtype, Hkv, d, ik, iv, bb, fresh, slots, k, v, scale)
    assert st[0] == PKV_OK and e1 == 0 and e2 == 0
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_more_host_ids_than_one_launch_carries():
    """4500 fresh ids: two launches; tokens land in blocks of both."""
    NB, Hkv, d = 5000, 1, 64
    ik, iv, bb, fresh, slots, k, v = _synthetic("bf16", NB, Hkv, d, 600, 4500, seed=12)
    gk, gv, st, scale = _run("bf16", NB, Hkv, d, ik, iv, fresh, slots, k, v)
    ok, ov, _, _ = _oracle("bf16", Hkv, d, ik, iv, bb, fresh, slots, k, v, scale)
    assert st[0] == PKV_OK
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_only_zero_and_only_write():
    NB, Hkv, d = 40, 2, 64
    ik, iv, bb, fresh, slots, k, v = _synthetic("bf16", NB, Hkv, d, 50, 6, seed=13)
    # zero only
    gk, gv, st, _ = _run("bf16", NB, Hkv, d, ik, iv, fresh, slots[:0], k[:0], v[:0])
    ok, ov, _, _ = _oracle("bf16", Hkv, d, ik, iv, bb, fresh, slots[:0], k[:0], v[:0], 1.0)
    assert st[0] == PKV_OK and np.array_equal(gk, ok) and np.array_equal(gv, ov)
    # write only
    none = np.zeros(0, np.int32)
    gk, gv, st, _ = _run("bf16", NB, Hkv, d, ik, iv, none, slots, k, v)
    ok, ov, _, _ = _oracle("bf16", Hkv, d, ik, iv, bb, none, slots, k, v, 1.0)
    assert st[0] == PKV_OK and np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_range_errors_are_reported_and_the_rest_is_done():
    NB, Hkv, d = 40, 2, 64
    ik, iv, bb, fresh, slots, k, v = _synthetic("bf16", NB, Hkv, d, 60, 5, seed=14)
    bad_ids = np.concatenate([fresh, np.array([NB + 7], np.int32)])
    gk, gv, st, _ = _run("bf16", NB, Hkv, d, ik, iv, bad_ids, slots, k, v)
    assert st[0] == PKV_ERR_RANGE
    ok, ov, e1, _ = _oracle("bf16", Hkv, d, ik, iv, bb, fresh, slots, k, v, 1.0)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)
    # an out-of-range slot: reported, the other tokens written
    bad_slots = slots.copy()
    j = int(np.flatnonzero(bad_slots >= 0)[0])
    bad_slots[j] = NB * 16 + 3
    gk, gv, st, _ = _run("bf16", NB, Hkv, d, ik, iv, fresh, bad_slots, k, v)
    assert st[0] == PKV_ERR_RANGE
    keep = bad_slots.copy()
    keep[j] = -1
    ok, ov, _, _ = _oracle("bf16", Hkv, d, ik, iv, bb, fresh, keep, k, v, 1.0)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)
