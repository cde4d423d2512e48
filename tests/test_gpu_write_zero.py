"""CUDA slot-mapped write and block zeroing against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import harness
import oracle
from paged_kv_cache_48_gb300 import (PagedKVCache, PagedKVError,
                                     paged_kv_write, paged_kv_zero_and_write,
                                     paged_kv_zero_blocks, pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu
PKV_OK, PKV_ERR_RANGE = 0, 5


def _pool(W):
    G = harness.upload(W, write_history=False)
    return G


@pytest.mark.parametrize("make", [
    wl.tiny_mha,
    lambda: wl.llama8b_gqa(small=True),
    lambda: wl.prefix_shared(small=True),
    lambda: wl.fp8_recycle(small=True),
    lambda: wl.make_workload("fp8_d64", 3, 4, 2, 64, 5, 90, 41,
                             kv_dtype="fp8_e4m3", fresh_policy="recycle515"),
], ids=["tiny", "llama_small", "prefix_small", "fp8_small", "fp8_d64"])
def test_full_write_zero_write_is_bit_exact(make):
    W = make()
    res = harness.run_gpu(W)
    assert res["status"] == PKV_OK
    kc, vc = harness.oracle_cache(W)
    assert np.array_equal(res["key"], kc)
    assert np.array_equal(res["value"], vc)


def test_fp8_write_extremes_bit_exact():
    """Values at the scale's edge (saturation to 448), ties, tiny values
    that round to signed zero, and subnormal codes."""
    rng = np.random.default_rng(5)
    NB, Hkv, d, T = 8, 2, 64, 100
    x = rng.standard_normal((T, Hkv, d)).astype(np.float32)
    x[0, 0, :8] = [448 * 0.5, -448 * 0.5, 1e-9, -1e-9, 600, -600, 0.0, -0.0]
    x[1] *= 1e-3
    bits = wl.bf16_bits(x)
    scale = np.float32(0.5)
    slots = rng.permutation(NB * 16)[:T].astype(np.int64)
    shape = (NB, 16, Hkv, d)
    kc = torch.full(shape, 0xAB, dtype=torch.uint8, device="cuda")
    vc = torch.full(shape, 0xCD, dtype=torch.uint8, device="cuda")
    cache = PagedKVCache(kc, vc, "fp8_e4m3", float(scale), float(scale))
    kt = torch.from_numpy(bits).view(torch.bfloat16).cuda()
    paged_kv_write(kt, kt, torch.from_numpy(slots).cuda(), cache)
    assert pkv_check()[0] == PKV_OK
    ok = np.full(NB * 16 * Hkv * d, 0xAB, np.uint8)
    ov = np.full(NB * 16 * Hkv * d, 0xCD, np.uint8)
    oracle.load().kv_write(ok, ov, oracle.DTYPE_FP8_E4M3, 16, Hkv, d,
                           float(scale), float(scale), bits, bits, slots)
    assert np.array_equal(kc.cpu().numpy().reshape(-1), ok)
    assert np.array_equal(vc.cpu().numpy().reshape(-1), ov)


_E4M3_SCALES = [1.0, 0.5, 3.0, 0.0123, 4.7 / 448, 1e30, 3e-38, 1e-39]


@pytest.mark.parametrize("fused", [False, True], ids=["write", "zero_and_write"])
@pytest.mark.parametrize("scale", _E4M3_SCALES)
def test_fp8_encode_every_bf16_value(scale, fused):
    """Every bf16 bit pattern through the E4M3 encode, for scales that make
    the quotient exact (1, 0.5), put ties within an ulp of x * RN(1/scale)
    (3), are awkward (0.0123, 4.7/448), large, tiny, or subnormal (the
    reciprocal overflows).  Bytes equal the oracle's IEEE quotient rounded
    to E4M3 for every value that is not a NaN; NaN inputs give a NaN code
    (0x7F or 0xFF) on both sides."""
    Hkv, d = 1, 128
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    T = allbits.size // (Hkv * d)
    NB = T // 16
    kbits = allbits.reshape(T, Hkv, d)
    vbits = allbits[::-1].copy().reshape(T, Hkv, d)
    slots = np.random.default_rng(9).permutation(NB * 16).astype(np.int64)
    s32 = float(np.float32(scale))
    shape = (NB, 16, Hkv, d)
    kc = torch.full(shape, 0xAB, dtype=torch.uint8, device="cuda")
    vc = torch.full(shape, 0xCD, dtype=torch.uint8, device="cuda")
    cache = PagedKVCache(kc, vc, "fp8_e4m3", s32, s32)
    kt = torch.from_numpy(kbits).view(torch.bfloat16).cuda()
    vt = torch.from_numpy(vbits).view(torch.bfloat16).cuda()
    st = torch.from_numpy(slots).cuda()
    if fused:
        paged_kv_zero_and_write(kt, vt, st, cache, np.zeros(0, np.int32))
    else:
        paged_kv_write(kt, vt, st, cache)
    assert pkv_check()[0] == PKV_OK
    ok = np.full(NB * 16 * Hkv * d, 0xAB, np.uint8)
    ov = np.full(NB * 16 * Hkv * d, 0xCD, np.uint8)
    assert oracle.load().kv_write(ok, ov, oracle.DTYPE_FP8_E4M3, 16, Hkv, d, s32, s32,
                                  kbits, vbits, slots) == 0
    for gpu, ref, bits in ((kc, ok, kbits), (vc, ov, vbits)):
        g = gpu.cpu().numpy().reshape(NB * 16, d)[slots]
        r = ref.reshape(NB * 16, d)[slots]
        b = bits.reshape(T, d)
        nan_in = (b & 0x7FFF) > 0x7F80
        assert np.array_equal(g[~nan_in], r[~nan_in])
        assert np.all((g[nan_in] & 0x7F) == 0x7F) and np.all((r[nan_in] & 0x7F) == 0x7F)


def test_write_skips_negative_and_reports_out_of_range():
    W = wl.tiny_mha()
    G = _pool(W)
    before = G.cache.key_cache.view(torch.uint8).clone()  # NaN canaries: compare bytes
    T = 4
    k = torch.zeros((T, W.num_kv_heads, W.head_dim), dtype=torch.bfloat16,
                    device="cuda")
    slots = torch.tensor([-1, -7, W.num_blocks * 16, W.num_blocks * 16 + 5],
                         dtype=torch.int64, device="cuda")
    paged_kv_write(k, k, slots, G.cache)
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail in (2, 3)
    assert torch.equal(G.cache.key_cache.view(torch.uint8), before)
    assert pkv_check()[0] == PKV_OK  # cleared


@pytest.mark.parametrize("on_host", [True, False])
def test_zero_blocks_only_named_blocks(on_host):
    W = wl.fp8_recycle(small=True)
    G = _pool(W)
    ids = W.fresh_blocks
    arg = ids if on_host else torch.from_numpy(ids).cuda()
    paged_kv_zero_blocks(G.cache, arg)
    assert pkv_check()[0] == PKV_OK
    kc, vc = W.init_key.copy(), W.init_value.copy()
    oracle.load().zero_blocks(kc, vc, W.block_bytes, ids)
    assert np.array_equal(G.cache.key_cache.cpu().numpy().reshape(-1), kc)
    assert np.array_equal(G.cache.value_cache.cpu().numpy().reshape(-1), vc)


def test_zero_blocks_many_host_ids_and_range_error():
    NB, Hkv, d = 9000, 1, 64
    shape = (NB, 16, Hkv, d)
    kc = torch.full(shape, 7, dtype=torch.bfloat16, device="cuda")
    vc = torch.full(shape, 9, dtype=torch.bfloat16, device="cuda")
    cache = PagedKVCache(kc, vc)
    rng = np.random.default_rng(3)
    ids = rng.permutation(NB)[:8500].astype(np.int32)  # three launches
    paged_kv_zero_blocks(cache, ids)
    assert pkv_check()[0] == PKV_OK
    zeroed = np.zeros(NB, bool)
    zeroed[ids] = True
    kz = (kc.view(NB, -1) == 0).all(dim=1).cpu().numpy()
    vz = (vc.view(NB, -1) == 0).all(dim=1).cpu().numpy()
    assert np.array_equal(kz, zeroed) and np.array_equal(vz, zeroed)
    untouched = (kc.view(NB, -1)[~torch.from_numpy(zeroed).cuda()] == 7).all()
    assert bool(untouched)
    paged_kv_zero_blocks(cache, np.array([3, NB, -2], np.int32))
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail in (1, 2)


def test_host_argument_errors():
    W = wl.tiny_mha()
    G = _pool(W)
    k = torch.zeros((2, W.num_kv_heads, W.head_dim), dtype=torch.bfloat16,
                    device="cuda")
    slots = torch.zeros(2, dtype=torch.int64, device="cuda")
    with pytest.raises(TypeError):
        paged_kv_write(k.float(), k, slots, G.cache)
    with pytest.raises(ValueError):
        paged_kv_write(k, k, slots[:1], G.cache)
    # the C ABI itself rejects an fp8 cache without a positive scale
    u8 = torch.zeros((4, 16, W.num_kv_heads, W.head_dim), dtype=torch.uint8,
                     device="cuda")
    no_scale = PagedKVCache(u8, u8.clone(), "fp8_e4m3", 0.0, 1.0)
    with pytest.raises(PagedKVError) as e:
        paged_kv_write(k, k, slots, no_scale)
    assert e.value.status == 1
