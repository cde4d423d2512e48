"""Pins of the CPU oracle against facts that do not come from the oracle.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises
AssertionError when the oracle disagrees with:
  - the E4M3 format definition (OCP OFP8 table, tests/golden/e4m3_values.txt)
    and torch's own float8_e4m3fn conversion (a library routine);
  - numpy scatter / slice assignment (library routines) for the write and
    zeroing steps;
  - closed forms of softmax attention (one key, equal keys, two keys,
    one-hot limit of very large logits);
  - torch's scaled_dot_product_attention in float64 on the contiguous case
    (a library routine), with GQA expanded by repeat_interleave;
  - invariants the pages state: the block table is only an indirection
    (identity, permuted and the pages' printed layouts give bit-identical
    results), a shared block is read, not copied, and stale bits outside a
    sequence never reach the result.

They are shared by ``test_oracle_pins.py`` (the real oracle) and
``test_oracle_mutants.py`` (deliberately broken copies, which must fail at
least one pin).
"""
from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np
import torch

from paged_kv_cache_48_gb300.workload import bf16_bits, bf16_values

GOLDEN = Path(__file__).resolve().parent / "golden"
BF16, FP8 = 0, 1
BS = 16


# ---------------------------------------------------------------------------
# helpers that build tiny paged inputs by hand (no oracle arithmetic)
# ---------------------------------------------------------------------------

def _rand_bf16(rng, shape, scale=1.0):
    return bf16_bits(rng.standard_normal(shape).astype(np.float32) * scale)


def _paged_from_contiguous(K, V, tables, num_blocks, fill=0xFF):
    """Place contiguous per-sequence token rows (uint16 [B][L_b, Hkv, d])
    into a bf16 pool at the blocks named by the tables."""
    Hkv, d = K[0].shape[1:]
    kc = np.full((num_blocks, BS, Hkv, d), 0xFFFF if fill == 0xFF else 0,
                 dtype=np.uint16)
    vc = kc.copy()
    for b, (kb, vb) in enumerate(zip(K, V)):
        for t in range(kb.shape[0]):
            blk = tables[b][t // BS]
            kc[blk, t % BS] = kb[t]
            vc[blk, t % BS] = vb[t]
    return kc.view(np.uint8).reshape(-1), vc.view(np.uint8).reshape(-1)


def _tables_array(tables, max_blocks):
    out = np.full((len(tables), max_blocks), -1, dtype=np.int32)
    for b, t in enumerate(tables):
        out[b, :len(t)] = t
    return out


def _run(oracle, q, kc, vc, tables, lens, Hkv, d, scale, dtype=BF16,
         k_scale=1.0, v_scale=1.0):
    out, err = oracle.attention_decode(q, kc, vc, dtype, k_scale, v_scale,
                                       BS, Hkv, d, tables, lens, scale)
    assert err == 0, f"oracle reported {err} range errors"
    return out


def _sdpa_reference(q_bits, K, V, scale):
    """torch SDPA in float64 on contiguous K/V (GQA by repeat_interleave)."""
    B, Hq, d = q_bits.shape
    outs = []
    for b in range(B):
        qb = torch.from_numpy(bf16_values(q_bits[b]).astype(np.float64))
        kb = torch.from_numpy(bf16_values(K[b]).astype(np.float64))
        vb = torch.from_numpy(bf16_values(V[b]).astype(np.float64))
        g = Hq // kb.shape[1]
        kb = kb.permute(1, 0, 2).repeat_interleave(g, dim=0)  # [Hq, L, d]
        vb = vb.permute(1, 0, 2).repeat_interleave(g, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qb[:, None, :], kb, vb, scale=scale)
        outs.append(o[:, 0, :].numpy())
    return np.stack(outs)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def pin_e4m3_decode_golden(oracle):
    """Values printed in the format definition's table."""
    for line in (GOLDEN / "e4m3_values.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        code, val = line.split()
        got = oracle.e4m3_to_double(int(code, 16))
        if val == "nan":
            assert math.isnan(got), (code, got)
        else:
            want = float(val)
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def pin_e4m3_decode_all_codes_vs_torch(oracle):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_e4m3_encode_round_trip_and_ties(oracle):
    for c in range(0x7F):
        for sgn in (0, 0x80):
            v = oracle.e4m3_to_double(c | sgn)
            assert oracle.e4m3_from_float(v) == (c | sgn), hex(c | sgn)
    # midpoints between neighbours go to the even code; one ulp either
    # side goes to the nearer code
    for c in range(0x7E):
        lo = oracle.e4m3_to_double(c)
        hi = oracle.e4m3_to_double(c + 1)
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_from_float(mid) == even, hex(c)
        below = np.nextafter(mid, np.float32(-1))
        above = np.nextafter(mid, np.float32(1e9))
        assert oracle.e4m3_from_float(below) == c, hex(c)
        assert oracle.e4m3_from_float(above) == c + 1, hex(c)


def pin_e4m3_encode_saturation_and_nan(oracle):
    assert oracle.e4m3_from_float(448.0) == 0x7E
    assert oracle.e4m3_from_float(463.9) == 0x7E
    assert oracle.e4m3_from_float(464.0) == 0x7E
    assert oracle.e4m3_from_float(1e30) == 0x7E
    assert oracle.e4m3_from_float(float("inf")) == 0x7E
    assert oracle.e4m3_from_float(float("-inf")) == 0xFE
    assert oracle.e4m3_from_float(-1000.0) == 0xFE
    assert oracle.e4m3_from_float(float("nan")) & 0x7F == 0x7F
    assert oracle.e4m3_from_float(0.0) == 0x00
    assert oracle.e4m3_from_float(-0.0) == 0x80
    # below half the smallest subnormal: rounds to a signed zero
    assert oracle.e4m3_from_float(2.0 ** -11) == 0x00
    assert oracle.e4m3_from_float(-(2.0 ** -11)) == 0x80


def pin_e4m3_encode_vs_torch(oracle):
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 40,
        rng.uniform(-447.9, 447.9, 2000).astype(np.float32),
        (rng.standard_normal(2000) * 0.01).astype(np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, ref), int(np.count_nonzero(got != ref))


def pin_bf16_decode(oracle):
    bits = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F,
                     0xFF7F, 0x7F80, 0xFF80], dtype=np.uint16)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for b, r in zip(bits, ref):
        got = oracle.bf16_to_double(int(b))
        assert got == r and math.copysign(1, got) == math.copysign(1, r), (hex(b), got, r)


def pin_quantize_is_fp32_quotient(oracle):
    rng = np.random.default_rng(12)
    x = _rand_bf16(rng, (3000,))
    for scale in (np.float32(0.0107), np.float32(1.0), np.float32(0.37)):
        q = (bf16_values(x) / scale).astype(np.float32)
        ok = np.abs(q) < 448
        ref = torch.from_numpy(q[ok]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = np.array([oracle.quantize_e4m3(int(b), float(scale)) for b in x[ok]],
                       np.uint8)
        assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# write and zeroing
# ---------------------------------------------------------------------------

def pin_kv_write_is_scatter(oracle):
    rng = np.random.default_rng(13)
    NB, Hkv, d, T = 10, 2, 8, 40
    k = _rand_bf16(rng, (T, Hkv, d))
    v = _rand_bf16(rng, (T, Hkv, d))
    slots = rng.permutation(NB * BS)[:T].astype(np.int64)
    slots[3] = -1
    slots[7] = -5
    kc = np.full((NB, BS, Hkv, d), 0x1234, np.uint16)
    vc = np.full((NB, BS, Hkv, d), 0x4321, np.uint16)
    ref_k, ref_v = kc.copy(), vc.copy()
    keep = slots >= 0
    ref_k[slots[keep] // BS, slots[keep] % BS] = k[keep]
    ref_v[slots[keep] // BS, slots[keep] % BS] = v[keep]
    kb, vb = kc.view(np.uint8).reshape(-1), vc.view(np.uint8).reshape(-1)
    err = oracle.kv_write(kb, vb, BF16, BS, Hkv, d, 1.0, 1.0, k, v, slots)
    assert err == 0
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)
    # out-of-range slots are counted and write nothing
    bad = np.array([NB * BS, NB * BS + 17], np.int64)
    before = kc.copy()
    err = oracle.kv_write(kb, vb, BF16, BS, Hkv, d, 1.0, 1.0, k[:2], v[:2], bad)
    assert err == 2 and np.array_equal(kc, before)


def pin_kv_write_fp8_is_quantised_scatter(oracle):
    rng = np.random.default_rng(14)
    NB, Hkv, d, T = 6, 2, 16, 30
    k = _rand_bf16(rng, (T, Hkv, d))
    v = _rand_bf16(rng, (T, Hkv, d), scale=3.0)
    ks = np.float32(np.abs(bf16_values(k)).max() / 448)
    vs = np.float32(np.abs(bf16_values(v)).max() / 448)
    slots = rng.permutation(NB * BS)[:T].astype(np.int64)
    kc = np.full((NB, BS, Hkv, d), 0xFF, np.uint8)
    vc = np.full((NB, BS, Hkv, d), 0xFF, np.uint8)
    ref_k, ref_v = kc.copy(), vc.copy()
    qk = torch.from_numpy((bf16_values(k) / ks).astype(np.float32))
    qv = torch.from_numpy((bf16_values(v) / vs).astype(np.float32))
    ref_k[slots // BS, slots % BS] = qk.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref_v[slots // BS, slots % BS] = qv.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    err = oracle.kv_write(kc.reshape(-1), vc.reshape(-1), FP8, BS, Hkv, d,
                          float(ks), float(vs), k, v, slots)
    assert err == 0
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)


def pin_zero_blocks_is_slice_assignment(oracle):
    rng = np.random.default_rng(15)
    NB, block_bytes = 12, 256
    kc = rng.integers(0, 256, NB * block_bytes, dtype=np.uint8)
    vc = rng.integers(0, 256, NB * block_bytes, dtype=np.uint8)
    ref_k, ref_v = kc.copy(), vc.copy()
    ids = np.array([7, 2, 9], np.int32)
    for i in ids:
        ref_k[i * block_bytes:(i + 1) * block_bytes] = 0
        ref_v[i * block_bytes:(i + 1) * block_bytes] = 0
    assert oracle.zero_blocks(kc, vc, block_bytes, ids) == 0
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)
    assert oracle.zero_blocks(kc, vc, block_bytes, np.array([-1, NB], np.int32)) == 2
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)


def pin_copy_blocks_is_ordered_block_assignment(oracle):
    rng = np.random.default_rng(28)
    NB, bb = 10, 64
    kc = rng.integers(0, 256, NB * bb, dtype=np.uint8)
    vc = rng.integers(0, 256, NB * bb, dtype=np.uint8)
    src = np.array([3, 7, 3, 0], np.int32)
    dst = np.array([5, 1, 9, 7], np.int32)  # block 7 is read, then written
    rk = kc.reshape(NB, bb).copy()
    rv = vc.reshape(NB, bb).copy()
    for a, b in zip(src, dst):  # numpy row assignment, in order
        rk[b] = rk[a]
        rv[b] = rv[a]
    assert oracle.copy_blocks(kc, vc, bb, src, dst) == 0
    assert np.array_equal(kc.reshape(NB, bb), rk)
    assert np.array_equal(vc.reshape(NB, bb), rv)
    assert oracle.copy_blocks(kc, vc, bb, np.array([NB], np.int32),
                              np.array([0], np.int32)) == 1
    assert np.array_equal(kc.reshape(NB, bb), rk)


def pin_swap_round_trip_is_gather_then_scatter(oracle):
    rng = np.random.default_rng(29)
    NB, bb = 12, 32
    kc = rng.integers(0, 256, NB * bb, dtype=np.uint8)
    vc = rng.integers(0, 256, NB * bb, dtype=np.uint8)
    ids = np.array([4, 11, 0, 6], np.int32)
    ok, ov, err = oracle.swap_out(kc, vc, bb, ids)
    assert err == 0
    assert np.array_equal(ok.reshape(-1, bb), kc.reshape(NB, bb)[ids])
    assert np.array_equal(ov.reshape(-1, bb), vc.reshape(NB, bb)[ids])
    # swap the same data back in elsewhere: equals copying the blocks
    k2, v2 = kc.copy(), vc.copy()
    dst = np.array([1, 2, 3, 5], np.int32)
    assert oracle.swap_in(k2, v2, bb, dst, ok, ov) == 0
    k3, v3 = kc.copy(), vc.copy()
    assert oracle.copy_blocks(k3, v3, bb, ids, dst) == 0
    assert np.array_equal(k2, k3) and np.array_equal(v2, v3)
    assert oracle.swap_out(kc, vc, bb, np.array([-1], np.int32))[2] == 1


def _state_table(rng, R=12, MB=8, ML=128):
    sbt = rng.permutation(R * MB + 10)[:R * MB].astype(np.int32).reshape(R, MB)
    snc = rng.integers(0, 100, R).astype(np.int32)
    tok = rng.integers(0, 50000, (R, ML)).astype(np.int32)
    return sbt, snc, tok


def pin_prepare_inputs_is_gather_and_cumsum(oracle):
    rng = np.random.default_rng(30)
    sbt, snc, tok = _state_table(rng)
    idx = np.array([7, 2, 11, 0, 5], np.int32)
    ns = np.array([1, 17, 1, 0, 9], np.int32)
    T = int(ns.sum())
    out, err = oracle.prepare_inputs(idx, ns, sbt, snc, tok, T)
    assert err == 0
    qsl = np.concatenate([[0], np.cumsum(ns)])
    assert np.array_equal(out["query_start_loc"], qsl)
    assert np.array_equal(out["block_tables"], sbt[idx])
    assert np.array_equal(out["seq_lens"], snc[idx] + ns)
    rows = np.repeat(idx, ns)
    pos = np.concatenate([snc[r] + np.arange(n) for r, n in zip(idx, ns)])
    assert np.array_equal(out["positions"], pos)
    assert np.array_equal(out["input_ids"], tok[rows, pos])
    assert np.array_equal(out["slot_mapping"],
                          sbt[rows, pos // 16].astype(np.int64) * 16 + pos % 16)
    # every new token's slot lies inside its request's last needed block
    last = qsl[1:] - 1
    for b in range(idx.size):
        if ns[b]:
            L = out["seq_lens"][b]
            assert out["slot_mapping"][last[b]] == sbt[idx[b], (L - 1) // 16] * 16 + (L - 1) % 16


def pin_prepare_inputs_range_errors(oracle):
    rng = np.random.default_rng(31)
    sbt, snc, tok = _state_table(rng, R=4, MB=2, ML=40)
    snc[:] = [0, 30, 5, 31]
    idx = np.array([0, 9, 1, 3], np.int32)       # row 9 does not exist
    ns = np.array([2, 3, 4, 1], np.int32)          # row 1: positions 30..33 > 32
    out, err = oracle.prepare_inputs(idx, ns, sbt, snc, tok, int(ns.sum()))
    assert err == 1 + 2                            # bad row, positions 32 and 33
    sl = out["slot_mapping"]
    assert list(sl[2:5]) == [-1, -1, -1]           # the bad row's tokens
    assert sl[5] >= 0 and sl[6] >= 0 and sl[7] == -1 and sl[8] == -1
    assert sl[9] == sbt[3, 1] * 16 + 15


def pin_prepare_inputs_negative_and_overflowing_counts(oracle):
    """A negative count schedules nothing; an entry whose tokens do not all
    fit below total_tokens writes nothing, while query_start_loc stays the
    exclusive prefix sum of the clamped counts.  Expected values written
    out by hand for this batch (total_tokens 8, counts 2, -3, 4, 5, 1):
      entry 0 (row 2, c 10): tokens 0, 1 at positions 10, 11;
      entry 1 (row 0, c 3):  count -3 -> 0 tokens, seq_len 3, an error;
      entry 2 (row 1, c 0):  tokens 2..5 at positions 0..3;
      entry 3 (row 3):       starts at 6, needs 6..10 > 7: nothing, an error;
      entry 4 (row 1):       starts at 11 > 7: nothing, an error."""
    sbt = np.array([[40, 41], [50, 51], [60, 61], [70, 71]], np.int32)
    snc = np.array([3, 0, 10, 5], np.int32)
    tok = np.arange(4 * 40, dtype=np.int32).reshape(4, 40) + 1000
    idx = np.array([2, 0, 1, 3, 1], np.int32)
    ns = np.array([2, -3, 4, 5, 1], np.int32)
    out, err = oracle.prepare_inputs(idx, ns, sbt, snc, tok, 8)
    assert err == 3
    assert list(out["query_start_loc"]) == [0, 2, 2, 6, 11, 12]
    assert list(out["seq_lens"][:3]) == [12, 3, 4]
    assert np.array_equal(out["block_tables"][:3], sbt[[2, 0, 1]])
    assert list(out["positions"][:6]) == [10, 11, 0, 1, 2, 3]
    assert list(out["input_ids"][:6]) == [1090, 1091, 1040, 1041, 1042, 1043]
    assert list(out["slot_mapping"][:6]) == [60 * 16 + 10, 60 * 16 + 11,
                                             50 * 16, 50 * 16 + 1, 50 * 16 + 2, 50 * 16 + 3]
    # entries 3 and 4 wrote nothing (the wrapper's fill value -7 remains),
    # not even the two slots of entry 3 that would have fitted
    assert list(out["seq_lens"][3:]) == [-7, -7]
    assert (out["block_tables"][3:] == -7).all()
    for k in ("positions", "input_ids", "slot_mapping"):
        assert list(out[k][6:]) == [-7, -7], k


# ---------------------------------------------------------------------------
# attention: closed forms
# ---------------------------------------------------------------------------

def pin_single_key_returns_its_value(oracle):
    rng = np.random.default_rng(16)
    Hkv, Hq, d = 2, 4, 16
    K = [_rand_bf16(rng, (1, Hkv, d))]
    V = [_rand_bf16(rng, (1, Hkv, d))]
    q = _rand_bf16(rng, (1, Hq, d))
    kc, vc = _paged_from_contiguous(K, V, [[3]], 5)
    out = _run(oracle, q, kc, vc, _tables_array([[3]], 2), np.array([1], np.int32),
               Hkv, d, 0.25)
    for h in range(Hq):
        assert np.array_equal(out[0, h], bf16_values(V[0][0, h // 2]).astype(np.float64))


def pin_single_key_fp8_returns_scaled_value(oracle):
    rng = np.random.default_rng(17)
    Hkv, Hq, d, NB = 1, 2, 16, 3
    kc = rng.integers(0, 0x7E, NB * BS * Hkv * d, dtype=np.uint8)
    vc = rng.integers(0, 0x7E, NB * BS * Hkv * d, dtype=np.uint8)
    vs = 0.03125
    q = _rand_bf16(rng, (1, Hq, d))
    out, err = oracle.attention_decode(q, kc, vc, FP8, 0.5, vs, BS, Hkv, d,
                                       _tables_array([[2]], 1),
                                       np.array([1], np.int32), 0.3)
    assert err == 0
    row = vc.reshape(NB, BS, Hkv, d)[2, 0, 0]
    ref = torch.from_numpy(row.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy() * vs
    for h in range(Hq):
        assert np.array_equal(out[0, h], ref)


def pin_equal_keys_give_mean_value(oracle):
    rng = np.random.default_rng(18)
    Hkv, Hq, d, L = 1, 2, 8, 37
    k_row = _rand_bf16(rng, (1, Hkv, d))
    K = [np.repeat(k_row, L, axis=0)]
    V = [_rand_bf16(rng, (L, Hkv, d))]
    q = _rand_bf16(rng, (1, Hq, d))
    tables = [[4, 0, 2]]
    kc, vc = _paged_from_contiguous(K, V, tables, 6)
    out = _run(oracle, q, kc, vc, _tables_array(tables, 3), np.array([L], np.int32),
               Hkv, d, 1.0 / math.sqrt(d))
    mean = bf16_values(V[0][:, 0]).astype(np.float64).mean(axis=0)
    for h in range(Hq):
        assert np.allclose(out[0, h], mean, rtol=0, atol=1e-12)


def pin_two_keys_sigmoid(oracle):
    rng = np.random.default_rng(19)
    Hkv, Hq, d = 1, 1, 8
    K = [_rand_bf16(rng, (2, Hkv, d))]
    V = [_rand_bf16(rng, (2, Hkv, d))]
    q = _rand_bf16(rng, (1, Hq, d))
    scale = 0.7
    kc, vc = _paged_from_contiguous(K, V, [[1]], 2)
    out = _run(oracle, q, kc, vc, _tables_array([[1]], 1), np.array([2], np.int32),
               Hkv, d, scale)
    qv = bf16_values(q[0, 0]).astype(np.float64)
    k = bf16_values(K[0][:, 0]).astype(np.float64)
    v = bf16_values(V[0][:, 0]).astype(np.float64)
    s1, s2 = scale * float(qv @ k[0]), scale * float(qv @ k[1])
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))
    ref = w1 * v[0] + (1.0 - w1) * v[1]
    assert np.allclose(out[0, 0], ref, rtol=1e-13, atol=1e-13)


def pin_huge_logits_pick_argmax(oracle):
    """scale so large that softmax is one-hot: the output is the V row of
    the largest score, and stays finite (no overflow)."""
    rng = np.random.default_rng(20)
    Hkv, Hq, d, L = 1, 1, 8, 20
    K = [_rand_bf16(rng, (L, Hkv, d))]
    V = [_rand_bf16(rng, (L, Hkv, d))]
    q = _rand_bf16(rng, (1, Hq, d))
    tables = [[0, 1]]
    kc, vc = _paged_from_contiguous(K, V, tables, 2)
    out = _run(oracle, q, kc, vc, _tables_array(tables, 2), np.array([L], np.int32),
               Hkv, d, 1.0e4)
    s = bf16_values(K[0][:, 0]).astype(np.float64) @ bf16_values(q[0, 0]).astype(np.float64)
    top = int(np.argmax(s))
    assert np.sort(s)[-1] - np.sort(s)[-2] > 1e-2
    assert np.all(np.isfinite(out))
    assert np.allclose(out[0, 0], bf16_values(V[0][top, 0]), rtol=0, atol=1e-12)


def pin_empty_sequence_gives_zeros(oracle):
    rng = np.random.default_rng(21)
    q = _rand_bf16(rng, (2, 2, 8))
    kc = np.full(2 * BS * 8 * 2, 0xFF, np.uint8)
    vc = kc.copy()
    out = _run(oracle, q, kc, vc, _tables_array([[], [0]], 1),
               np.array([0, 1], np.int32), 1, 8, 0.5)
    assert np.array_equal(out[0], np.zeros((2, 8)))
    assert np.all(np.isnan(out[1]))  # the one key is the 0xFF canary = NaN


# ---------------------------------------------------------------------------
# attention: library special case and invariants
# ---------------------------------------------------------------------------

def _random_case(seed, B=3, Hq=4, Hkv=2, d=16, lens=(5, 16, 41)):
    rng = np.random.default_rng(seed)
    K = [_rand_bf16(rng, (L, Hkv, d)) for L in lens]
    V = [_rand_bf16(rng, (L, Hkv, d)) for L in lens]
    q = _rand_bf16(rng, (B, Hq, d))
    return rng, K, V, q


def pin_matches_sdpa_on_contiguous_layout(oracle):
    lens = (5, 16, 41, 1)
    rng, K, V, q = _random_case(22, B=4, Hq=6, Hkv=2, d=16, lens=lens)
    nb = [(L + BS - 1) // BS for L in lens]
    tables, nxt = [], 0
    for n in nb:
        tables.append(list(range(nxt, nxt + n)))
        nxt += n
    kc, vc = _paged_from_contiguous(K, V, tables, nxt)
    scale = 1.0 / math.sqrt(16)
    out = _run(oracle, q, kc, vc, _tables_array(tables, max(nb)),
               np.array(lens, np.int32), 2, 16, scale)
    ref = _sdpa_reference(q, K, V, scale)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def pin_block_table_is_only_indirection(oracle):
    """Identity, seeded-permuted and the pages' printed layouts give
    bit-identical results; NaN canaries fill every slot outside the
    sequences (including the unused tail of the last block)."""
    layouts = json.loads((GOLDEN / "page_table_layouts.json").read_text())["layouts"]
    rng = np.random.default_rng(23)
    Hkv, Hq, d = 2, 4, 16
    for lay in layouts:
        seqs = lay["sequences"]
        lens = [len(s) * BS - (3 if i == 0 else 9) for i, s in enumerate(seqs)]
        K = [_rand_bf16(rng, (L, Hkv, d)) for L in lens]
        V = [_rand_bf16(rng, (L, Hkv, d)) for L in lens]
        q = _rand_bf16(rng, (len(seqs), Hq, d))
        mb = max(len(s) for s in seqs)
        ident, nxt = [], 0
        for s in seqs:
            ident.append(list(range(nxt, nxt + len(s))))
            nxt += len(s)
        perm = rng.permutation(lay["num_blocks"])
        shuffled = [[int(perm[i]) for i in t] for t in ident]
        results = []
        for tables in (ident, seqs, shuffled):
            kc, vc = _paged_from_contiguous(K, V, tables, lay["num_blocks"])
            results.append(_run(oracle, q, kc, vc, _tables_array(tables, mb + 2),
                                np.array(lens, np.int32), Hkv, d, 0.25))
        assert np.all(np.isfinite(results[0]))
        assert np.array_equal(results[0], results[1])
        assert np.array_equal(results[0], results[2])
        # the pages' free blocks are never read: poison them differently
        kc, vc = _paged_from_contiguous(K, V, seqs, lay["num_blocks"])
        kk = kc.view(np.uint16).reshape(lay["num_blocks"], BS, Hkv, d)
        for f in lay["free_blocks"]:
            kk[f] = 0x7F80  # +Inf
        again = _run(oracle, q, kc, vc, _tables_array(seqs, mb),
                     np.array(lens, np.int32), Hkv, d, 0.25)
        assert np.array_equal(again, results[0])


def pin_gqa_equals_replicated_mha(oracle):
    lens = (7, 33)
    rng, K, V, q = _random_case(24, B=2, Hq=6, Hkv=2, d=16, lens=lens)
    tables = [[0], [3, 1, 4]]
    kc, vc = _paged_from_contiguous(K, V, tables, 5)
    gqa = _run(oracle, q, kc, vc, _tables_array(tables, 3), np.array(lens, np.int32),
               2, 16, 0.25)
    Kr = [np.repeat(k, 3, axis=1) for k in K]
    Vr = [np.repeat(v, 3, axis=1) for v in V]
    kc6, vc6 = _paged_from_contiguous(Kr, Vr, tables, 5)
    mha = _run(oracle, q, kc6, vc6, _tables_array(tables, 3), np.array(lens, np.int32),
               6, 16, 0.25)
    assert np.array_equal(gqa, mha)


def pin_shared_prefix_read_not_copied(oracle):
    """Sequences whose tables point at the same prefix blocks (refcount > 1)
    read those blocks in place: the caches are unchanged by attention, and
    two sequences with the same prefix and the same private suffix data
    give identical outputs."""
    rng = np.random.default_rng(25)
    Hkv, Hq, d, NB = 2, 4, 16, 10
    prefix = [6, 2]            # shared blocks
    suffix_a, suffix_b = [9], [0]
    L = 2 * BS + 5
    Kp = _rand_bf16(rng, (2 * BS, Hkv, d))
    Vp = _rand_bf16(rng, (2 * BS, Hkv, d))
    Ks = _rand_bf16(rng, (5, Hkv, d))
    Vs = _rand_bf16(rng, (5, Hkv, d))
    K = [np.concatenate([Kp, Ks])] * 2
    V = [np.concatenate([Vp, Vs])] * 2
    tables = [prefix + suffix_a, prefix + suffix_b]
    kc, vc = _paged_from_contiguous(K, V, tables, NB)
    before = (kc.copy(), vc.copy())
    q1 = _rand_bf16(rng, (1, Hq, d))
    q = np.concatenate([q1, q1])
    out = _run(oracle, q, kc, vc, _tables_array(tables, 3), np.array([L, L], np.int32),
               Hkv, d, 0.25)
    assert np.array_equal(out[0], out[1])
    assert np.array_equal(kc, before[0]) and np.array_equal(vc, before[1])
    ref = _sdpa_reference(q[:1], K[:1], V[:1], 0.25)
    assert np.allclose(out[:1], ref, rtol=1e-12, atol=1e-12)


def pin_fp8_attention_matches_dequantised_sdpa(oracle):
    rng = np.random.default_rng(26)
    Hkv, Hq, d, NB = 2, 4, 16, 4
    kc = rng.integers(0, 0x7E, NB * BS * Hkv * d, dtype=np.uint8)
    vc = rng.integers(0, 0x7E, NB * BS * Hkv * d, dtype=np.uint8)
    kc |= (rng.integers(0, 2, kc.size, dtype=np.uint8) << 7)
    vc |= (rng.integers(0, 2, vc.size, dtype=np.uint8) << 7)
    ks, vs = 0.01, 0.02
    q = _rand_bf16(rng, (1, Hq, d))
    tables, L = [[3, 1]], 29
    out, err = oracle.attention_decode(q, kc, vc, FP8, ks, vs, BS, Hkv, d,
                                       _tables_array(tables, 2),
                                       np.array([L], np.int32), 0.25)
    assert err == 0
    deq = lambda c: torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    k4 = deq(kc).reshape(NB, BS, Hkv, d) * ks
    v4 = deq(vc).reshape(NB, BS, Hkv, d) * vs
    Kc = np.concatenate([k4[3], k4[1]])[:L]
    Vc = np.concatenate([v4[3], v4[1]])[:L]
    qq = torch.from_numpy(bf16_values(q[0]).astype(np.float64))
    kk = torch.from_numpy(Kc).permute(1, 0, 2).repeat_interleave(2, dim=0)
    vv = torch.from_numpy(Vc).permute(1, 0, 2).repeat_interleave(2, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qq[:, None, :], kk, vv, scale=0.25)[:, 0].numpy()
    assert np.allclose(out[0], ref, rtol=1e-12, atol=1e-12)


def pin_range_errors_reported(oracle):
    rng = np.random.default_rng(27)
    q = _rand_bf16(rng, (2, 2, 8))
    kc = np.zeros(3 * BS * 8 * 2, np.uint8)
    out, err = oracle.attention_decode(q, kc, kc.copy(), BF16, 1, 1, BS, 1, 8,
                                       np.array([[5], [0]], np.int32),
                                       np.array([3, 2 * BS], np.int32), 0.5)
    assert err == 4  # 2 sequences x 2 heads, each row counted
    assert np.array_equal(out, np.zeros_like(out))


# ---------------------------------------------------------------------------
# prefill / chunked prefill (causal within each sequence's chunk)
# ---------------------------------------------------------------------------

def _prefill_case(seed, lens, nq, Hq=6, Hkv=2, d=16, permute=True):
    """Sequences of lens[b] tokens whose last nq[b] are this step's query
    tokens; blocks placed at seeded random physical ids."""
    rng = np.random.default_rng(seed)
    K = [_rand_bf16(rng, (L, Hkv, d)) for L in lens]
    V = [_rand_bf16(rng, (L, Hkv, d)) for L in lens]
    nb = [(L + BS - 1) // BS for L in lens]
    ids = rng.permutation(sum(nb) + 5) if permute else np.arange(sum(nb) + 5)
    tables, nxt = [], 0
    for n in nb:
        tables.append([int(x) for x in ids[nxt:nxt + n]])
        nxt += n
    kc, vc = _paged_from_contiguous(K, V, tables, sum(nb) + 5)
    qsl = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = _rand_bf16(rng, (int(qsl[-1]), Hq, d))
    return K, V, q, kc, vc, _tables_array(tables, max(nb)), qsl


def _causal_sdpa_reference(q_bits, K, V, lens, qsl, scale):
    """torch SDPA in float64 per sequence with an explicit boolean mask:
    query i of sequence b (position lens[b] - n_b + i) may see key t iff
    t <= that position."""
    T, Hq, d = q_bits.shape
    out = np.zeros((T, Hq, d))
    for b, L in enumerate(lens):
        a, e = int(qsl[b]), int(qsl[b + 1])
        n = e - a
        if n == 0:
            continue
        qb = torch.from_numpy(bf16_values(q_bits[a:e]).astype(np.float64))
        kb = torch.from_numpy(bf16_values(K[b]).astype(np.float64))
        vb = torch.from_numpy(bf16_values(V[b]).astype(np.float64))
        g = Hq // kb.shape[1]
        kb = kb.permute(1, 0, 2).repeat_interleave(g, dim=0)  # [Hq, L, d]
        vb = vb.permute(1, 0, 2).repeat_interleave(g, dim=0)
        pos = torch.arange(L - n, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos                 # [n, L]
        o = torch.nn.functional.scaled_dot_product_attention(
            qb.permute(1, 0, 2), kb, vb, attn_mask=mask, scale=scale)
        out[a:e] = o.permute(1, 0, 2).numpy()
    return out


def _run_prefill(oracle, q, kc, vc, tables, lens, qsl, Hkv, d, scale, rows=None):
    out, err = oracle.attention_prefill(q, kc, vc, BF16, 1.0, 1.0, BS, Hkv, d,
                                        tables, np.array(lens, np.int32), qsl,
                                        scale, rows=rows)
    return out, err


def pin_prefill_matches_causal_sdpa(oracle):
    """Whole prompts, chunks after a history, a one-token (decode) entry and
    an empty entry, against torch SDPA with an explicit causal mask."""
    lens, nq = (5, 16, 41, 33, 7), (5, 3, 20, 1, 0)
    K, V, q, kc, vc, tables, qsl = _prefill_case(40, lens, nq)
    scale = 1.0 / math.sqrt(16)
    out, err = _run_prefill(oracle, q, kc, vc, tables, lens, qsl, 2, 16, scale)
    assert err == 0
    ref = _causal_sdpa_reference(q, K, V, lens, qsl, scale)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def pin_prefill_first_prompt_token_returns_its_value(oracle):
    """A prompt's first token attends to itself alone: its output is exactly
    its own V row (per kv head of its group)."""
    lens, nq = (9, 20), (9, 20)
    K, V, q, kc, vc, tables, qsl = _prefill_case(41, lens, nq, Hq=4, Hkv=2)
    out, err = _run_prefill(oracle, q, kc, vc, tables, lens, qsl, 2, 16, 0.3)
    assert err == 0
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out[qsl[b], h], bf16_values(V[b][0, h // 2]))


def pin_prefill_ignores_keys_after_each_position(oracle):
    """Changing the K/V of the chunk's last token changes the last query row
    only; every earlier row of the chunk is bit-identical."""
    lens, nq = (30,), (12,)
    K, V, q, kc, vc, tables, qsl = _prefill_case(42, lens, nq, permute=False)
    out1, _ = _run_prefill(oracle, q, kc, vc, tables, lens, qsl, 2, 16, 0.25)
    K2 = [K[0].copy()]
    V2 = [V[0].copy()]
    rng = np.random.default_rng(43)
    K2[0][-1] = _rand_bf16(rng, K2[0][-1].shape)
    V2[0][-1] = _rand_bf16(rng, V2[0][-1].shape)
    kc2, vc2 = _paged_from_contiguous(K2, V2, [list(tables[0][tables[0] >= 0])],
                                      kc.size // (BS * 2 * 16 * 2))
    out2, _ = _run_prefill(oracle, q, kc2, vc2, tables, lens, qsl, 2, 16, 0.25)
    assert np.array_equal(out1[:-1], out2[:-1])
    assert not np.allclose(out1[-1], out2[-1])


def pin_prefill_rows_subset_and_range_errors(oracle):
    """A selected (token, head) subset equals the same rows of the full
    result; a sequence whose chunk is longer than its length is an error
    and its rows stay zero."""
    lens, nq = (21, 18), (6, 4)
    K, V, q, kc, vc, tables, qsl = _prefill_case(44, lens, nq)
    full, err = _run_prefill(oracle, q, kc, vc, tables, lens, qsl, 2, 16, 0.2)
    assert err == 0
    rows = np.array([[0, 5], [3, 0], [9, 2], [7, 4]], np.int32)
    part, err = _run_prefill(oracle, q, kc, vc, tables, lens, qsl, 2, 16, 0.2,
                             rows=rows)
    assert err == 0
    for t, h in rows:
        assert np.array_equal(part[t, h], full[t, h])
    bad, err = _run_prefill(oracle, q, kc, vc, tables, (21, 3), qsl, 2, 16, 0.2)
    assert err == 4 * 6
    assert np.array_equal(bad[6:], np.zeros_like(bad[6:]))
    assert np.array_equal(bad[:6], full[:6])


ALL_PINS = [obj for name, obj in sorted(globals().items())
            if name.startswith("pin_") and callable(obj)]
