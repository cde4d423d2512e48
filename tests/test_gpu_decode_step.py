"""paged_attention_decode_step (the new token's write inside the decode
kernel) against the two-call step and the fp64 oracle.

A decode step writes each sequence's new token (position seq_lens[b] - 1)
into the block its table names, zeroing that block first when the token
opens it (vLLM v0.17.1 notes, "修复方案"), then attends.  The one-call
step must leave the same cache bytes as paged_kv_zero_and_write with the
opened blocks listed as fresh, and give bit for bit the output of
paged_attention_decode on that cache; both are checked against the
oracle's cache (byte-exact) and attention (|gpu - ref| <= 1e-2 + 1e-2
|ref|, 3e-2 for an E4M3 cache).  Cases span bf16 and E4M3 caches, head_dim
64 and 128, group sizes 1, 4, 5, 8 and 16, CTA-shared and warp-owned
partitions, tokens that open a block and tokens that do not, an empty
sequence, a table entry outside the pool and a length above the host
bound; tails of several new tokens per sequence (the fp8 recycling step,
tails that start mid-block or at a block start and cross partitions), and
a tail longer than its sequence.
"""
import numpy as np
import pytest
import torch

import harness
from paged_kv_cache_48_gb300 import (paged_attention_decode,
                                     paged_attention_decode_step,
                                     paged_kv_zero_and_write, pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu
PKV_OK, PKV_ERR_RANGE = 0, 5


def _new_tokens(W, G):
    """k_new / v_new [B, Hkv, d]: each sequence's new-token row of the
    step's writes (found by its slot)."""
    B = W.batch
    slots = W.step_slots.tolist()
    k = torch.zeros((B, W.num_kv_heads, W.head_dim), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    for b in range(B):
        L = int(W.seq_lens[b])
        if L == 0:
            continue
        s = int(W.block_tables[b, (L - 1) // 16]) * 16 + (L - 1) % 16
        i = slots.index(s)
        k[b] = G.step_k[i]
        v[b] = G.step_v[i]
    return k, v


def _caches(G):
    return (G.cache.key_cache.view(torch.uint8).cpu().numpy().reshape(-1),
            G.cache.value_cache.view(torch.uint8).cpu().numpy().reshape(-1))


def _step(W, G, pt, max_seq_len=None, tables=None):
    k, v = _new_tokens(W, G)
    return paged_attention_decode_step(
        G.q, k, v, G.cache, G.tables if tables is None else tables, G.seq_lens, W.scale,
        max_seq_len=W.max_seq_len if max_seq_len is None else max_seq_len,
        partition_tokens=pt)


def _new_token_only(W):
    """Every step write is a sequence's new token (the 'new_token' fresh
    policy: the only fresh blocks are blocks the new token opens)."""
    n = int((W.seq_lens > 0).sum())
    return W.step_slots.size == n


CASES = {
    # name: (workload factory, partition_tokens)
    "tiny_mha_d64": (lambda: wl.tiny_mha(), 0),
    "llama_small_auto": (lambda: wl.llama8b_gqa(small=True), 0),
    "llama_small_pt64": (lambda: wl.llama8b_gqa(small=True), 64),       # warp-owned
    "long_small_pt1024": (lambda: wl.long_context(small=True), 1024),  # g = 8, CTA-shared, split
    "long_small_pt512": (lambda: wl.long_context(small=True), 512),    # g = 8, warp-owned
    "g5_fp8": (lambda: wl.make_workload("g5_fp8", 6, 40, 8, 128, 1, 400, 17,
                                        kv_dtype="fp8_e4m3"), 0),
    "g5_fp8_pt32": (lambda: wl.make_workload("g5_fp8", 6, 40, 8, 128, 1, 400, 17,
                                             kv_dtype="fp8_e4m3"), 32),
    "d64_fp8_opening": (lambda: wl.make_workload(
        "d64_fp8", 5, 16, 4, 64, 0, 0, 8, kv_dtype="fp8_e4m3",
        seq_lens=[1, 17, 33, 48, 129]), 0),
    "opening_blocks_bf16": (lambda: wl.make_workload(
        "open_bf16", 6, 32, 8, 128, 0, 0, 9, seq_lens=[1, 16, 17, 513, 1024, 1025]), 0),
    # g = 16: two query sub-groups per kv head, whose warps both write the
    # token's (identical) bytes
    "g16_two_writers": (lambda: wl.make_workload(
        "g16", 4, 32, 2, 128, 0, 0, 10, seq_lens=[1, 33, 200, 700]), 0),
    "g16_two_writers_pt64": (lambda: wl.make_workload(
        "g16", 4, 32, 2, 128, 0, 0, 10, seq_lens=[1, 33, 200, 700]), 64),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_step_matches_two_call_step_and_oracle(name):
    make, pt = CASES[name]
    W = make()
    assert _new_token_only(W)
    # the two-call step: zero + write in one launch, then attention
    A = harness.upload(W)
    out_a = harness.gpu_step(W, A, partition_tokens=pt, fused=True)
    assert pkv_check()[0] == PKV_OK
    # the one-call step on a fresh copy of the same pool
    G = harness.upload(W)
    out_b = _step(W, G, pt)
    assert pkv_check()[0] == PKV_OK
    ka, va = _caches(A)
    kb, vb = _caches(G)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    assert torch.equal(out_a, out_b)
    kc, vc = harness.oracle_cache(W)
    assert np.array_equal(kb, kc.view(np.uint8).reshape(-1))
    assert np.array_equal(vb, vc.view(np.uint8).reshape(-1))
    harness.assert_close(out_b.float().cpu().numpy(), harness.oracle_out(W, kc, vc),
                         W.kv_dtype)


def test_step_empty_sequence_and_repeat():
    """A sequence of length 0 writes nothing and gives a zero row; a second
    identical step rewrites the same bytes and gives the same output."""
    W = wl.make_workload("empty", 4, 32, 8, 128, 0, 0, 21, seq_lens=[0, 16, 1, 300])
    G = harness.upload(W)
    out1 = _step(W, G, 0).clone()
    k1, v1 = _caches(G)
    out2 = _step(W, G, 0)
    assert pkv_check()[0] == PKV_OK
    k2, v2 = _caches(G)
    assert torch.equal(out1, out2)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    assert torch.all(out1[0] == 0)
    kc, vc = harness.oracle_cache(W)
    assert np.array_equal(k1, kc.view(np.uint8).reshape(-1))
    harness.assert_close(out1.float().cpu().numpy(), harness.oracle_out(W, kc, vc), "bf16")


def test_step_bad_block_id_writes_nothing_and_is_reported():
    """The new token's table entry points outside the pool: nothing is
    written, pkv_check reports a range error, and the other sequences are
    attended and written as usual."""
    W = wl.make_workload("badw", 4, 32, 8, 128, 0, 0, 23, seq_lens=[40, 33, 100, 17])
    G = harness.upload(W)
    before_k, before_v = _caches(G)
    tables = W.block_tables.copy()
    L1 = int(W.seq_lens[1])
    tables[1, (L1 - 1) // 16] = W.num_blocks + 5
    out = _step(W, G, 0, tables=torch.from_numpy(tables).cuda())
    st, _ = pkv_check()
    assert st == PKV_ERR_RANGE
    # the reference: the same step without sequence 1's write
    A = harness.upload(W)
    keep = np.array([s // 16 != int(W.block_tables[1, (L1 - 1) // 16]) for s in W.step_slots])
    fresh = np.array([f for f in W.fresh_blocks if f != int(W.block_tables[1, (L1 - 1) // 16])],
                     np.int32)
    idx = torch.from_numpy(np.nonzero(keep)[0]).cuda()
    paged_kv_zero_and_write(A.step_k[idx].contiguous(), A.step_v[idx].contiguous(),
                            A.step_slots[idx].contiguous(), A.cache, fresh)
    ref = paged_attention_decode(A.q, A.cache, A.tables, A.seq_lens, W.scale, W.max_seq_len)
    assert pkv_check()[0] == PKV_OK
    ka, va = _caches(A)
    kb, vb = _caches(G)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    rows = [0, 2, 3]
    assert torch.equal(out[rows], ref[rows])
    assert not np.array_equal(before_k, kb)  # the other sequences did write


def test_step_length_above_bound_writes_nothing():
    """A length above max_seq_len is attended clamped and reported, and its
    new token is not written: nothing lands at the clamped position."""
    W = wl.make_workload("longer", 2, 32, 8, 128, 0, 0, 29, seq_lens=[40, 100])
    G = harness.upload(W)
    _step(W, G, 0, max_seq_len=64)
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail == 1
    # the reference: sequence 0's token alone (neither token opens a block)
    A = harness.upload(W)
    s0 = int(W.block_tables[0, 39 // 16]) * 16 + 39 % 16
    i0 = W.step_slots.tolist().index(s0)
    paged_kv_zero_and_write(A.step_k[i0:i0 + 1].contiguous(), A.step_v[i0:i0 + 1].contiguous(),
                            A.step_slots[i0:i0 + 1].contiguous(), A.cache,
                            np.zeros(0, np.int32))
    assert pkv_check()[0] == PKV_OK
    ka, va = _caches(A)
    kb, vb = _caches(G)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)


def _tail_step(W, G, start_loc, pt, max_seq_len=None, tables=None):
    """The one-call step with the step's rows as the new tokens, delimited
    per sequence by start_loc (the rows are in sequence and position
    order)."""
    return paged_attention_decode_step(
        G.q, G.step_k, G.step_v, G.cache, G.tables if tables is None else tables,
        G.seq_lens, W.scale, max_seq_len=W.max_seq_len if max_seq_len is None else max_seq_len,
        partition_tokens=pt,
        new_start_loc=torch.from_numpy(np.asarray(start_loc, np.int32)).cuda())


def _check_against_two_call(W, start_loc, pt):
    A = harness.upload(W)
    out_a = harness.gpu_step(W, A, partition_tokens=pt, fused=True)
    assert pkv_check()[0] == PKV_OK
    G = harness.upload(W)
    out_b = _tail_step(W, G, start_loc, pt)
    assert pkv_check()[0] == PKV_OK
    ka, va = _caches(A)
    kb, vb = _caches(G)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    assert torch.equal(out_a, out_b)
    kc, vc = harness.oracle_cache(W)
    assert np.array_equal(kb, kc.view(np.uint8).reshape(-1))
    assert np.array_equal(vb, vc.view(np.uint8).reshape(-1))
    harness.assert_close(out_b.float().cpu().numpy(), harness.oracle_out(W, kc, vc),
                         W.kv_dtype)


@pytest.mark.parametrize("pt", [0, 64])
def test_step_recycled_tail_fp8(pt):
    """The fp8 recycling step (its recycled blocks are each sequence's last
    four or five, every valid slot rewritten, the new token included) as one
    call: each sequence's rewritten tail is its new tokens."""
    W = wl.fp8_recycle(small=True)
    rows, start = W.new_token_tail()
    assert np.array_equal(rows, np.arange(W.step_slots.size))
    _check_against_two_call(W, start, pt)


TAILS = [1, 5, 16, 17, 20, 33, 0, 40]


@pytest.mark.parametrize("pt,kv_dtype", [(0, "bf16"), (64, "bf16"), (32, "fp8_e4m3")])
def test_step_tails_of_several_tokens(pt, kv_dtype):
    """Tails of 0 to 40 tokens: starting mid-block (the block keeps its
    earlier rows), at a block start (the block opens: rows past the sequence
    zeroed), across several blocks and across partitions of 32 and 64
    tokens; a sequence with no new token writes nothing."""
    base = (wl.llama8b_gqa(small=True) if kv_dtype == "bf16" else
            wl.make_workload("tails_fp8", 8, 32, 8, 128, 20, 700, 5, kv_dtype="fp8_e4m3"))
    W = wl.with_step_tail(base, TAILS, seed=11)
    start = np.concatenate([[0], np.cumsum(np.minimum(TAILS, base.seq_lens))])
    _check_against_two_call(W, start, pt)


def test_step_tail_longer_than_sequence_writes_nothing():
    """A sequence whose new-token count exceeds its length is reported and
    writes nothing; the others are written as usual."""
    base = wl.make_workload("tail_bad", 3, 32, 8, 128, 0, 0, 31, seq_lens=[20, 40, 9])
    W = wl.with_step_tail(base, [3, 2, 9], seed=4)
    G = harness.upload(W)
    # sequence 2 claims 12 new tokens (rows 5 .. 16) but holds 9 positions
    k = torch.cat([G.step_k, G.step_k[-3:]])
    v = torch.cat([G.step_v, G.step_v[-3:]])
    paged_attention_decode_step(G.q, k.contiguous(), v.contiguous(), G.cache, G.tables,
                                G.seq_lens, W.scale, W.max_seq_len,
                                new_start_loc=torch.tensor([0, 3, 5, 17], dtype=torch.int32,
                                                           device="cuda"))
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail == 2
    # the reference: the rows of sequences 0 and 1 only (their tails open
    # no block)
    A = harness.upload(W)
    paged_kv_zero_and_write(A.step_k[:5].contiguous(), A.step_v[:5].contiguous(),
                            A.step_slots[:5].contiguous(), A.cache, np.zeros(0, np.int32))
    assert pkv_check()[0] == PKV_OK
    ka, va = _caches(A)
    kb, vb = _caches(G)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)


@pytest.mark.parametrize("pt", [0, 512])
def test_step_full_size_llama8b(pt):
    """The Llama-8B decode step at full size in the bench's launch
    configuration (the table width as the host bound): cache bytes equal the
    oracle's, and sampled rows match the oracle."""
    W = wl.llama8b_gqa()
    G = harness.upload(W)
    out = _step(W, G, pt, max_seq_len=W.max_blocks * 16)
    assert pkv_check()[0] == PKV_OK
    kc, vc = harness.oracle_cache(W)
    kb, vb = _caches(G)
    assert np.array_equal(kb, kc.view(np.uint8).reshape(-1))
    assert np.array_equal(vb, vc.view(np.uint8).reshape(-1))
    rng = np.random.default_rng(pt + 1)
    pairs = np.array([[b, h] for b in range(W.batch) for h in rng.choice(W.num_heads, 2,
                                                                          replace=False)],
                     np.int32)
    ref = harness.oracle_out(W, kc, vc, pairs=pairs)
    gpu = out.float().cpu().numpy()
    harness.assert_close(gpu[pairs[:, 0], pairs[:, 1]], ref[pairs[:, 0], pairs[:, 1]], "bf16")
