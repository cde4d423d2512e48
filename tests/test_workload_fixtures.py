"""Host-side fixtures of the block pool and the generated workloads (no GPU).

The vLLM pages state invariants of the paged layout that every generated
workload must keep, whatever the kernels do with it:
  - blocks are handed out whole; at most one block per sequence is partly
    filled, so at most 15 slots per sequence are wasted (internals post,
    §1.2);
  - a shared prompt prefix is the same physical blocks in every member's
    table, with a reference count, never a copy (internals post, §1.1 and
    Figure 1);
  - only freshly allocated blocks are zeroed, and they belong to exactly
    one sequence (v0.17.1 notes, "修复方案");
  - every cached token has exactly one slot, reached through its
    sequence's table (concept page, "15 分钟专家深入" item 2).
"""
import numpy as np
import pytest

from paged_kv_cache_48_gb300 import workload as wl

BS = 16


def test_block_pool_allocate_share_free():
    pool = wl.BlockPool(5, np.random.default_rng(0))
    got = [pool.allocate() for _ in range(5)]
    assert sorted(got) == list(range(5))
    with pytest.raises(RuntimeError):
        pool.allocate()
    b = got[0]
    pool.share(b)
    pool.share(b)
    assert pool.refcount[b] == 3
    pool.free(b)
    pool.free(b)
    assert pool.refcount[b] == 1 and pool.used == 5
    pool.free(b)
    assert pool.refcount[b] == 0 and pool.used == 4
    with pytest.raises(ValueError):
        pool.free(b)               # double free
    with pytest.raises(ValueError):
        pool.share(b)              # sharing a free block
    assert pool.allocate() == b    # the freed block is handed out again


DECODE = [wl.tiny_mha(), wl.llama8b_gqa(small=True), wl.prefix_shared(small=True),
          wl.long_context(small=True), wl.fp8_recycle(small=True)]


@pytest.mark.parametrize("W", DECODE, ids=[W.name for W in DECODE])
def test_decode_workload_layout(W):
    nblk = (W.seq_lens + BS - 1) // BS
    occurrences = np.zeros(W.num_blocks, np.int64)
    for b in range(W.batch):
        row = W.block_tables[b]
        n = int(nblk[b])
        # whole blocks, at most one partly filled: waste <= 15 slots
        assert n * BS - int(W.seq_lens[b]) <= BS - 1
        assert np.all((row[:n] >= 0) & (row[:n] < W.num_blocks))
        assert np.all(row[n:] == -1)
        assert len(set(row[:n].tolist())) == n   # no block twice in one table
        np.add.at(occurrences, row[:n], 1)
    # reference counts equal table occurrences
    assert np.array_equal(W.refcount, occurrences)
    # every cached token has exactly one slot, through its own table
    slots = np.concatenate([W.hist_slots, W.step_slots])
    assert len(set(slots.tolist())) == slots.size
    expect = set()
    for b in range(W.batch):
        t = np.arange(int(W.seq_lens[b]))
        expect.update((W.block_tables[b, t // BS].astype(np.int64) * BS + t % BS).tolist())
    assert set(slots.tolist()) == expect
    # fresh blocks: owned, not shared, and all their tokens written in the step
    for blk in W.fresh_blocks.tolist():
        assert W.refcount[blk] == 1
    step = set(W.step_slots.tolist())
    for blk in W.fresh_blocks.tolist():
        owned = [s for s in expect if s // BS == blk]
        assert set(owned) <= step


def test_prefix_groups_share_physical_blocks():
    W = wl.prefix_shared(small=True)
    for grp in W.groups:
        pb = grp["prefix_blocks"]
        for b in grp["members"]:
            assert list(W.block_tables[b, :len(pb)]) == list(pb)
        for blk in pb:
            assert W.refcount[blk] == len(grp["members"])
    # private blocks are private
    shared = {blk for grp in W.groups for blk in grp["prefix_blocks"]}
    for b in range(W.batch):
        n = (int(W.seq_lens[b]) + BS - 1) // BS
        for blk in W.block_tables[b, :n].tolist():
            if blk not in shared:
                assert W.refcount[blk] == 1


def test_recycled_blocks_hold_stale_patterns_before_zeroing():
    """The fp8 workload's recycled blocks start with fp32 NaN / +-Inf bit
    patterns (the stale state the v0.17.1 notes describe), so a kernel that
    skipped the zeroing would read them."""
    W = wl.fp8_recycle(small=True)
    assert W.fresh_blocks.size == 3 * 5 + (W.batch - 3) * 4
    bb = W.block_bytes
    words = set()
    for blk in W.fresh_blocks.tolist():
        chunk = W.init_key[blk * bb:(blk + 1) * bb].view(np.uint32)
        words.update(int(x) for x in chunk[:64])
    assert {0x7FC00000, 0x7F800000, 0xFF800000} & words


@pytest.mark.parametrize("cfg", sorted(wl.PREFILL_CONFIGS))
def test_prefill_workload_layout(cfg):
    W = wl.PREFILL_CONFIGS[cfg](small=True)
    qsl = W.query_start_loc
    assert qsl[0] == 0 and qsl[-1] == W.num_tokens and np.all(np.diff(qsl) >= 0)
    for b in range(W.batch):
        L = int(W.seq_lens[b])
        n = (L + BS - 1) // BS
        assert n * BS - L <= BS - 1
        row = W.block_tables[b]
        # the chunk's slots are positions history .. history + chunk - 1
        t = np.arange(int(W.history[b]), L)
        want = row[t // BS].astype(np.int64) * BS + t % BS
        assert np.array_equal(W.step_slots[qsl[b]:qsl[b + 1]], want)
    assert W.attention_flops() == sum(
        int(c) * int(h) + int(c) * (int(c) + 1) // 2
        for h, c in zip(W.history, W.chunk)) * W.num_heads * 4 * W.head_dim


def test_step_tail_fixture_writes_every_position():
    """with_step_tail (the decode-step tests' fixture): every position below
    each sequence's length is written, at set-up or in the step; the step
    writes exactly the requested tails; the fresh blocks are the blocks that
    open inside a tail; and new_token_tail recovers the layout whenever
    every tail is non-empty."""
    from paged_kv_cache_48_gb300 import workload as wl
    base = wl.llama8b_gqa(small=True)
    tails = [1, 5, 16, 17, 20, 33, 0, 40]
    W = wl.with_step_tail(base, tails, seed=11)
    bs = W.block_size
    written = set(W.hist_slots.tolist()) | set(W.step_slots.tolist())
    step = set(W.step_slots.tolist())
    opened = set()
    for b in range(W.batch):
        L = int(W.seq_lens[b])
        slot = lambda t: int(W.block_tables[b, t // bs]) * bs + t % bs
        assert all(slot(t) in written for t in range(L))
        n = min(tails[b], L)
        assert {slot(t) for t in range(L - n, L)} <= step
        opened |= {int(W.block_tables[b, j]) for j in range(-(-(L - n) // bs), (L - 1) // bs + 1)
                   if n}
    assert W.step_slots.size == sum(min(t, int(L)) for t, L in zip(tails, W.seq_lens))
    assert set(W.fresh_blocks.tolist()) == opened
    assert W.new_token_tail() is None           # sequence 6 has no new token
    W1 = wl.with_step_tail(base, [3] * base.batch, seed=2)
    rows, start = W1.new_token_tail()
    assert list(start) == [3 * b for b in range(base.batch + 1)]
    assert np.array_equal(rows, np.arange(3 * base.batch))
