"""Seeded synthetic decode workloads for the paged KV-cache path.

This module only draws inputs: sequence lengths, a shuffled physical block
pool with reference counts, per-sequence block tables, slot mappings, query
and key/value values, the list of freshly allocated blocks and the initial
(stale) bytes of the pool.  It performs none of the method's arithmetic (no
write, zeroing, quantisation or attention), so both the CUDA path and the
CPU oracle consume exactly the same inputs from here.

Structure follows the vLLM pages:
 - vLLM concept page (compassingai.com), "15 分钟专家深入" item 2: blocks of
   16 tokens, a page table per sequence, blocks allocated on demand, shared
   prompt prefixes pointing at the same physical blocks;
 - vLLM internals (naphjohn.github.io), §1.1 and Figure 1: blocks scattered
   anywhere in the pool, reference counts on shared prefix blocks, at most
   one partially filled block per sequence;
 - vLLM v0.17.1 notes (admirer.cn), "重点：35219": recycled blocks still hold
   fp32 bit patterns (NaN/Inf among them) when they are handed out again.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16

# Explicit fp32 bit patterns planted in recycled blocks: quiet NaN, +Inf, -Inf.
STALE_PATTERNS = (0x7FC00000, 0x7F800000, 0xFF800000)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even) and return
    the 16-bit patterns.  Used only to draw bf16 inputs."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not np.isfinite(x).all():
        raise ValueError("bf16_bits draws finite values only")
    u = x.view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))) >> 16
    return rounded.astype(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """The float32 value of bfloat16 bit patterns (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(
        np.float32)


class BlockPool:
    """Physical block pool with a seeded shuffled free list and reference
    counts.  A block with refcount > 1 is shared (a common prompt prefix);
    freeing drops one reference and returns the block to the pool when the
    count reaches zero."""

    def __init__(self, num_blocks: int, rng: np.random.Generator):
        self.num_blocks = int(num_blocks)
        self.free_list = deque(int(b) for b in rng.permutation(self.num_blocks))
        self.refcount = np.zeros(self.num_blocks, dtype=np.int32)

    @property
    def used(self) -> int:
        return int(np.count_nonzero(self.refcount))

    def allocate(self) -> int:
        if not self.free_list:
            raise RuntimeError("block pool exhausted")
        b = self.free_list.popleft()
        self.refcount[b] = 1
        return b

    def share(self, block: int) -> int:
        if self.refcount[block] <= 0:
            raise ValueError("sharing a free block")
        self.refcount[block] += 1
        return block

    def free(self, block: int) -> None:
        if self.refcount[block] <= 0:
            raise ValueError("double free")
        self.refcount[block] -= 1
        if self.refcount[block] == 0:
            self.free_list.append(int(block))


@dataclass
class Workload:
    """One decode step's inputs plus the history that precedes it."""
    name: str
    batch: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str                 # "bf16" or "fp8_e4m3"
    num_blocks: int
    max_blocks: int
    seq_lens: np.ndarray          # int32 [B]
    block_tables: np.ndarray      # int32 [B, max_blocks], -1 = unused
    q: np.ndarray                 # uint16 bf16 bits [B, Hq, d]
    hist_k: np.ndarray            # uint16 [Th, Hkv, d] written at set-up
    hist_v: np.ndarray
    hist_slots: np.ndarray        # int64 [Th]
    step_k: np.ndarray            # uint16 [Ts, Hkv, d] written in the step
    step_v: np.ndarray
    step_slots: np.ndarray        # int64 [Ts]
    fresh_blocks: np.ndarray      # int32 [n] zeroed in the step
    init_key: np.ndarray          # uint8 [NB * block_bytes] pool bytes
    init_value: np.ndarray
    k_scale: float = 1.0
    v_scale: float = 1.0
    scale: float = 0.0
    block_size: int = BLOCK_SIZE
    refcount: np.ndarray = field(default=None)   # int32 [NB]
    groups: list = field(default_factory=list)   # prefix-sharing groups
    seed: int = 0

    def new_token_tail(self):
        """(rows, start_loc) when the step's writes are, for every
        sequence, its last n_b >= 1 positions, and the fresh blocks are
        exactly the blocks whose first position is among them (the layout of
        a decode step that appends new tokens): rows orders the step's write
        rows sequence by sequence, position by position, and start_loc
        (int32 [batch + 1]) delimits each sequence's rows.  Otherwise None."""
        bs = self.block_size
        pos = {int(s): i for i, s in enumerate(self.step_slots)}
        rows, start, opened = [], [0], set()
        for b in range(self.batch):
            L = int(self.seq_lens[b])
            t, mine = L - 1, []
            while t >= 0:
                i = pos.get(int(self.block_tables[b, t // bs]) * bs + t % bs)
                if i is None:
                    break
                mine.append(i)
                t -= 1
            if not mine:
                return None
            w0 = t + 1
            rows += mine[::-1]
            start.append(len(rows))
            for j in range(-(-w0 // bs), (L - 1) // bs + 1):
                opened.add(int(self.block_tables[b, j]))
        if len(rows) != self.step_slots.size or \
                set(int(f) for f in self.fresh_blocks) != opened:
            return None
        return np.asarray(rows, dtype=np.int64), np.asarray(start, dtype=np.int32)

    @property
    def elem_bytes(self) -> int:
        return 2 if self.kv_dtype == "bf16" else 1

    @property
    def block_bytes(self) -> int:
        return self.block_size * self.num_kv_heads * self.head_dim * self.elem_bytes

    @property
    def group_size(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.batch else 0

    def kv_read_bytes(self) -> int:
        """Algorithmic K+V bytes one decode step reads (logical, per
        sequence; shared prefix blocks count once per sequence)."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * \
            self.head_dim * 2 * self.elem_bytes

    def unique_kv_read_bytes(self) -> int:
        """K+V bytes of the distinct cached tokens the step reads."""
        seen = {}
        for b in range(self.batch):
            L = int(self.seq_lens[b])
            for j in range((L + self.block_size - 1) // self.block_size):
                blk = int(self.block_tables[b, j])
                n = min(self.block_size, L - j * self.block_size)
                seen[blk] = max(seen.get(blk, 0), n)
        return sum(seen.values()) * self.num_kv_heads * self.head_dim * 2 * \
            self.elem_bytes


def _draw_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def make_workload(name: str, batch: int, num_heads: int, num_kv_heads: int,
                  head_dim: int, len_lo: int, len_hi: int, seed: int,
                  kv_dtype: str = "bf16", pool_factor: float = 1.2,
                  seq_lens=None, num_blocks=None, max_len=None,
                  prefix_groups: int = 0, prefix_len: int = 0,
                  fresh_policy: str = "new_token") -> Workload:
    """Draw one workload.

    seq_lens uniform in [len_lo, len_hi] unless given.  The pool holds
    ceil(pool_factor * blocks needed) blocks (or ``num_blocks``), handed out
    in a seeded shuffled order.  With ``prefix_groups`` > 0 the batch is cut
    into that many equal groups whose first ``prefix_len`` tokens (a whole
    number of blocks) share the same physical blocks; seq_lens then count
    the prefix plus a private suffix drawn from [len_lo, len_hi].

    fresh_policy:
      "new_token"  -- a block is fresh when the step's new token (position
                      L-1) is its first slot;
      "recycle515" -- the last four logical blocks of every sequence plus the
                      fifth-last block of sequences 0, 1 and 2.
    Tokens that live in fresh blocks, and every sequence's new token, are
    written during the step (after zeroing); all others at set-up.
    """
    bs = BLOCK_SIZE
    rng = np.random.default_rng(seed)
    if seq_lens is None:
        lens = rng.integers(len_lo, len_hi + 1, size=batch).astype(np.int64)
    else:
        lens = np.asarray(seq_lens, dtype=np.int64)
    if prefix_groups:
        assert prefix_len % bs == 0 and batch % prefix_groups == 0
        lens = lens + prefix_len
    nblk = (lens + bs - 1) // bs
    if max_len is None:
        max_len = int(lens.max()) if batch else 0
    max_blocks = max(1, (int(max_len) + bs - 1) // bs)
    prefix_blocks = prefix_len // bs
    if prefix_groups:
        needed = prefix_groups * prefix_blocks + int((nblk - prefix_blocks).sum())
    else:
        needed = int(nblk.sum())
    if num_blocks is None:
        num_blocks = int(np.ceil(pool_factor * needed))
    pool = BlockPool(num_blocks, rng)

    tables = np.full((batch, max_blocks), -1, dtype=np.int32)
    groups = []
    if prefix_groups:
        per = batch // prefix_groups
        for gi in range(prefix_groups):
            shared = [pool.allocate() for _ in range(prefix_blocks)]
            members = list(range(gi * per, (gi + 1) * per))
            groups.append({"members": members, "prefix_blocks": shared})
            for b in members:
                for j, blk in enumerate(shared):
                    tables[b, j] = pool.share(blk) if b != members[0] else blk
                for j in range(prefix_blocks, int(nblk[b])):
                    tables[b, j] = pool.allocate()
    else:
        for b in range(batch):
            for j in range(int(nblk[b])):
                tables[b, j] = pool.allocate()

    fresh = []
    if fresh_policy == "new_token":
        for b in range(batch):
            L = int(lens[b])
            if L > 0 and (L - 1) % bs == 0:
                fresh.append(int(tables[b, (L - 1) // bs]))
    elif fresh_policy == "recycle515":
        for b in range(batch):
            n = int(nblk[b])
            take = 5 if b < 3 else 4
            for j in range(max(0, n - take), n):
                fresh.append(int(tables[b, j]))
    elif fresh_policy != "none":
        raise ValueError(fresh_policy)
    fresh_set = set(fresh)

    # Token positions: shared prefix tokens once per group, then each
    # sequence's private tokens.
    hkd = (num_kv_heads, head_dim)
    fresh_arr = np.asarray(sorted(fresh_set), dtype=np.int64)
    hist_parts, step_parts = [], []
    for grp in groups:
        t = np.arange(prefix_len, dtype=np.int64)
        blks = np.asarray(grp["prefix_blocks"], dtype=np.int64)[t // bs]
        hist_parts.append(blks * bs + t % bs)
    for b in range(batch):
        L = int(lens[b])
        start = prefix_len if prefix_groups else 0
        t = np.arange(start, L, dtype=np.int64)
        blks = tables[b, t // bs].astype(np.int64)
        slots = blks * bs + t % bs
        in_step = np.isin(blks, fresh_arr) | (t == L - 1)
        step_parts.append(slots[in_step])
        hist_parts.append(slots[~in_step])
    hist_slots = np.concatenate(hist_parts) if hist_parts else \
        np.zeros(0, np.int64)
    step_slots = np.concatenate(step_parts) if step_parts else \
        np.zeros(0, np.int64)

    q = _draw_bf16(rng, (batch, num_heads, head_dim))
    hist_k = _draw_bf16(rng, (hist_slots.size, *hkd))
    hist_v = _draw_bf16(rng, (hist_slots.size, *hkd))
    step_k = _draw_bf16(rng, (step_slots.size, *hkd))
    step_v = _draw_bf16(rng, (step_slots.size, *hkd))

    k_scale = v_scale = 1.0
    if kv_dtype == "fp8_e4m3":
        # per-tensor scale: largest magnitude written maps to 448, the
        # largest finite E4M3 value.
        def amax(*arrs):
            m = 0.0
            for a in arrs:
                if a.size:
                    m = max(m, float(np.abs(bf16_values(a)).max()))
            return m
        k_scale = float(np.float32(amax(hist_k, step_k) / 448.0))
        v_scale = float(np.float32(amax(hist_v, step_v) / 448.0))
    elif kv_dtype != "bf16":
        raise ValueError(kv_dtype)

    eb = 2 if kv_dtype == "bf16" else 1
    block_bytes = bs * num_kv_heads * head_dim * eb
    # Pool bytes before the step: 0xFF everywhere (NaN in bf16 and in E4M3,
    # so any read of a slot that is not part of a sequence is visible), and
    # random fp32 words with planted NaN/Inf in the freshly allocated blocks.
    init_key = np.full(num_blocks * block_bytes, 0xFF, dtype=np.uint8)
    init_value = np.full(num_blocks * block_bytes, 0xFF, dtype=np.uint8)
    for arr in (init_key, init_value):
        for blk in fresh:
            words = rng.integers(0, 2**32, size=block_bytes // 4,
                                 dtype=np.uint64).astype(np.uint32)
            words[: len(STALE_PATTERNS)] = STALE_PATTERNS
            pos = rng.integers(0, words.size, size=len(STALE_PATTERNS))
            words[pos] = STALE_PATTERNS
            arr[blk * block_bytes:(blk + 1) * block_bytes] = words.view(np.uint8)

    return Workload(
        name=name, batch=batch, num_heads=num_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, kv_dtype=kv_dtype,
        num_blocks=num_blocks, max_blocks=max_blocks,
        seq_lens=lens.astype(np.int32), block_tables=tables, q=q,
        hist_k=hist_k, hist_v=hist_v, hist_slots=hist_slots,
        step_k=step_k, step_v=step_v, step_slots=step_slots,
        fresh_blocks=np.asarray(fresh, dtype=np.int32),
        init_key=init_key, init_value=init_value, k_scale=k_scale,
        v_scale=v_scale, scale=1.0 / float(np.sqrt(head_dim)),
        refcount=pool.refcount.copy(), groups=groups, seed=seed)


def with_step_tail(W: Workload, tails, seed: int) -> Workload:
    """W with a different step: sequence b rewrites its last tails[b]
    positions (at most its length) with fresh seeded values, and the fresh
    blocks are the blocks whose first position is among them.  W's own step
    writes that the new tails leave out move to the set-up history, so that
    every position below seq_lens is written."""
    from dataclasses import replace
    bs = W.block_size
    rng = np.random.default_rng(seed)
    slots, fresh = [], set()
    for b in range(W.batch):
        L = int(W.seq_lens[b])
        w0 = L - min(int(tails[b]), L)
        for t in range(w0, L):
            slots.append(int(W.block_tables[b, t // bs]) * bs + t % bs)
        for j in range(-(-w0 // bs), (L - 1) // bs + 1 if L else 0):
            fresh.add(int(W.block_tables[b, j]))
    hkd = (W.num_kv_heads, W.head_dim)
    keep = ~np.isin(W.step_slots, np.asarray(slots, dtype=np.int64))
    return replace(W, step_k=_draw_bf16(rng, (len(slots), *hkd)),
                   step_v=_draw_bf16(rng, (len(slots), *hkd)),
                   step_slots=np.asarray(slots, dtype=np.int64),
                   fresh_blocks=np.asarray(sorted(fresh), dtype=np.int32),
                   hist_k=np.concatenate([W.hist_k, W.step_k[keep]]),
                   hist_v=np.concatenate([W.hist_v, W.step_v[keep]]),
                   hist_slots=np.concatenate([W.hist_slots, W.step_slots[keep]]))


# ---------------------------------------------------------------------------
# The five decode workloads, full size and a small variant of each that the
# fp64 oracle finishes in seconds while still spanning several blocks,
# several 512-token partitions and a ragged last block.
# ---------------------------------------------------------------------------

def tiny_mha(seed: int = 0) -> Workload:
    """4 sequences, lengths {1,17,33,64}, 8 q = 8 kv heads, head_dim 64,
    a 64-block pool whose blocks are taken in a seeded permuted order."""
    return make_workload("tiny_mha", 4, 8, 8, 64, 0, 0, seed,
                         seq_lens=[1, 17, 33, 64], num_blocks=64)


def llama8b_gqa(seed: int = 5, small: bool = False) -> Workload:
    """Llama-8B-shaped GQA decode: 32 q / 8 kv heads, head_dim 128,
    seq_lens uniform in [512, 4096], pool 20% larger than needed.  The
    default seed draws 4 sequences whose new token opens a block, the
    expected count for 64 sequences and 16-token blocks."""
    if small:
        return make_workload("llama8b_gqa_small", 8, 32, 8, 128, 20, 700,
                             seed)
    return make_workload("llama8b_gqa", 64, 32, 8, 128, 512, 4096, seed,
                         max_len=4096)


def prefix_shared(seed: int = 2, small: bool = False) -> Workload:
    """16 groups x 16 sequences sharing a 1024-token prefix (64 blocks,
    refcount 16) plus private suffixes uniform in [32, 512]."""
    if small:
        return make_workload("prefix_shared_small", 8, 32, 8, 128, 5, 60,
                             seed, prefix_groups=2, prefix_len=64)
    return make_workload("prefix_shared", 256, 32, 8, 128, 32, 512, seed,
                         prefix_groups=16, prefix_len=1024,
                         max_len=1024 + 512)


def long_context(seed: int = 3, small: bool = False) -> Workload:
    """Long-context decode: batch 8, seq_lens uniform in [32768, 131072],
    64 q / 8 kv heads, head_dim 128 (split into 512-token partitions)."""
    if small:
        return make_workload("long_context_small", 2, 64, 8, 128, 1500, 3000,
                             seed)
    return make_workload("long_context", 8, 64, 8, 128, 32768, 131072, seed,
                         max_len=131072)


def fp8_recycle(seed: int = 4, small: bool = False) -> Workload:
    """fp8 E4M3 KV with a per-tensor scale, batch 128, 40 q / 8 kv heads,
    head_dim 128, seq_lens uniform in [1024, 8192]; 515 recycled blocks
    holding stale fp32 bit patterns are zeroed before the step's writes."""
    if small:
        return make_workload("fp8_recycle_small", 6, 40, 8, 128, 40, 300,
                             seed, kv_dtype="fp8_e4m3",
                             fresh_policy="recycle515")
    return make_workload("fp8_recycle", 128, 40, 8, 128, 1024, 8192, seed,
                         kv_dtype="fp8_e4m3", fresh_policy="recycle515",
                         max_len=8192)


CONFIGS = {
    "tiny_mha": tiny_mha,
    "llama8b_gqa": llama8b_gqa,
    "prefix_shared": prefix_shared,
    "long_context": long_context,
    "fp8_recycle": fp8_recycle,
}


# ---------------------------------------------------------------------------
# Chunked-prefill workloads (vLLM concept page, "Continuous Batching":
# long prompts are cut into chunks that run inside ordinary steps).  Each
# sequence has `history` tokens cached by earlier steps and brings a chunk of
# `chunk` new tokens whose K/V the step writes before attention reads them.
# ---------------------------------------------------------------------------

@dataclass
class PrefillWorkload:
    """One chunked-prefill step: the cached history and the chunk's tokens."""
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    max_blocks: int
    history: np.ndarray           # int32 [B] tokens cached before the step
    chunk: np.ndarray             # int32 [B] query tokens of the step
    block_tables: np.ndarray      # int32 [B, max_blocks], -1 = unused
    q: np.ndarray                 # uint16 bf16 bits [T, Hq, d]
    hist_k: np.ndarray            # uint16 [Th, Hkv, d] in the pool at set-up
    hist_v: np.ndarray
    hist_slots: np.ndarray        # int64 [Th]
    step_k: np.ndarray            # uint16 [T, Hkv, d] written in the step
    step_v: np.ndarray
    step_slots: np.ndarray        # int64 [T]
    init_key: np.ndarray          # uint8 pool bytes before set-up
    init_value: np.ndarray
    scale: float = 0.0
    kv_dtype: str = "bf16"
    k_scale: float = 1.0
    v_scale: float = 1.0
    block_size: int = BLOCK_SIZE
    seed: int = 0

    @property
    def batch(self) -> int:
        return int(self.chunk.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.chunk.sum())

    @property
    def seq_lens(self) -> np.ndarray:
        return (self.history + self.chunk).astype(np.int32)

    @property
    def query_start_loc(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.chunk)]).astype(np.int32)

    @property
    def max_query_len(self) -> int:
        return int(self.chunk.max()) if self.batch else 0

    @property
    def elem_bytes(self) -> int:
        return 2 if self.kv_dtype == "bf16" else 1

    @property
    def block_bytes(self) -> int:
        return self.block_size * self.num_kv_heads * self.head_dim * self.elem_bytes

    def attention_flops(self) -> int:
        """Algorithmic multiply-add flops of the step's attention: every
        (query token, q head) row sees history + i + 1 keys and spends
        2 d flops on each score and 2 d on each value row."""
        n = self.chunk.astype(np.int64)
        keys = n * self.history.astype(np.int64) + n * (n + 1) // 2
        return int(keys.sum()) * self.num_heads * 4 * self.head_dim


def make_prefill_workload(name: str, history, chunk, num_heads: int,
                          num_kv_heads: int, head_dim: int, seed: int,
                          pool_factor: float = 1.2,
                          kv_dtype: str = "bf16") -> PrefillWorkload:
    """Draw a chunked-prefill step: blocks for every sequence taken from a
    shuffled pool 20% larger than needed, the whole pool first filled with
    0xFF bytes (NaN in bf16 and in E4M3) so that any read of an unwritten
    slot shows, history K/V drawn N(0,1) in place, the chunk's K/V and q
    drawn N(0,1).  For an E4M3 cache each tensor's scale maps its largest
    magnitude to 448 (the values are quantised by the write step)."""
    rng = np.random.default_rng(seed)
    history = np.asarray(history, dtype=np.int32)
    chunk = np.asarray(chunk, dtype=np.int32)
    lens = history + chunk
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    max_blocks = max(1, int(nblk.max()) if len(nblk) else 1)
    num_blocks = max(8, int(np.ceil(pool_factor * int(nblk.sum()))))
    pool = BlockPool(num_blocks, rng)
    tables = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    for b, n in enumerate(nblk):
        for j in range(int(n)):
            tables[b, j] = pool.allocate()
    Hkv, d = num_kv_heads, head_dim

    def slots_of(b, lo, hi):
        t = np.arange(lo, hi, dtype=np.int64)
        return tables[b, t // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE + t % BLOCK_SIZE

    hist_slots = np.concatenate([slots_of(b, 0, int(history[b]))
                                 for b in range(len(lens))] or [np.zeros(0, np.int64)])
    step_slots = np.concatenate([slots_of(b, int(history[b]), int(lens[b]))
                                 for b in range(len(lens))] or [np.zeros(0, np.int64)])
    Th, T = hist_slots.size, step_slots.size
    elt = 2 if kv_dtype == "bf16" else 1
    pool_bytes = num_blocks * BLOCK_SIZE * Hkv * d * elt
    q = _draw_bf16(rng, (T, num_heads, d))
    hist_k, hist_v = _draw_bf16(rng, (Th, Hkv, d)), _draw_bf16(rng, (Th, Hkv, d))
    step_k, step_v = _draw_bf16(rng, (T, Hkv, d)), _draw_bf16(rng, (T, Hkv, d))
    k_scale = v_scale = 1.0
    if kv_dtype != "bf16":
        amax = lambda *a: max(float(np.abs(bf16_values(x)).max()) if x.size else 0.0
                              for x in a)
        k_scale = float(np.float32(amax(hist_k, step_k) / 448.0))
        v_scale = float(np.float32(amax(hist_v, step_v) / 448.0))
    return PrefillWorkload(
        name=name, num_heads=num_heads, num_kv_heads=Hkv, head_dim=d,
        num_blocks=num_blocks, max_blocks=max_blocks, history=history,
        chunk=chunk, block_tables=tables, q=q,
        hist_k=hist_k, hist_v=hist_v, hist_slots=hist_slots,
        step_k=step_k, step_v=step_v, step_slots=step_slots,
        init_key=np.full(pool_bytes, 0xFF, dtype=np.uint8),
        init_value=np.full(pool_bytes, 0xFF, dtype=np.uint8),
        scale=1.0 / float(np.sqrt(d)), kv_dtype=kv_dtype, k_scale=k_scale,
        v_scale=v_scale, seed=seed)


def prefill_8k(seed: int = 6, small: bool = False,
               kv_dtype: str = "bf16") -> PrefillWorkload:
    """Prefill step of about 8K tokens (the vLLM v0.17.1 notes' prefill
    batch size): 8 fresh prompts of 1024 tokens, Llama-8B shape (32 q /
    8 kv heads, head_dim 128)."""
    if small:
        return make_prefill_workload("prefill_8k_small", [0, 0, 0],
                                     [300, 129, 17], 32, 8, 128, seed,
                                     kv_dtype=kv_dtype)
    return make_prefill_workload("prefill_8k", [0] * 8, [1024] * 8, 32, 8, 128,
                                 seed, kv_dtype=kv_dtype)


def chunked_prefill_8k(seed: int = 7, small: bool = False,
                       kv_dtype: str = "bf16") -> PrefillWorkload:
    """Chunked prefill of about 8K tokens: 8 chunks of 1024 tokens, each
    after a history uniform in [1024, 7168] tokens, Llama-8B shape."""
    rng = np.random.default_rng(seed)
    if small:
        hist = [int(x) for x in rng.integers(50, 600, 4)]
        return make_prefill_workload("chunked_prefill_8k_small", hist,
                                     [200, 37, 1, 130], 32, 8, 128, seed,
                                     kv_dtype=kv_dtype)
    hist = [int(x) for x in rng.integers(1024, 7169, 8)]
    return make_prefill_workload("chunked_prefill_8k", hist, [1024] * 8, 32, 8,
                                 128, seed, kv_dtype=kv_dtype)


def chunked_prefill_8k_fp8(seed: int = 7, small: bool = False) -> PrefillWorkload:
    """The chunked-prefill step on an E4M3 cache with per-tensor scales."""
    return chunked_prefill_8k(seed, small, kv_dtype="fp8_e4m3")


PREFILL_CONFIGS = {
    "prefill_8k": prefill_8k,
    "chunked_prefill_8k": chunked_prefill_8k,
    "chunked_prefill_8k_fp8": chunked_prefill_8k_fp8,
}
