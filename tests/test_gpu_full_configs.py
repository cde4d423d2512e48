"""The five workloads at full size, each in exactly the step bench.py times:
the zeroing of fresh blocks and the write of the step's tokens in one
paged_kv_zero_and_write launch, then decode attention with the table width
(max_blocks * 16) as the host bound and automatic partitioning; the
long-context workload also with the 512-token partitions it specifies.  One
more case runs the fp8 workload with the zeroing and the write as separate
calls and the longest sequence as the bound.

Per case:
 - both caches after zeroing and writing equal the oracle's byte for byte;
 - sampled output rows (every query head of two sequences, four heads of
   every other sequence) match the fp64 oracle within the tolerance;
 - every output row is finite and the device error word is clear.
"""
import numpy as np
import pytest
import torch

import harness
from paged_kv_cache_48_gb300 import pkv_check
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu

# (id, workload, partition_tokens, fused zeroing + write, host bound)
CASES = [
    ("llama8b_gqa", wl.llama8b_gqa, 0, True, "table"),
    ("prefix_shared", wl.prefix_shared, 0, True, "table"),
    ("long_context", wl.long_context, 0, True, "table"),
    ("long_context_p512", wl.long_context, 512, True, "table"),
    ("fp8_recycle", wl.fp8_recycle, 0, True, "table"),
    ("fp8_recycle_separate_calls", wl.fp8_recycle, 0, False, "longest"),
    ("tiny_mha", wl.tiny_mha, 0, True, "table"),
]


def _pairs(W, rng):
    pairs = []
    full = {0, W.batch - 1}
    for b in range(W.batch):
        heads = range(W.num_heads) if b in full else sorted(
            {0, W.num_heads - 1, W.group_size - 1,
             int(rng.integers(0, W.num_heads))})
        pairs += [(b, h) for h in heads]
    return np.asarray(pairs, dtype=np.int32)


@pytest.mark.parametrize("name,make,pt,fused,bound", CASES, ids=[c[0] for c in CASES])
def test_full_size_parity(name, make, pt, fused, bound):
    W = make()
    if name == "fp8_recycle":
        assert W.fresh_blocks.size == 515   # the recycled blocks, zeroed in the fused launch
    res = harness.run_gpu(W, partition_tokens=pt, want_cache=True, fused=fused,
                          max_seq_len=W.max_blocks * 16 if bound == "table" else None)
    assert res["status"] == 0, res["status"]
    kc, vc = harness.oracle_cache(W)
    assert np.array_equal(res["key"], kc), "key cache differs from the oracle"
    assert np.array_equal(res["value"], vc), "value cache differs from the oracle"
    del res["key"], res["value"]
    out = res["out"]
    assert np.all(np.isfinite(out))
    pairs = _pairs(W, np.random.default_rng(123))
    ref = harness.oracle_out(W, kc, vc, pairs=pairs)
    mask = np.zeros(out.shape[:2], dtype=bool)
    mask[pairs[:, 0], pairs[:, 1]] = True
    harness.assert_close(out, ref, W.kv_dtype, mask=mask)
    assert pkv_check()[0] == 0
    torch.cuda.empty_cache()


def test_prefix_blocks_are_shared_not_copied():
    """The prefix-shared workload holds one copy of each group's 64 prefix
    blocks (refcount 16), and attention leaves both caches untouched."""
    W = wl.prefix_shared()
    groups = W.groups
    assert len(groups) == 16
    for grp in groups:
        assert len(grp["prefix_blocks"]) == 64
        assert all(W.refcount[b] == 16 for b in grp["prefix_blocks"])
        for b in grp["members"]:
            assert list(W.block_tables[b, :64]) == grp["prefix_blocks"]
    private = int(sum(((W.seq_lens - 1024 + 15) // 16)))
    assert int(np.count_nonzero(W.refcount)) == 16 * 64 + private
    G = harness.upload(W)
    harness.gpu_step(W, G)  # zero + write before attention
    torch.cuda.synchronize()
    kb = G.cache.key_cache.view(torch.uint8).clone()
    vb = G.cache.value_cache.view(torch.uint8).clone()
    from paged_kv_cache_48_gb300 import paged_attention_decode
    paged_attention_decode(G.q, G.cache, G.tables, G.seq_lens, W.scale,
                           max_seq_len=W.max_seq_len)
    torch.cuda.synchronize()
    assert torch.equal(G.cache.key_cache.view(torch.uint8), kb)
    assert torch.equal(G.cache.value_cache.view(torch.uint8), vb)
