"""Cascade (shared-prefix) decode against the fp64 decode oracle.

Cascade decode must return what plain decode returns: the oracle is the
decode oracle on the same seeded inputs (|gpu - ref| <= 1e-2 + 1e-2 |ref|).
Cases: the prefix-sharing workload (small and full size), groups with
different prefix lengths next to ungrouped sequences and single-member
groups, a member whose table breaks the sharing contract (reported, still
correct), and the split of long suffixes into several partitions.
"""
import numpy as np
import pytest
import torch

import harness
from paged_kv_cache_48_gb300 import (paged_attention_decode,
                                     paged_attention_decode_cascade, pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu
PKV_OK, PKV_ERR_RANGE = 0, 5


def _i32(a):
    return torch.tensor(np.asarray(a, np.int32), device="cuda")


def _cascade(W, G, group_start, prefix_len, tables=None, partition_tokens=0):
    sizes = np.diff(group_start)
    return paged_attention_decode_cascade(
        G.q, G.cache, G.tables if tables is None else tables, G.seq_lens,
        _i32(group_start), _i32(prefix_len), W.scale, max_seq_len=W.max_seq_len,
        max_group_size=int(sizes.max()) if sizes.size else 0,
        max_prefix_len=int(max(prefix_len)) if len(prefix_len) else 0,
        partition_tokens=partition_tokens)


def _groups_of(W):
    per = len(W.groups[0]["members"])
    gs = [grp["members"][0] for grp in W.groups] + [W.groups[-1]["members"][-1] + 1]
    assert all(grp["members"] == list(range(grp["members"][0], grp["members"][0] + per))
               for grp in W.groups)
    plen = [16 * len(grp["prefix_blocks"]) for grp in W.groups]
    return np.array(gs, np.int32), np.array(plen, np.int32)


@pytest.mark.parametrize("pt", [0, 32])
def test_cascade_prefix_shared_small(pt):
    W = wl.prefix_shared(small=True)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    gs, plen = _groups_of(W)
    out = _cascade(W, G, gs, plen, partition_tokens=pt)
    assert pkv_check()[0] == PKV_OK
    kc, vc = harness.oracle_cache(W)
    harness.assert_close(out.float().cpu().numpy(), harness.oracle_out(W, kc, vc), "bf16")


def test_cascade_mixed_groups_and_ungrouped_sequences():
    """Groups of 3, 2 and 1 members with prefixes of 64, 128 and 16 tokens,
    two sequences in no group, on the Llama-8B shape (g = 4)."""
    W = wl.llama8b_gqa(small=True)          # 8 sequences, lengths 20..700
    order = np.argsort(-W.seq_lens)          # longest first: prefixes fit
    for name in ("seq_lens", "block_tables", "q", "step_k", "step_v", "step_slots"):
        setattr(W, name, getattr(W, name)[order].copy())
    tables = W.block_tables.copy()
    gs = np.array([0, 3, 5, 6], np.int32)   # sequences 6, 7 in no group
    plen = np.array([64, 128, 16], np.int32)
    plen = np.minimum(plen, [int(W.seq_lens[gs[i]:gs[i + 1]].min()) // 16 * 16
                             for i in range(3)]).astype(np.int32)
    for gi in range(3):
        lead = gs[gi]
        for m in range(gs[gi] + 1, gs[gi + 1]):
            tables[m, :plen[gi] // 16] = tables[lead, :plen[gi] // 16]
    W.block_tables = tables
    G = harness.upload(W)
    harness.gpu_step(W, G)
    out = _cascade(W, G, gs, plen)
    assert pkv_check()[0] == PKV_OK
    kc, vc = harness.oracle_cache(W)
    harness.assert_close(out.float().cpu().numpy(), harness.oracle_out(W, kc, vc), "bf16")


def test_cascade_contract_violation_is_reported_and_still_correct():
    W = wl.prefix_shared(small=True)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    gs, plen = _groups_of(W)
    # member 2 of group 0 points its first prefix block elsewhere: its own
    # table is the truth for the oracle, the group prefix no longer applies
    bad = W.block_tables.copy()
    bad[2, 0] = W.groups[1]["prefix_blocks"][0]  # written data, another group's
    out = _cascade(W, G, gs, plen, tables=torch.from_numpy(bad).cuda())
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail == 2 * W.max_blocks + 0
    W2 = wl.Workload(**{**W.__dict__})
    W2.block_tables = bad
    kc, vc = harness.oracle_cache(W)
    harness.assert_close(out.float().cpu().numpy(), harness.oracle_out(W2, kc, vc), "bf16")


def test_cascade_full_size_matches_decode_and_oracle_samples():
    """The full prefix-sharing workload (256 sequences in 16 groups sharing
    1024 tokens): cascade and plain decode agree within the tolerance
    everywhere, and sampled rows match the oracle."""
    W = wl.prefix_shared()
    G = harness.upload(W)
    harness.gpu_step(W, G)
    gs, plen = _groups_of(W)
    out = _cascade(W, G, gs, plen).float().cpu().numpy()
    dec = paged_attention_decode(G.q, G.cache, G.tables, G.seq_lens, W.scale,
                                 max_seq_len=W.max_seq_len).float().cpu().numpy()
    assert pkv_check()[0] == PKV_OK
    harness.assert_close(out, dec.astype(np.float64), "bf16")
    rng = np.random.default_rng(1)
    seqs = sorted(set(rng.choice(W.batch, 10, replace=False).tolist()) | {0, 15, 255})
    pairs = np.array([(b, h) for b in seqs for h in range(W.num_heads)], np.int32)
    kc, vc = harness.oracle_cache(W)
    ref = harness.oracle_out(W, kc, vc, pairs=pairs)
    harness.assert_close(out[seqs], ref[seqs], "bf16")


def test_cascade_fp8_cache_matches_oracle():
    """E4M3 cache with per-tensor scales: the prefix pass runs on f16
    operands, the suffix pass in the fp8 decode kernel."""
    W = wl.make_workload("prefix_fp8", 8, 40, 8, 128, 5, 60, 21,
                         kv_dtype="fp8_e4m3", prefix_groups=2, prefix_len=64)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    gs, plen = _groups_of(W)
    out = _cascade(W, G, gs, plen)
    assert pkv_check()[0] == PKV_OK
    kc, vc = harness.oracle_cache(W)
    harness.assert_close(out.float().cpu().numpy(), harness.oracle_out(W, kc, vc),
                         "fp8_e4m3")


def test_cascade_bad_group_falls_back_to_full_attention():
    """A group whose prefix is not a multiple of 16 breaks the contract: it
    is reported, and its members are attended in full (still the oracle's
    result); the other group still uses its shared prefix."""
    W = wl.prefix_shared(small=True)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    gs, plen = _groups_of(W)
    plen = plen.copy()
    plen[1] = 40
    out = _cascade(W, G, gs, np.array(plen, np.int32))
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail in range(int(gs[1]), int(gs[2]))
    kc, vc = harness.oracle_cache(W)
    harness.assert_close(out.float().cpu().numpy(), harness.oracle_out(W, kc, vc), "bf16")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_cascade_long_prefix_in_several_partitions(kv_dtype):
    """Two groups of 4 sharing a 2304-token prefix: 16 (group, kv head)
    units leave most SMs free, so the prefix is cut into several partitions
    (the last one short) whose slots the merge combines."""
    W = wl.make_workload("prefix_long", 8, 32, 8, 128, 5, 200, 23, kv_dtype=kv_dtype,
                         prefix_groups=2, prefix_len=2304)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    gs, plen = _groups_of(W)
    out = _cascade(W, G, gs, plen)
    assert pkv_check()[0] == PKV_OK
    kc, vc = harness.oracle_cache(W)
    harness.assert_close(out.float().cpu().numpy(), harness.oracle_out(W, kc, vc), kv_dtype)


def test_cascade_merge_waits_for_a_prefix_pass_longer_than_a_wave():
    """40 groups of 2 sharing 2048-token prefixes with 1-16 private tokens:
    the prefix pass (320 CTAs, more than one wave) is the long pole and the
    decode pass beside it ends first, so a merge that did not wait for the
    prefix pass would read unwritten slots.  Three calls in a row on one
    stream give bitwise-equal outputs that match the oracle."""
    W = wl.make_workload("prefix_wave", 80, 32, 8, 128, 1, 16, 31,
                         prefix_groups=40, prefix_len=2048)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    gs, plen = _groups_of(W)
    outs = [_cascade(W, G, gs, plen) for _ in range(3)]
    assert pkv_check()[0] == PKV_OK
    first = outs[0].float().cpu().numpy()
    for o in outs[1:]:
        assert np.array_equal(o.float().cpu().numpy(), first)
    kc, vc = harness.oracle_cache(W)
    harness.assert_close(first, harness.oracle_out(W, kc, vc), "bf16")
