"""CUDA decode attention against the fp64 oracle on the same seeded inputs.

Small variants of the five workloads span several blocks, several
partitions and a ragged last block; the oracle computes every output.
Bitwise properties (determinism, placement independence, split with one
partition == no split, one key == its V row) need no oracle.
"""
import numpy as np
import pytest
import torch

import harness
from paged_kv_cache_48_gb300 import (paged_attention_decode,
                                     paged_attention_partition_tokens,
                                     paged_kv_zero_blocks, pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu
PKV_OK, PKV_ERR_RANGE, PKV_ERR_TIMEOUT = 0, 5, 6

SMALL = {
    "tiny": wl.tiny_mha,
    "llama_small": lambda: wl.llama8b_gqa(small=True),
    "prefix_small": lambda: wl.prefix_shared(small=True),
    "long_small": lambda: wl.long_context(small=True),
    "fp8_small": lambda: wl.fp8_recycle(small=True),
    "gqa16_d64": lambda: wl.make_workload("gqa16_d64", 3, 32, 2, 64, 1, 200, 31),
    "fp8_d64": lambda: wl.make_workload("fp8_d64", 3, 12, 4, 64, 2, 150, 32,
                                        kv_dtype="fp8_e4m3",
                                        fresh_policy="recycle515"),
    "mha_d128": lambda: wl.make_workload("mha_d128", 5, 4, 4, 128, 1, 90, 33),
    # many items per warp under the balanced schedule
    "many_mid": lambda: wl.make_workload("many_mid", 512, 8, 2, 128, 16, 200, 34),
    # empty sequences first, in the middle and last (cursor skips them)
    "gaps": lambda: wl.make_workload("gaps", 7, 8, 2, 128, 0, 0, 35,
                                     seq_lens=[0, 300, 0, 0, 45, 1, 0]),
}

_cache = {}


def _case(name):
    if name not in _cache:
        W = SMALL[name]()
        kc, vc = harness.oracle_cache(W)
        _cache[name] = (W, harness.oracle_out(W, kc, vc))
    return _cache[name]


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("partition_tokens", [0, 16, 64, 512])
def test_matches_oracle(name, partition_tokens):
    W, ref = _case(name)
    res = harness.run_gpu(W, partition_tokens=partition_tokens, want_cache=False)
    assert res["status"] == PKV_OK, res
    harness.assert_close(res["out"], ref, W.kv_dtype)


@pytest.mark.parametrize("name", ["tiny", "fp8_small", "long_small"])
def test_stale_bits_without_zeroing_still_match(name):
    """Negative control: skip the zeroing.  Stale fp32 patterns (NaN/Inf)
    stay in the unwritten tail slots of fresh blocks, and the output must
    not change, because positions past seq_len are selected out."""
    W, ref = _case(name)
    res = harness.run_gpu(W, skip_zero=True, want_cache=False)
    assert res["status"] == PKV_OK
    harness.assert_close(res["out"], ref, W.kv_dtype)


def test_deterministic_and_split_equivalence():
    W, _ = _case("long_small")
    G = harness.upload(W)
    a = harness.gpu_step(W, G).clone()
    b = harness.gpu_step(W, G).clone()
    assert torch.equal(a, b)
    e = harness.gpu_step(W, G, partition_tokens=512).clone()
    f = harness.gpu_step(W, G, partition_tokens=512).clone()
    assert torch.equal(e, f)
    whole = ((W.max_seq_len + 15) // 16) * 16
    c = harness.gpu_step(W, G, partition_tokens=whole).clone()
    d = harness.gpu_step(W, G, partition_tokens=whole + 16).clone()
    assert torch.equal(c, d)  # one partition either way: same kernel path
    assert pkv_check()[0] == PKV_OK


def _relocate(W, rng):
    """Same logical content, blocks moved to other physical slots."""
    perm = rng.permutation(W.num_blocks).astype(np.int64)
    bb = W.block_bytes
    W2 = wl.Workload(**{**W.__dict__})
    W2.block_tables = np.where(W.block_tables >= 0,
                               perm[np.maximum(W.block_tables, 0)], -1
                               ).astype(np.int32)
    remap = lambda s: (perm[s // 16] * 16 + s % 16).astype(np.int64)
    W2.hist_slots = remap(W.hist_slots)
    W2.step_slots = remap(W.step_slots)
    W2.fresh_blocks = perm[W.fresh_blocks].astype(np.int32)
    for src, name in ((W.init_key, "init_key"), (W.init_value, "init_value")):
        dst = np.empty_like(src)
        dst.reshape(W.num_blocks, bb)[perm] = src.reshape(W.num_blocks, bb)
        setattr(W2, name, dst)
    return W2


@pytest.mark.parametrize("name", ["llama_small", "fp8_small", "prefix_small"])
@pytest.mark.parametrize("partition_tokens", [0, 64])
def test_block_placement_does_not_change_bits(name, partition_tokens):
    W, _ = _case(name)
    W2 = _relocate(W, np.random.default_rng(9))
    a = harness.run_gpu(W, partition_tokens=partition_tokens, want_cache=False)["out"]
    b = harness.run_gpu(W2, partition_tokens=partition_tokens, want_cache=False)["out"]
    assert np.array_equal(a, b)


def test_single_key_returns_its_value_exactly():
    W = wl.make_workload("one_key", 6, 16, 4, 128, 1, 1, 7)
    res = harness.run_gpu(W, want_cache=False)
    assert res["status"] == PKV_OK
    v = wl.bf16_values(W.step_v)  # the one token of each sequence
    for b in range(W.batch):
        for h in range(W.num_heads):
            assert np.array_equal(res["out"][b, h], v[b, h // 4])


@pytest.mark.parametrize("partition_tokens", [0, 16])
def test_empty_sequence_gives_zeros_and_others_unaffected(partition_tokens):
    W = wl.make_workload("with_empty", 4, 8, 2, 128, 0, 0, 8,
                         seq_lens=[0, 40, 0, 17])
    kc, vc = harness.oracle_cache(W)
    ref = harness.oracle_out(W, kc, vc)
    res = harness.run_gpu(W, partition_tokens=partition_tokens, want_cache=False)
    assert res["status"] == PKV_OK
    assert np.array_equal(res["out"][[0, 2]], np.zeros_like(res["out"][[0, 2]]))
    harness.assert_close(res["out"], ref, "bf16")


def test_bad_block_id_is_reported_not_faulted():
    W, _ = _case("tiny")
    G = harness.upload(W)
    tables = G.tables.clone()
    tables[3, 1] = W.num_blocks + 100
    paged_attention_decode(G.q, G.cache, tables, G.seq_lens, W.scale,
                           max_seq_len=W.max_seq_len)
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail == 3
    assert pkv_check()[0] == PKV_OK


@pytest.mark.parametrize("partition_tokens", [0, 64])
def test_fp8_bad_block_inside_a_pair_is_masked(partition_tokens):
    """E4M3 decode takes blocks two at a time: a bad block id inside a pair
    is reported, contributes nothing, and leaves every other sequence equal
    to the oracle."""
    W, ref = _case("fp8_small")
    b = int(np.argmax(W.seq_lens))
    assert W.seq_lens[b] > 6 * 16
    G = harness.upload(W)
    harness.gpu_step(W, G)
    tables = G.tables.clone()
    tables[b, 5] = W.num_blocks + 7
    out = paged_attention_decode(G.q, G.cache, tables, G.seq_lens, W.scale,
                                 max_seq_len=W.max_seq_len,
                                 partition_tokens=partition_tokens)
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail == b
    got = out.float().cpu().numpy()
    keep = [i for i in range(W.batch) if i != b]
    harness.assert_close(got[keep], ref[keep], "fp8_e4m3")
    assert np.isfinite(got[b]).all()


def test_seq_len_beyond_bound_is_reported():
    W, _ = _case("tiny")
    G = harness.upload(W)
    lens = G.seq_lens.clone()
    lens[1] = W.max_blocks * 16 + 50
    paged_attention_decode(G.q, G.cache, G.tables, lens, W.scale,
                           max_seq_len=W.max_seq_len)
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail == 1


def test_auto_partition_choice_is_reported():
    auto = paged_attention_partition_tokens(64, 32, 8, 4096, 0)
    assert auto > 0 and auto % 256 == 0
    assert paged_attention_partition_tokens(8, 64, 8, 131072, 512) == 512
    assert paged_attention_partition_tokens(8, 64, 8, 131072, 17) == -1


@pytest.mark.parametrize("decode_first", [True, False])
def test_check_reports_the_earliest_error_across_kernels(decode_first):
    """Two range errors recorded by different kernels (decode attention and
    block zeroing) in a known stream order: pkv_check reports the earlier
    one, then everything is cleared."""
    W, _ = _case("tiny")
    G = harness.upload(W)
    tables = G.tables.clone()
    tables[3, 1] = W.num_blocks + 100                    # decode: detail 3
    bad_ids = np.array([1, 2, 4, 5, W.num_blocks + 7], np.int32)   # zeroing: detail 4

    def decode():
        paged_attention_decode(G.q, G.cache, tables, G.seq_lens, W.scale,
                               max_seq_len=W.max_seq_len)

    def zero():
        paged_kv_zero_blocks(G.cache, bad_ids)

    first, second = (decode, zero) if decode_first else (zero, decode)
    first()
    torch.cuda.synchronize()
    torch.cuda._sleep(20000)   # a gap of GPU time between the two records
    second()
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail == (3 if decode_first else 4)
    assert pkv_check()[0] == PKV_OK


@pytest.mark.parametrize("name,partition_tokens", [
    ("llama_small", 0), ("llama_small", 64), ("fp8_small", 0), ("fp8_small", 32)])
def test_timeout_path_reports_and_spares_other_sequences(name, partition_tokens):
    """The bounded-wait failure path, reached through the test hook (every
    warp on one sequence gives up after its first block as if its wait had
    run out; no wait is shortened): pkv_check reports PKV_ERR_TIMEOUT with
    that sequence, its row stays finite, every other sequence still matches
    the oracle, and with the hook off the next call is clean again."""
    from paged_kv_cache_48_gb300 import _native
    W, ref = _case(name)
    victim = int(np.argmax(W.seq_lens))          # long enough to have a second block
    assert W.seq_lens[victim] > 16 * 8
    _native.lib().pkv_testing_fail_decode_sequence(victim)
    try:
        res = harness.run_gpu(W, partition_tokens=partition_tokens, want_cache=False)
    finally:
        _native.lib().pkv_testing_fail_decode_sequence(-1)
    assert res["status"] == PKV_ERR_TIMEOUT and res["detail"] == victim
    assert np.all(np.isfinite(res["out"]))
    others = np.ones(W.batch, bool)
    others[victim] = False
    harness.assert_close(res["out"][others], ref[others], W.kv_dtype)
    again = harness.run_gpu(W, partition_tokens=partition_tokens, want_cache=False)
    assert again["status"] == PKV_OK
    harness.assert_close(again["out"], ref, W.kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_thousands_of_partitions_per_row(kv_dtype):
    """16-token partitions over sequences of up to 40,000 tokens: one warp
    per 16-token partition and more than 2048 partials in a row, so the
    one-CTA-per-row merge walks its weights in several chunks.  Matches
    the oracle on every row; bitwise equal on a second run."""
    W = wl.make_workload(f"many_parts_{kv_dtype}", 3, 8, 2, 128, 0, 0, 36,
                         kv_dtype=kv_dtype, seq_lens=[40000, 33000, 17],
                         fresh_policy="recycle515" if kv_dtype != "bf16" else "new_token")
    assert (W.seq_lens.max() + 15) // 16 > 2048
    kc, vc = harness.oracle_cache(W)
    ref = harness.oracle_out(W, kc, vc)
    res = harness.run_gpu(W, partition_tokens=16, want_cache=False)
    assert res["status"] == PKV_OK, res
    harness.assert_close(res["out"], ref, W.kv_dtype)
    again = harness.run_gpu(W, partition_tokens=16, want_cache=False)
    assert np.array_equal(res["out"], again["out"])
