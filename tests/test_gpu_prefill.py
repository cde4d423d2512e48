"""Chunked-prefill attention on the tcgen05 path against the fp64 oracle.

Every case writes the history and then the chunk's K/V through
paged_kv_write into a pool whose unwritten bytes are 0xFF (bf16 NaN), runs
paged_attention_prefill and compares every row with the oracle on the same
seeded inputs (|gpu - ref| <= 1e-2 + 1e-2 |ref|).  Shapes span several
128-key tiles, several query tiles, ragged tails, one-token chunks, empty
chunks and group sizes 1, 4, 5 and 8, for bf16 and E4M3 caches (fp8 bound
3e-2 + 3e-2 |ref|).
"""
import numpy as np
import pytest
import torch

import harness
import oracle
from paged_kv_cache_48_gb300 import (paged_attention_decode,
                                     paged_attention_prefill, pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu
PKV_OK, PKV_ERR_RANGE = 0, 5

CASES = {
    # name: (history, chunk, Hq, Hkv, d)
    "mha_d64": ([0, 5, 40, 100], [150, 11, 1, 64], 8, 8, 64),
    "gqa4_chunks": ([569, 393, 426, 543], [200, 37, 1, 130], 32, 8, 128),
    "gqa4_prompts": ([0, 0, 0], [300, 129, 17], 32, 8, 128),
    "gqa5": ([0, 200, 333], [77, 130, 26], 40, 8, 128),
    "gqa8_long": ([1500, 0], [40, 257], 64, 8, 128),
    "tile_edges": ([0, 128, 0, 112], [128, 128, 256, 16], 32, 8, 128),
    "with_empty": ([10, 0, 64], [0, 33, 0], 32, 8, 64),
}


def _run_case(W):
    G = harness.upload_prefill(W)
    out = harness.gpu_prefill_step(W, G)
    st, detail = pkv_check()
    assert st == PKV_OK, (st, detail)
    return out.float().cpu().numpy(), G


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(name, kv_dtype):
    hist, chunk, Hq, Hkv, d = CASES[name]
    W = wl.make_prefill_workload(name, hist, chunk, Hq, Hkv, d, seed=len(name),
                                 kv_dtype=kv_dtype)
    gpu, _ = _run_case(W)
    kc, vc = harness.oracle_prefill_cache(W)
    ref = harness.oracle_prefill_out(W, kc, vc)
    harness.assert_close(gpu, ref, kv_dtype)


@pytest.mark.parametrize("cfg", ["prefill_8k", "chunked_prefill_8k"])
def test_prefill_small_configs(cfg):
    W = wl.PREFILL_CONFIGS[cfg](small=True)
    gpu, _ = _run_case(W)
    kc, vc = harness.oracle_prefill_cache(W)
    harness.assert_close(gpu, harness.oracle_prefill_out(W, kc, vc), "bf16")


def test_prefill_is_deterministic_and_chunking_invariant():
    """Two runs are bitwise equal, and a 300-token prompt computed as one
    chunk or as chunks of 200 + 100 gives bitwise-equal rows (each row's
    arithmetic depends only on its own query and the fixed key tiles)."""
    W = wl.make_prefill_workload("one", [0], [300], 32, 8, 128, seed=9)
    a, G = _run_case(W)
    b = paged_attention_prefill(G.q, G.cache, G.tables, G.seq_lens, G.qsl,
                                W.scale, W.max_query_len).float().cpu().numpy()
    assert np.array_equal(a, b)
    # same cache, same queries, the prompt cut in two steps
    qsl1 = torch.tensor([0, 200], dtype=torch.int32, device="cuda")
    qsl2 = torch.tensor([0, 100], dtype=torch.int32, device="cuda")
    o1 = paged_attention_prefill(G.q[:200].contiguous(), G.cache, G.tables,
                                 torch.tensor([200], dtype=torch.int32, device="cuda"),
                                 qsl1, W.scale, 200)
    o2 = paged_attention_prefill(G.q[200:].contiguous(), G.cache, G.tables,
                                 torch.tensor([300], dtype=torch.int32, device="cuda"),
                                 qsl2, W.scale, 100)
    assert pkv_check()[0] == PKV_OK
    assert np.array_equal(torch.cat([o1, o2]).float().cpu().numpy(), a)


def test_prefill_one_token_chunks_match_decode():
    """Chunks of one token are decode steps: both kernels match the oracle
    on the same cache."""
    W = wl.make_prefill_workload("dec", [17, 300, 1023, 0], [1, 1, 1, 1], 32, 8,
                                 128, seed=3)
    gpu, G = _run_case(W)
    dec = paged_attention_decode(G.q, G.cache, G.tables, G.seq_lens, W.scale,
                                 max_seq_len=int(W.seq_lens.max()))
    assert pkv_check()[0] == PKV_OK
    kc, vc = harness.oracle_prefill_cache(W)
    ref = harness.oracle_prefill_out(W, kc, vc)
    harness.assert_close(gpu, ref, "bf16")
    harness.assert_close(dec.float().cpu().numpy(), ref, "bf16")


def test_prefill_bad_block_id_is_reported_and_rows_zeroed():
    W = wl.make_prefill_workload("bad", [40, 0], [20, 30], 32, 8, 128, seed=4)
    G = harness.upload_prefill(W)
    harness.gpu_prefill_step(W, G)
    assert pkv_check()[0] == PKV_OK
    tables = W.block_tables.copy()
    tables[1, 1] = W.num_blocks + 3
    out = torch.full_like(G.q, 7.0)
    paged_attention_prefill(G.q, G.cache, torch.from_numpy(tables).cuda(),
                            G.seq_lens, G.qsl, W.scale, W.max_query_len, out=out)
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail == 1 * W.max_blocks + 1
    o = out.float().cpu().numpy()
    assert np.all(o[20:] == 0.0)
    kc, vc = harness.oracle_prefill_cache(W)
    ref = harness.oracle_prefill_out(W, kc, vc)
    harness.assert_close(o[:20], ref[:20], "bf16")


def test_prefill_fp8_is_deterministic_and_matches_oracle():
    """fp8 KV (g = 5): two runs are bitwise equal, and the f16 tensor-core
    path (E4M3 tiles converted to f16 in shared memory) agrees with the
    oracle on the same cache bytes (|err| <= 3e-2 + 3e-2 |ref|)."""
    W = wl.make_prefill_workload("f8", [300, 0], [200, 150], 40, 8, 128, seed=12,
                                 kv_dtype="fp8_e4m3")
    a, G = _run_case(W)
    b = paged_attention_prefill(G.q, G.cache, G.tables, G.seq_lens, G.qsl,
                                W.scale, W.max_query_len).float().cpu().numpy()
    assert np.array_equal(a, b)
    kc, vc = harness.oracle_prefill_cache(W)
    harness.assert_close(a, harness.oracle_prefill_out(W, kc, vc), "fp8_e4m3")


@pytest.mark.parametrize("make,kv_dtype", [
    (wl.chunked_prefill_8k, "bf16"), (wl.chunked_prefill_8k, "fp8_e4m3"),
    (wl.prefill_8k, "bf16"), (wl.prefill_8k, "fp8_e4m3")],
    ids=["chunked_bf16", "chunked_fp8", "prompts_bf16", "prompts_fp8"])
def test_prefill_full_size_sampled_rows(make, kv_dtype):
    """The full 8K-token prefill steps (8 chunks of 1024 tokens after a
    history, and 8 fresh 1024-token prompts) in the bench's launch
    configuration; rows sampled across every sequence (first, last and
    seeded random tokens, heads from several groups) against the oracle."""
    W = make(kv_dtype=kv_dtype)
    gpu, _ = _run_case(W)
    rng = np.random.default_rng(0)
    qsl = W.query_start_loc
    toks = set()
    for b in range(W.batch):
        toks.update([int(qsl[b]), int(qsl[b + 1]) - 1])
        toks.update(int(t) for t in rng.integers(qsl[b], qsl[b + 1], 3))
    rows = np.array([[t, h] for t in sorted(toks) for h in (0, 5, 17, 31)],
                    np.int32)
    kc, vc = harness.oracle_prefill_cache(W)
    ref = harness.oracle_prefill_out(W, kc, vc, rows=rows)
    harness.assert_close(gpu[rows[:, 0], rows[:, 1]], ref[rows[:, 0], rows[:, 1]],
                         kv_dtype)


def _sweep_cases(n=12, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        g = int(rng.choice([1, 2, 4, 5, 8]))
        Hkv = int(rng.choice([1, 2, 8])) if g < 8 else int(rng.choice([1, 4]))
        d = int(rng.choice([64, 128]))
        B = int(rng.integers(1, 6))
        hist = [int(x) for x in rng.integers(0, 700, B) * (rng.random(B) < 0.7)]
        chunk = [int(x) for x in rng.integers(0, 260, B)]
        if sum(chunk) == 0:
            chunk[0] = 1
        kv = str(rng.choice(["bf16", "fp8_e4m3"]))
        cases.append((i, hist, chunk, g * Hkv, Hkv, d, kv))
    return cases


@pytest.mark.parametrize("case", _sweep_cases(), ids=lambda c: f"sweep{c[0]}")
def test_prefill_random_sweep(case):
    """Seeded random shapes: group sizes 1-8, 1-8 kv heads, head_dim 64 and
    128, both cache dtypes, zero to several hundred tokens of history and
    chunk per sequence."""
    i, hist, chunk, Hq, Hkv, d, kv = case
    W = wl.make_prefill_workload(f"sweep{i}", hist, chunk, Hq, Hkv, d,
                                 seed=100 + i, kv_dtype=kv)
    gpu, _ = _run_case(W)
    kc, vc = harness.oracle_prefill_cache(W)
    harness.assert_close(gpu, harness.oracle_prefill_out(W, kc, vc), kv)


def test_prefill_bad_query_start_loc_is_reported():
    """A chunk longer than its sequence (query_start_loc past seq_len) is a
    device range error; the other sequence is still right."""
    W = wl.make_prefill_workload("badq", [30, 10], [20, 8], 32, 8, 128, seed=5)
    G = harness.upload_prefill(W)
    harness.gpu_prefill_step(W, G)
    assert pkv_check()[0] == PKV_OK
    lens = G.seq_lens.clone()
    lens[1] = 4                                   # shorter than its 8-token chunk
    out = torch.full_like(G.q, 3.0)
    paged_attention_prefill(G.q, G.cache, G.tables, lens, G.qsl, W.scale,
                            W.max_query_len, out=out)
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail == 1
    kc, vc = harness.oracle_prefill_cache(W)
    ref = harness.oracle_prefill_out(W, kc, vc)
    harness.assert_close(out.float().cpu().numpy()[:20], ref[:20], "bf16")
