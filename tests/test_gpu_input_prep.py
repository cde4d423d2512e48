"""GPU step-input preparation from a persistent request state table against
the oracle (bit-exact), and a decode step driven entirely by its outputs."""
import numpy as np
import pytest
import torch

import harness
import oracle
from paged_kv_cache_48_gb300 import (paged_attention_decode, paged_kv_write,
                                     paged_prepare_inputs, pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu
PKV_OK, PKV_ERR_RANGE = 0, 5


def _state(rng, R, MB, ML, max_computed):
    sbt = rng.permutation(R * MB + 100)[:R * MB].astype(np.int32).reshape(R, MB)
    snc = rng.integers(0, max_computed + 1, R).astype(np.int32)
    tok = rng.integers(0, 151000, (R, ML)).astype(np.int32)
    return sbt, snc, tok


def _run(idx, ns, sbt, snc, tok, T):
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = paged_prepare_inputs(c(idx), c(ns), c(sbt), c(snc), c(tok), T)
    # fill untouched outputs the same way as the oracle's wrapper
    return {k: v.cpu().numpy() for k, v in out.items()}


def _defined(idx, ns, R, T):
    """Which outputs the oracle header defines for these inputs: entries
    whose tokens all fit below T (`fits`), of which those with a valid row
    (`valid`), and the token indices such entries own (`written`)."""
    n = np.maximum(ns.astype(np.int64), 0)
    qsl = np.concatenate([[0], np.cumsum(n)])
    fits = qsl[1:] <= T
    valid = fits & (idx >= 0) & (idx < R)
    written = np.zeros(T, bool)
    for b in range(idx.size):
        if fits[b]:
            written[qsl[b]:qsl[b + 1]] = True
    return fits, valid, written


def _compare(gpu, ref, ns, idx, R):
    """Element-wise equality on every output position the oracle defines."""
    T = ref["slot_mapping"].size
    _, valid, written = _defined(idx, ns, R, T)
    assert np.array_equal(gpu["query_start_loc"], ref["query_start_loc"])
    assert np.array_equal(gpu["seq_lens"][valid], ref["seq_lens"][valid])
    assert np.array_equal(gpu["block_tables"][valid], ref["block_tables"][valid])
    assert np.array_equal(gpu["slot_mapping"][written], ref["slot_mapping"][written])
    assert (ref["slot_mapping"][~written] == -7).all()   # the oracle left them alone
    has_row = np.zeros(T, bool)
    qsl = ref["query_start_loc"]
    for b in np.flatnonzero(valid):
        has_row[qsl[b]:qsl[b] + max(ns[b], 0)] = True
    assert np.array_equal(gpu["positions"][has_row], ref["positions"][has_row])
    ok = written & (ref["slot_mapping"] >= 0)
    assert np.array_equal(gpu["input_ids"][ok], ref["input_ids"][ok])
    return written


@pytest.mark.parametrize("kind", ["decode", "mixed", "large"])
def test_prepare_inputs_matches_oracle(kind):
    rng = np.random.default_rng({"decode": 1, "mixed": 2, "large": 3}[kind])
    R, MB, ML = (300, 64, 1024) if kind != "large" else (5000, 16, 256)
    B = {"decode": 64, "mixed": 40, "large": 3000}[kind]
    sbt, snc, tok = _state(rng, R, MB, ML, max_computed=ML - 320 if kind != "large" else 200)
    idx = rng.permutation(R)[:B].astype(np.int32)
    if kind == "decode":
        ns = np.ones(B, np.int32)
    elif kind == "mixed":
        ns = np.where(rng.random(B) < 0.25, rng.integers(2, 300, B), 1).astype(np.int32)
        ns[3] = 0
    else:
        ns = rng.integers(0, 20, B).astype(np.int32)
    T = int(ns.sum())
    gpu = _run(idx, ns, sbt, snc, tok, T)
    assert pkv_check()[0] == PKV_OK
    ref, err = oracle.load().prepare_inputs(idx, ns, sbt, snc, tok, T)
    assert err == 0
    assert _compare(gpu, ref, ns, idx, R).all()   # every token is an output


def test_prepare_inputs_reports_range_errors():
    rng = np.random.default_rng(4)
    sbt, snc, tok = _state(rng, 6, 2, 40, 0)
    snc[:] = [0, 30, 5, 31, 0, 0]
    idx = np.array([0, 9, 1, 3], np.int32)
    ns = np.array([2, 3, 4, 1], np.int32)
    T = int(ns.sum())
    gpu = _run(idx, ns, sbt, snc, tok, T)
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail in (1, 2)
    ref, err = oracle.load().prepare_inputs(idx, ns, sbt, snc, tok, T)
    assert err == 3
    assert list(gpu["slot_mapping"]) == list(ref["slot_mapping"])


def test_decode_step_driven_by_prepared_inputs():
    """State table built from a workload's sequences (rows shuffled, batch
    order different from row order): the prepared slots equal the new
    tokens' slots, and the decode step run on the prepared tables and
    lengths matches the oracle."""
    W = wl.llama8b_gqa(small=True)
    rng = np.random.default_rng(5)
    B, MB = W.batch, W.max_blocks
    R = B + 7
    rows = rng.permutation(R)[:B].astype(np.int32)       # row of sequence b
    sbt = np.full((R, MB), -1, np.int32)
    snc = np.zeros(R, np.int32)
    sbt[rows] = W.block_tables
    snc[rows] = W.seq_lens - 1                            # all but the new token
    tok = rng.integers(0, 151000, (R, MB * 16)).astype(np.int32)
    order = rng.permutation(B)                            # batch order of this step
    idx = rows[order]
    ns = np.ones(B, np.int32)
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    prep = paged_prepare_inputs(c(idx), c(ns), c(sbt), c(snc), c(tok), B)
    assert pkv_check()[0] == PKV_OK
    assert np.array_equal(prep["slot_mapping"].cpu().numpy(), W.step_slots[order])
    G = harness.upload(W)
    paged_kv_write(G.step_k[torch.from_numpy(order).cuda()],
                   G.step_v[torch.from_numpy(order).cuda()],
                   prep["slot_mapping"], G.cache)
    q = G.q[torch.from_numpy(order).cuda()].contiguous()
    out = paged_attention_decode(q, G.cache, prep["block_tables"], prep["seq_lens"],
                                 W.scale, max_seq_len=W.max_seq_len)
    assert pkv_check()[0] == PKV_OK
    kc, vc = harness.oracle_cache(W)
    ref = harness.oracle_out(W, kc, vc)[order]
    harness.assert_close(out.float().cpu().numpy(), ref, W.kv_dtype)


def test_prepare_inputs_negative_and_overflowing_counts():
    """Negative counts schedule nothing; entries whose tokens do not all fit
    below total_tokens write nothing while query_start_loc keeps the prefix
    sum of the clamped counts.  The GPU reports a range error and matches
    the oracle on every output the oracle defines."""
    # the hand-checked batch of the oracle's own pin
    sbt = np.array([[40, 41], [50, 51], [60, 61], [70, 71]], np.int32)
    snc = np.array([3, 0, 10, 5], np.int32)
    tok = np.arange(4 * 40, dtype=np.int32).reshape(4, 40) + 1000
    idx = np.array([2, 0, 1, 3, 1], np.int32)
    ns = np.array([2, -3, 4, 5, 1], np.int32)
    gpu = _run(idx, ns, sbt, snc, tok, 8)
    st, detail = pkv_check()
    assert st == PKV_ERR_RANGE and detail in (1, 3, 4)
    ref, err = oracle.load().prepare_inputs(idx, ns, sbt, snc, tok, 8)
    assert err == 3
    assert _compare(gpu, ref, ns, idx, 4).sum() == 6
    # a larger batch spanning several scan chunks: scattered negative counts
    # and a token buffer that ends inside the batch
    rng = np.random.default_rng(6)
    R, MB, ML = 400, 32, 512
    sbt, snc, tok = _state(rng, R, MB, ML, max_computed=ML - 64)
    B = 2500
    idx = rng.integers(0, R, B).astype(np.int32)
    ns = rng.integers(0, 40, B).astype(np.int32)
    ns[rng.choice(B, 37, replace=False)] = -rng.integers(1, 100, 37)
    T = int(np.maximum(ns, 0).sum() * 0.6)
    gpu = _run(idx, ns, sbt, snc, tok, T)
    assert pkv_check()[0] == PKV_ERR_RANGE
    ref, err = oracle.load().prepare_inputs(idx, ns, sbt, snc, tok, T)
    fits, _, _ = _defined(idx, ns, R, T)
    assert err == 37 + int((~fits).sum())
    written = _compare(gpu, ref, ns, idx, R)
    assert 0 < written.sum() <= T
