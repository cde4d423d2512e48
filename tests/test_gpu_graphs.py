"""Every entry point inside a captured CUDA graph gives, on replay, exactly
the eager result.

A serving step runner captures its step once and replays it; the library's
launches (programmatic dependent launch, launch parameters carrying host
ids, the cascade path's decode pass running beside its prefix pass) must
survive capture.  Each case runs eagerly, then is captured on a side stream and
replayed twice; outputs must be bitwise equal and pkv_check clean.
"""
import numpy as np
import pytest
import torch

import harness
from paged_kv_cache_48_gb300 import (paged_attention_decode,
                                     paged_attention_decode_cascade,
                                     paged_attention_decode_step,
                                     paged_attention_prefill,
                                     paged_prepare_inputs, pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _capture(fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def _replay_matches(fn, out):
    fn()
    torch.cuda.synchronize()
    eager = out.clone()
    out.fill_(0)
    g = _capture(fn)
    for _ in range(2):
        out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert pkv_check()[0] == 0
    return eager


def test_decode_step_in_graph():
    W = wl.llama8b_gqa(small=True)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    out = torch.empty_like(G.q)
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    _replay_matches(lambda: paged_attention_decode(
        G.q, G.cache, G.tables, G.seq_lens, W.scale, W.max_seq_len, out=out,
        partition_tokens=64, workspace=ws), out)


@pytest.mark.parametrize("pt", [0, 64])
def test_one_call_decode_step_in_graph(pt):
    """paged_attention_decode_step (the new tokens written by the decode
    kernel) replayed from a graph: the same output, and the cache keeps the
    oracle's bytes (the replays rewrite the same tokens)."""
    W = wl.llama8b_gqa(small=True)
    G = harness.upload(W)
    slots = W.step_slots.tolist()
    rows = [slots.index(int(W.block_tables[b, (L - 1) // 16]) * 16 + (L - 1) % 16)
            for b, L in enumerate(W.seq_lens.tolist())]
    idx = torch.tensor(rows, device="cuda")
    kn, vn = G.step_k[idx].contiguous(), G.step_v[idx].contiguous()
    out = torch.empty_like(G.q)
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    _replay_matches(lambda: paged_attention_decode_step(
        G.q, kn, vn, G.cache, G.tables, G.seq_lens, W.scale, W.max_seq_len, out=out,
        partition_tokens=pt, workspace=ws), out)
    kc, vc = harness.oracle_cache(W)
    assert np.array_equal(G.cache.key_cache.view(torch.uint8).cpu().numpy().reshape(-1),
                          kc.view(np.uint8).reshape(-1))
    assert np.array_equal(G.cache.value_cache.view(torch.uint8).cpu().numpy().reshape(-1),
                          vc.view(np.uint8).reshape(-1))


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_prefill_in_graph(kv_dtype):
    W = wl.chunked_prefill_8k(small=True, kv_dtype=kv_dtype)
    G = harness.upload_prefill(W)
    harness.gpu_prefill_step(W, G)
    out = torch.empty_like(G.q)
    eager = _replay_matches(lambda: paged_attention_prefill(
        G.q, G.cache, G.tables, G.seq_lens, G.qsl, W.scale, W.max_query_len,
        out=out), out)
    kc, vc = harness.oracle_prefill_cache(W)
    harness.assert_close(eager.float().cpu().numpy(),
                         harness.oracle_prefill_out(W, kc, vc), kv_dtype)


def test_cascade_decode_in_graph():
    W = wl.prefix_shared(small=True)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    per = len(W.groups[0]["members"])
    gs = torch.tensor([g["members"][0] for g in W.groups] + [W.batch],
                      dtype=torch.int32, device="cuda")
    plen_h = [16 * len(g["prefix_blocks"]) for g in W.groups]
    plen = torch.tensor(plen_h, dtype=torch.int32, device="cuda")
    out = torch.empty_like(G.q)
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    eager = _replay_matches(lambda: paged_attention_decode_cascade(
        G.q, G.cache, G.tables, G.seq_lens, gs, plen, W.scale, W.max_seq_len,
        per, max(plen_h), out=out, workspace=ws), out)
    kc, vc = harness.oracle_cache(W)
    harness.assert_close(eager.float().cpu().numpy(),
                         harness.oracle_out(W, kc, vc), "bf16")


def test_input_prep_in_graph():
    rng = np.random.default_rng(8)
    R, MB, ML, B = 40, 16, 256, 12
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    sbt = c(rng.permutation(R * MB).astype(np.int32).reshape(R, MB))
    snc = c(rng.integers(0, 100, R).astype(np.int32))
    tok = c(rng.integers(0, 1000, (R, ML)).astype(np.int32))
    idx = c(rng.permutation(R)[:B].astype(np.int32))
    ns = c(rng.integers(1, 9, B).astype(np.int32))
    T = int(ns.sum())
    outs = paged_prepare_inputs(idx, ns, sbt, snc, tok, T)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in outs.items()}
    g = _capture(lambda: paged_prepare_inputs(idx, ns, sbt, snc, tok, T, out=outs))
    for v in outs.values():
        v.fill_(-3)
    g.replay()
    torch.cuda.synchronize()
    for k in eager:
        assert torch.equal(outs[k], eager[k]), k
    assert pkv_check()[0] == 0
