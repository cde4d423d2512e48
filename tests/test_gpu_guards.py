"""Guard regions: no entry point writes outside the memory it is given.

Each output (and the decode workspace past its declared size) is a window
into a larger buffer whose other bytes hold 0xA5; after the call those
bytes must be unchanged.  Rows of q that no sequence owns must not be
written by prefill either.
"""
import numpy as np
import pytest
import torch

import harness
from paged_kv_cache_48_gb300 import (paged_attention_cascade_workspace_bytes,
                                     paged_attention_decode,
                                     paged_attention_decode_cascade,
                                     paged_attention_prefill,
                                     paged_attention_workspace_bytes,
                                     paged_kv_swap_out, paged_prepare_inputs,
                                     pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu
CANARY = 0xA5


def _guarded(shape, dtype, pad_rows=2):
    """A buffer with pad_rows guard rows on each side of the window."""
    rows = shape[0] + 2 * pad_rows
    buf = torch.empty((rows,) + tuple(shape[1:]), dtype=dtype, device="cuda")
    buf.view(torch.uint8).fill_(CANARY)
    return buf, buf[pad_rows:pad_rows + shape[0]]


def _guards_intact(buf, pad_rows=2):
    b = buf.view(torch.uint8).reshape(buf.shape[0], -1)
    return bool((b[:pad_rows] == CANARY).all()) and bool((b[-pad_rows:] == CANARY).all())


@pytest.mark.parametrize("pt", [0, 64])
def test_decode_output_and_workspace_guards(pt):
    W = wl.llama8b_gqa(small=True)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    buf, out = _guarded(tuple(G.q.shape), torch.bfloat16)
    need = paged_attention_workspace_bytes(W.batch, W.num_heads, W.num_kv_heads,
                                           W.head_dim, W.max_seq_len, pt)
    ws = torch.full((need + 4096,), CANARY, dtype=torch.uint8, device="cuda")
    paged_attention_decode(G.q, G.cache, G.tables, G.seq_lens, W.scale,
                           W.max_seq_len, out=out, partition_tokens=pt,
                           workspace=ws)
    assert pkv_check()[0] == 0
    assert _guards_intact(buf)
    assert bool((ws[need:] == CANARY).all())
    kc, vc = harness.oracle_cache(W)
    harness.assert_close(out.float().cpu().numpy(), harness.oracle_out(W, kc, vc), "bf16")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_prefill_output_guards_and_unowned_rows(kv_dtype):
    """q carries 37 rows after the last sequence's chunk that no sequence
    owns: their output rows, and the guard rows around out, stay 0xA5."""
    W = wl.make_prefill_workload("guard", [100, 0], [77, 130], 32, 8, 128, seed=3,
                                 kv_dtype=kv_dtype)
    G = harness.upload_prefill(W)
    harness.gpu_prefill_step(W, G)
    T = W.num_tokens
    extra = torch.randn((37,) + tuple(G.q.shape[1:]), device="cuda").to(torch.bfloat16)
    q = torch.cat([G.q, extra])
    buf, out = _guarded(tuple(q.shape), torch.bfloat16)
    paged_attention_prefill(q, G.cache, G.tables, G.seq_lens, G.qsl, W.scale,
                            W.max_query_len, out=out)
    assert pkv_check()[0] == 0
    assert _guards_intact(buf)
    assert bool((out[T:].view(torch.uint8) == CANARY).all())
    kc, vc = harness.oracle_prefill_cache(W)
    harness.assert_close(out[:T].float().cpu().numpy(),
                         harness.oracle_prefill_out(W, kc, vc), kv_dtype)


def test_cascade_output_and_workspace_guards():
    W = wl.prefix_shared(small=True)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    per = len(W.groups[0]["members"])
    gs = torch.tensor([g["members"][0] for g in W.groups] + [W.batch],
                      dtype=torch.int32, device="cuda")
    plen_h = [16 * len(g["prefix_blocks"]) for g in W.groups]
    plen = torch.tensor(plen_h, dtype=torch.int32, device="cuda")
    need = paged_attention_cascade_workspace_bytes(
        W.batch, W.num_heads, W.num_kv_heads, W.head_dim, W.max_seq_len, max(plen_h), 0)
    ws = torch.full((need + 4096,), CANARY, dtype=torch.uint8, device="cuda")
    buf, out = _guarded(tuple(G.q.shape), torch.bfloat16)
    paged_attention_decode_cascade(G.q, G.cache, G.tables, G.seq_lens, gs, plen,
                                   W.scale, W.max_seq_len, per, max(plen_h),
                                   out=out, workspace=ws)
    assert pkv_check()[0] == 0
    assert _guards_intact(buf)
    assert bool((ws[need:] == CANARY).all())


def test_input_prep_output_guards():
    rng = np.random.default_rng(12)
    R, MB, ML, B = 30, 8, 128, 9
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    sbt = c(rng.permutation(R * MB).astype(np.int32).reshape(R, MB))
    snc = c(rng.integers(0, 60, R).astype(np.int32))
    tok = c(rng.integers(0, 1000, (R, ML)).astype(np.int32))
    idx = c(rng.permutation(R)[:B].astype(np.int32))
    ns = c(rng.integers(0, 6, B).astype(np.int32))
    T = int(ns.sum())
    guards = {}
    outs = {}
    for k, (shape, dt) in {"block_tables": ((B, MB), torch.int32),
                           "seq_lens": ((B,), torch.int32),
                           "query_start_loc": ((B + 1,), torch.int32),
                           "positions": ((T,), torch.int32),
                           "input_ids": ((T,), torch.int32),
                           "slot_mapping": ((T,), torch.int64)}.items():
        guards[k], outs[k] = _guarded(shape, dt)
    paged_prepare_inputs(idx, ns, sbt, snc, tok, T, out=outs)
    assert pkv_check()[0] == 0
    for k, buf in guards.items():
        assert _guards_intact(buf), k


def test_swap_out_host_guard():
    W = wl.llama8b_gqa(small=True)
    G = harness.upload(W)
    bb = W.block_bytes
    ids = np.array([3, 1, 7], np.int32)
    host_k = torch.full((5 * bb,), CANARY, dtype=torch.uint8).pin_memory()
    host_v = torch.full((5 * bb,), CANARY, dtype=torch.uint8).pin_memory()
    paged_kv_swap_out(G.cache, ids, host_k[bb:4 * bb], host_v[bb:4 * bb])
    assert pkv_check()[0] == 0
    for h in (host_k, host_v):
        assert bool((h[:bb] == CANARY).all()) and bool((h[4 * bb:] == CANARY).all())
