"""Split decode writes per-partition partials into the caller's workspace
and merges them with a log-sum-exp reduce; the library never zeroes the
workspace.  So the result must not depend on what the workspace held before
the call: zeros, fill patterns, random bytes, or what an earlier call with
another layout left there.  Every variant must give bit-for-bit the same
output, and that output must match the fp64 oracle (log-sum-exp merge of the
partitions, the split-KV row of the scope; the pages themselves are silent
on the split)."""
import numpy as np
import pytest
import torch

import harness
from paged_kv_cache_48_gb300 import (paged_attention_decode,
                                     paged_attention_workspace_bytes, pkv_check)
from paged_kv_cache_48_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _decode(W, G, pt, ws):
    out = torch.full_like(G.q, float("nan"))
    paged_attention_decode(G.q, G.cache, G.tables, G.seq_lens, W.scale, W.max_seq_len,
                           out=out, partition_tokens=pt, workspace=ws)
    torch.cuda.synchronize()
    assert pkv_check()[0] == 0
    return out


def _fills(need, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    rnd = torch.randint(0, 256, (need,), dtype=torch.uint8, generator=g).cuda()
    yield "zero", torch.zeros(need, dtype=torch.uint8, device="cuda")
    yield "a5", torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")
    yield "ff", torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    yield "random", rnd


@pytest.mark.parametrize("make,pt", [
    (lambda: wl.llama8b_gqa(small=True), 64),     # up to 9 partitions
    (lambda: wl.llama8b_gqa(small=True), 16),     # up to 36: the > 32 merge path
    (lambda: wl.long_context(small=True), 64),    # g = 8, up to 43 partitions
    (lambda: wl.fp8_recycle(small=True), 32),     # g = 5, E4M3 cache
], ids=["gqa_pt64", "gqa_pt16", "long_pt64", "fp8_pt32"])
def test_result_does_not_depend_on_workspace_contents(make, pt):
    W = make()
    G = harness.upload(W)
    harness.gpu_step(W, G)
    need = paged_attention_workspace_bytes(W.batch, W.num_heads, W.num_kv_heads,
                                           W.head_dim, W.max_seq_len, pt)
    assert need > 0
    first = None
    for name, ws in _fills(need, seed=pt):
        for rep in range(2):  # the second call finds the partials this call left
            got = _decode(W, G, pt, ws)
            if first is None:
                first = got.clone()
                kc, vc = harness.oracle_cache(W)
                harness.assert_close(got.float().cpu().numpy(), harness.oracle_out(W, kc, vc),
                                     W.kv_dtype)
            assert torch.equal(got, first), (name, rep)


def test_workspace_reused_across_layouts():
    """One buffer used by calls of different batch size and partition
    length: each call's partials land at other offsets than the
    previous call's, so every call starts on another call's leftovers."""
    W = wl.llama8b_gqa(small=True)
    G = harness.upload(W)
    harness.gpu_step(W, G)
    kc, vc = harness.oracle_cache(W)
    ref = harness.oracle_out(W, kc, vc)
    big = max(paged_attention_workspace_bytes(W.batch, W.num_heads, W.num_kv_heads,
                                              W.head_dim, W.max_seq_len, pt)
              for pt in (16, 32, 64, 128))
    ws = torch.full((big,), 0x5A, dtype=torch.uint8, device="cuda")
    outs = {}
    for pt in (64, 16, 128, 32, 64, 16):
        got = _decode(W, G, pt, ws)
        harness.assert_close(got.float().cpu().numpy(), ref, "bf16")
        if pt in outs:
            assert torch.equal(got, outs[pt])
        outs[pt] = got.clone()
    # a sub-batch through the same buffer (other row count, other offsets)
    half = W.batch // 2
    out = torch.empty_like(G.q[:half])
    paged_attention_decode(G.q[:half].contiguous(), G.cache, G.tables[:half].contiguous(),
                           G.seq_lens[:half].contiguous(), W.scale, W.max_seq_len, out=out,
                           partition_tokens=16, workspace=ws)
    torch.cuda.synchronize()
    assert pkv_check()[0] == 0
    assert torch.equal(out, outs[16][:half])
