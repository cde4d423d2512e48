"""Host-side pieces of bench.py, on CPU: the reference arm's JSON line (the
oracle timed on the host cores), the buffer packing of a step's inputs, the
profile lookup that supplies roofline traffic, the host CPU name, and the
choice of the one-call decode step."""
import json
import subprocess
import sys
from pathlib import Path

import numpy as np
import pytest
import torch

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))
import bench  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                        "--workload", "tiny_mha", "--steps", "1", "--warmup", "0",
                        "--cpu-sample-seqs", "4"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["config"]["workload"] == "tiny_mha"
    assert d["higher_is_better"] is True and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["one_core"]["cores"] == 1 and cb["one_core"]["value"] > 0
    assert cb["cpu"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_packed_views_hold_the_tensors_at_aligned_offsets():
    ts = [torch.arange(7, dtype=torch.int32), torch.randn(3, 5).to(torch.bfloat16),
          torch.arange(11, dtype=torch.int64), torch.zeros(0, dtype=torch.int32)]
    buf, views = bench.packed(ts)
    assert buf.dtype == torch.uint8
    for v, t in zip(views, ts):
        assert v.dtype == t.dtype and v.shape == t.shape and torch.equal(v, t)
        if v.numel():  # an empty view may report a null data pointer
            assert (v.data_ptr() - buf.data_ptr()) % 256 == 0
    # the views alias the buffer: a write through one is seen in the other
    views[0][0] = 99
    assert int(buf[:4].view(torch.int32)[0]) == 99


def test_profile_traffic_follows_the_kernel_source_hash(tmp_path):
    sha = bench.kernel_sha(bench.KERNEL_SOURCES)
    good = tmp_path / "good.md"
    good.write_text(f"kernel_source_sha256: {sha}\ndram_bytes_per_launch: 123456\n")
    assert bench.profiled_traffic(good, bench.KERNEL_SOURCES) == 123456.0
    stale = tmp_path / "stale.md"
    stale.write_text("kernel_source_sha256: 0000000000000000\ndram_bytes_per_launch: 1\n")
    assert bench.profiled_traffic(stale, bench.KERNEL_SOURCES) is None
    assert bench.profiled_traffic(tmp_path / "missing.md", bench.KERNEL_SOURCES) is None
    # every committed profile that names a source hash parses
    for p in (ROOT / "profiles").glob("*.md"):
        text = p.read_text()
        if "kernel_source_sha256:" in text:
            assert "dram_bytes_per_launch:" in text, p.name


def test_host_cpu_model_names_the_cores():
    s = bench.host_cpu_model()
    assert isinstance(s, str) and s.endswith("cores")


def test_profile_summaries_name_only_committed_commands():
    """Every ncu summary gives the command that made it, and that command
    runs files of the repository (bench.py), never a scratch script."""
    for p in (ROOT / "profiles").glob("*.md"):
        text = p.read_text()
        assert "ncu " in text and "--clock-control none" in text, p.name
        assert "python bench.py" in text, p.name
        assert "_work" not in text, p.name


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 runs and prints the reference line; the
    other ranks exit 0 at once."""
    env = dict(__import__("os").environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                        "--workload", "tiny_mha", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.strip().startswith("{")]


def test_new_token_tail_layout():
    """Workload.new_token_tail, which bench.py uses to run a step as one
    paged_attention_decode_step call: it applies exactly when every
    sequence's writes are its last positions and the fresh blocks are the
    blocks that open among them, and gives those tokens in sequence and
    position order, delimited per sequence.  The recycled-block workload
    has that layout (its 515 blocks are the sequences' last blocks, every
    valid slot rewritten); a sequence without a write, or a fresh block the
    tail does not open, has not."""
    from paged_kv_cache_48_gb300 import workload as wl
    W = wl.llama8b_gqa(small=True)
    rows, start = W.new_token_tail()
    assert list(start) == list(range(W.batch + 1))
    for b, i in enumerate(rows):
        L = int(W.seq_lens[b])
        assert W.step_slots[i] == W.block_tables[b, (L - 1) // 16] * 16 + (L - 1) % 16
    R = wl.fp8_recycle(small=True)
    rows, start = R.new_token_tail()
    for b in range(R.batch):
        L, n = int(R.seq_lens[b]), int(start[b + 1] - start[b])
        assert n >= 1
        for k, i in enumerate(rows[start[b]:start[b + 1]]):
            t = L - n + k
            assert R.step_slots[i] == R.block_tables[b, t // 16] * 16 + t % 16
    W0 = wl.make_workload("empty", 3, 8, 8, 64, 0, 0, 1, seq_lens=[0, 5, 9])
    assert W0.new_token_tail() is None
    W.fresh_blocks = np.append(W.fresh_blocks, np.int32(W.num_blocks - 1))
    assert W.new_token_tail() is None
