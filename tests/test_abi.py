"""The C ABI library builds, loads and exports every declared entry point;
host-side argument checks answer without touching a GPU (no compute)."""
import ctypes

import pytest

from paged_kv_cache_48_gb300 import _native, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _native.declared_functions()
    assert {"paged_kv_write", "paged_kv_zero_blocks", "paged_attention_decode",
            "paged_attention_workspace_bytes", "pkv_check"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert n in _native._SIGNATURES, f"{n} has no binding signature"


def test_status_strings_and_version(lib):
    for code, name in _native.STATUS_NAMES.items():
        s = lib.pkv_status_str(code)
        assert s and s != b"unknown status", name
    assert lib.pkv_status_str(99) == b"unknown status"
    assert lib.pkv_version() >= 100


def _cache(**kw):
    c = _native.PkvCache(16, 16, 4, 16, 2, 128, 0, 1.0, 1.0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value,status", [
    ("key_cache", None, 1),
    ("block_size", 32, 3),
    ("head_dim", 96, 3),
    ("dtype", 7, 2),
    ("num_blocks", 0, 3),
    ("key_cache", 24, 1),      # not 16-byte aligned
])
def test_cache_validation_before_any_cuda_call(lib, field, value, status):
    c = _cache(**{field: value})
    st = lib.paged_kv_write(16, 16, 16, 1, ctypes.byref(c), None)
    assert st == status
    st = lib.paged_kv_zero_blocks(ctypes.byref(c), 16, 1, 1, None)
    assert st == status


def test_argument_validation(lib):
    c = _cache()
    assert lib.paged_kv_write(None, 16, 16, 1, ctypes.byref(c), None) == 1
    assert lib.paged_kv_write(16, 16, 16, -1, ctypes.byref(c), None) == 1
    assert lib.paged_kv_write(16, 16, 16, 0, ctypes.byref(c), None) == 0
    assert lib.paged_kv_zero_blocks(ctypes.byref(c), None, 3, 1, None) == 1
    assert lib.paged_kv_zero_blocks(ctypes.byref(c), None, 0, 1, None) == 0
    # num_heads not a multiple of num_kv_heads
    assert lib.paged_attention_decode(16, ctypes.byref(c), 16, 4, 16, 2, 3,
                                      0.1, 16, 64, 0, None, 0, None) == 3
    # partition length not a multiple of 16
    assert lib.paged_attention_decode(16, ctypes.byref(c), 16, 4, 16, 2, 4,
                                      0.1, 16, 64, 24, None, 0, None) == 1
    # empty batch is a no-op
    assert lib.paged_attention_decode(16, ctypes.byref(c), 16, 4, 16, 0, 4,
                                      0.1, 16, 64, 0, None, 0, None) == 0
    assert lib.paged_attention_partition_tokens(8, 64, 8, 1000, 17) == -1
    # grid limits are checked on the host: batch (grid z) and partitions
    # (grid y) at most 65535
    assert lib.paged_attention_decode(16, ctypes.byref(c), 16, 4, 16, 65536, 4,
                                      0.1, 16, 64, 0, None, 0, None) == 1
    assert lib.paged_attention_decode(16, ctypes.byref(c), 16, 1 << 16, 16, 2, 4,
                                      0.1, 16, 16 * 65536, 16, None, 0, None) == 1


def test_missing_library_fails_loudly():
    """Without the built library every call raises: the package has no CPU
    or PyTorch fallback to take over."""
    import subprocess
    import sys
    code = (
        "from pathlib import Path\n"
        "from paged_kv_cache_48_gb300 import _native\n"
        "_native.LIBRARY = Path('/nonexistent/libpagedkv.so')\n"
        "_native._LIB = None\n"
        "import paged_kv_cache_48_gb300 as pk\n"
        "try:\n"
        "    pk.pkv_check()\n"
        "except RuntimeError as e:\n"
        "    print('raised:', 'missing' in str(e))\n"
    )
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300, cwd=str(_native.PKG.parent))
    assert r.returncode == 0, r.stderr[-2000:]
    assert "raised: True" in r.stdout


def test_cascade_argument_validation(lib):
    """Shared-prefix decode rejects bad arguments on the host, before any
    CUDA call: unaligned prefix bound, non-positive scale, groups wider than
    128 query heads per kv head, too many groups, missing workspace."""
    c = _cache()

    def call(batch=2, num_heads=4, num_groups=1, max_prefix_len=32, scale=0.1,
             workspace=None, workspace_bytes=0, partition_tokens=16):
        return lib.paged_attention_decode_cascade(
            16, ctypes.byref(c), 16, 8, 16, batch, num_heads, 16, 16, num_groups, 2,
            max_prefix_len, scale, 16, 128, partition_tokens, workspace,
            workspace_bytes, None)

    assert call(max_prefix_len=24) == 1
    assert call(scale=0.0) == 1
    assert call(scale=-1.0) == 1
    assert call(num_heads=2 * 130) == 3
    assert call(num_groups=65536) == 1
    assert call() == 7                       # no workspace
    need = lib.paged_attention_cascade_workspace_bytes(2, 4, 2, 128, 128, 32, 16)
    assert need > 0
    assert call(workspace=256, workspace_bytes=need - 1) == 7
    assert call(batch=0) == 0                # empty batch: nothing to do


def test_decode_step_argument_validation(lib):
    """The decode step rejects a missing or unaligned new-token buffer and a
    row count that does not match on the host, before any CUDA call, and
    treats an empty batch as a no-op."""
    c = _cache()

    def call(k=16, v=16, batch=2, nsl=None, n_new=2):
        return lib.paged_attention_decode_step(16, k, v, nsl, n_new, ctypes.byref(c), 16, 8, 16,
                                               batch, 4, 0.1, 16, 128, 0, None, 0, None)

    assert call(k=None) == 1
    assert call(v=None) == 1
    assert call(k=24) == 1
    assert call(v=8) == 1
    assert call(n_new=3) == 1              # one row per sequence without new_start_loc
    assert call(nsl=16, n_new=-1) == 1
    assert call(nsl=16, n_new=5, k=24) == 1
    assert call(batch=0, n_new=0) == 0


def test_prefill_argument_validation(lib):
    """Chunked prefill rejects bad arguments on the host, before any CUDA
    call, and treats an empty step as a no-op."""
    c = _cache()

    def call(batch=2, num_heads=4, num_tokens=10, scale=0.1, max_query_len=8, q=16,
             cache=c):
        return lib.paged_attention_prefill(q, ctypes.byref(cache), 16, 8, 16, 16, batch,
                                           num_heads, num_tokens, scale, 16, max_query_len,
                                           None)

    assert call(scale=0.0) == 1
    assert call(scale=float("nan")) == 1
    assert call(num_tokens=-1) == 1
    assert call(num_heads=3) == 3            # not a multiple of the kv heads
    assert call(num_heads=2 * 130) == 3      # more than 128 query heads per kv head
    assert call(q=8) == 1                    # q not 16-byte aligned
    assert call(batch=65536) == 1
    assert call(num_tokens=1 << 31) == 1
    assert call(batch=0) == 0 and call(num_tokens=0) == 0 and call(max_query_len=0) == 0
    fp8_no_scale = _cache(dtype=1, k_scale=0.0)
    assert call(cache=fp8_no_scale) == 1


def test_blocks_write_and_prep_argument_validation(lib):
    """Block copy / swap, the fused zeroing + write and step input
    preparation reject bad arguments on the host, before any CUDA call."""
    c = _cache()
    cp = ctypes.byref(c)
    # copy-on-write and swap: negative counts, missing id lists; empty = no-op
    assert lib.paged_kv_copy_blocks(cp, 16, 16, -1, 1, None) == 1
    assert lib.paged_kv_copy_blocks(cp, None, 16, 3, 1, None) == 1
    assert lib.paged_kv_copy_blocks(cp, 16, 16, 0, 1, None) == 0
    for fn in (lib.paged_kv_swap_out, lib.paged_kv_swap_in):
        assert fn(cp, 16, -1, 1, 16, 16, None) == 1
        assert fn(cp, None, 3, 1, 16, 16, None) == 1
        assert fn(cp, 16, 0, 1, 16, 16, None) == 0
    # zeroing + write in one launch
    zw = lib.paged_kv_zero_and_write
    assert zw(16, 16, 16, -1, cp, 16, 1, 1, None) == 1
    assert zw(8, 16, 16, 1, cp, 16, 0, 1, None) == 1     # k not 16-byte aligned
    assert zw(16, 16, 16, 1, cp, None, 2, 1, None) == 1  # ids missing
    assert zw(16, 16, 16, 0, cp, None, 0, 1, None) == 0  # nothing to do
    # step input preparation
    def prep(batch=2, max_blocks=8, max_model_len=128, num_rows=4, total=5,
             qsl=16, positions=16):
        return lib.paged_prepare_inputs(16, 16, batch, 16, max_blocks, 16, 16, max_model_len,
                                        num_rows, total, 16, 16, qsl, positions, 16, 16, None)
    assert prep(batch=-1) == 1
    assert prep(max_blocks=0) == 1
    assert prep(max_model_len=0) == 1
    assert prep(qsl=None) == 1
    assert prep(positions=None) == 1
    assert prep(max_blocks=1 << 27) == 1     # max_blocks * 16 past int32
