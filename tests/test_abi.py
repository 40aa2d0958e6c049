"""The C ABI library: it builds, loads, exports every declared entry point,
and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "prhs.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^[A-Za-z_][\w\s\*]*?\b(prhs_\w+)\s*\(", src, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    from sparse_kv_selection_gb300 import build as B
    B.build()
    from sparse_kv_selection_gb300 import binding
    return binding.load()


def test_header_lists_entry_points():
    names = declared_functions()
    for must in ("prhs_score_select", "prhs_cis_dilate", "prhs_sparse_attn", "prhs_dense_attn",
                 "prhs_workspace_size", "prhs_last_error", "prhs_status_str"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from sparse_kv_selection_gb300 import binding
    names = declared_functions()
    assert sorted(names) == sorted(binding.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_library_is_sm103a_build():
    from sparse_kv_selection_gb300 import build as B
    assert B.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def _kv(binding, **over):
    d = binding.prhs_kv()
    d.dtype, d.B, d.Hq, d.Hkv, d.d = binding.PRHS_BF16, 1, 4, 4, 128
    d.k, d.v, d.seq_lens = 4096, 8192, 256
    d.t_max, d.block_table, d.block_size, d.max_blocks, d.num_blocks = 1024, None, 0, 0, 0
    for k, v in over.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("over,status", [
    (dict(d=96), 2),                     # head dim not built
    (dict(Hq=6, Hkv=2), 2),              # group of 3 not built
    (dict(Hq=5, Hkv=2), 1),              # Hq not a multiple of Hkv
    (dict(B=0), 1),
    (dict(k=4100), 1),                   # misaligned K
    (dict(seq_lens=None), 1),
    (dict(t_max=0), 1),
    (dict(block_table=512, block_size=8, max_blocks=4, num_blocks=4), 1),
    (dict(block_table=512, block_size=16, max_blocks=0, num_blocks=4), 1),
    (dict(dtype=7), 1),
    (dict(B=513, Hq=32, Hkv=32), 2),     # 16416 query heads: above the 16384 the kernels take
])
def test_descriptor_rejected_on_host(lib, over, status):
    from sparse_kv_selection_gb300 import binding
    kv = _kv(binding, **over)
    st = lib.prhs_sparse_attn(ctypes.byref(kv), 64, 0.1, 64, 64, 8, 64, 64, 256, 1 << 20, None)
    assert st == status
    assert lib.prhs_last_message().decode() != ""
    assert lib.prhs_workspace_size(ctypes.byref(kv), 8) == 0


def test_null_arguments_rejected(lib):
    from sparse_kv_selection_gb300 import binding
    kv = _kv(binding)
    assert lib.prhs_score_select(None, 64, 0.1, 8, None, 0, 0, None, 64, 64, 8, 64, None, None, 0,
                                 None, 256, 1 << 20, None) == binding.PRHS_EINVAL
    # N <= 0 without a per-sequence budget
    assert lib.prhs_score_select(ctypes.byref(kv), 64, 0.1, 0, None, 0, 0, None, 64, 64, 8, 64, None,
                                 None, 0, None, 256, 1 << 20, None) == binding.PRHS_EINVAL
    # capacity below the budget
    assert lib.prhs_score_select(ctypes.byref(kv), 64, 0.1, 16, None, 0, 0, None, 64, 64, 8, 64, None,
                                 None, 0, None, 256, 1 << 20, None) == binding.PRHS_EINVAL
    # anchor buffers must come together
    assert lib.prhs_score_select(ctypes.byref(kv), 64, 0.1, 8, None, 0, 0, None, 64, 64, 8, 64, 64,
                                 None, 8, None, 256, 1 << 20, None) == binding.PRHS_EINVAL
    # forced keys: non-negative, with the anchor buffers, and t_max <= 131072
    assert lib.prhs_score_select(ctypes.byref(kv), 64, 0.1, 8, None, -1, 0, None, 64, 64, 8, 64, 64,
                                 64, 8, 64, 256, 1 << 20, None) == binding.PRHS_EINVAL
    assert lib.prhs_score_select(ctypes.byref(kv), 64, 0.1, 8, None, 2, 2, None, 64, 64, 8, 64, None,
                                 None, 0, None, 256, 1 << 20, None) == binding.PRHS_EINVAL
    big = _kv(binding, t_max=1 << 18)
    assert lib.prhs_score_select(ctypes.byref(big), 64, 0.1, 8, None, 0, 4, None, 64, 64, 8, 64, 64,
                                 64, 8, 64, 256, 1 << 20, None) == binding.PRHS_EUNSUPPORTED
    assert lib.prhs_append_kv(ctypes.byref(kv), None, 64, None) == binding.PRHS_EINVAL
    # retrieval needs out and lse
    assert lib.prhs_retrieve(ctypes.byref(kv), 64, 0.1, 8, None, 0, 0, None, 64, 64, 8, 64, None, None,
                             0, None, None, 64, 256, 1 << 20, None) == binding.PRHS_EINVAL
    assert lib.prhs_retrieve(ctypes.byref(kv), 64, 0.1, 8, None, 0, 0, None, 64, 64, 8, 64, None, None,
                             0, None, 64, None, 256, 1 << 20, None) == binding.PRHS_EINVAL
    # dilation radius and dilated capacity
    assert lib.prhs_cis_dilate(ctypes.byref(kv), 64, 64, 8, 64, 64, -1, 0, 0, 0, 0.8, 0, None, 64, 64, 64, 64, None) == binding.PRHS_EINVAL
    assert lib.prhs_cis_dilate(ctypes.byref(kv), 64, 64, 8, 64, 64, 2, 0, 0, 0, 0.8, 0, None, 64, 64, 39, 64, None) == binding.PRHS_EINVAL
    # the dilated capacity must hold the forced keys too
    assert lib.prhs_cis_dilate(ctypes.byref(kv), 64, 64, 8, 64, 64, 2, 0, 2, 2, 0.8, 0, None, 64, 64, 40, 64, None) == binding.PRHS_EINVAL
    # a bounded reuse run needs the per-head age counters; a negative bound is invalid
    assert lib.prhs_cis_dilate(ctypes.byref(kv), 64, 64, 8, 64, 64, 2, 0, 0, 0, 0.8, 4, None, 64, 64, 64, 64, None) == binding.PRHS_EINVAL
    assert lib.prhs_cis_dilate(ctypes.byref(kv), 64, 64, 8, 64, 64, 2, 0, 0, 0, 0.8, -1, 64, 64, 64, 64, 64, None) == binding.PRHS_EINVAL
    assert lib.prhs_dense_attn(ctypes.byref(kv), None, 0.1, 64, 64, 256, 1 << 20, None) == binding.PRHS_EINVAL
    assert lib.prhs_workspace_init(None, 0, None) == binding.PRHS_EWORKSPACE
    # the dilation budget's denominator is non-negative
    assert lib.prhs_cis_dilate(ctypes.byref(kv), 64, 64, 8, 64, 64, 2, -1, 0, 0, 0.8, 0, None, 64, 64,
                               64, 64, None) == binding.PRHS_EINVAL
    # a gate array must be 16-byte aligned like q
    assert lib.prhs_decode_step(ctypes.byref(kv), 64, 72, 0.1, 8, None, 0, 0, 2, 0, 0.8, 0, None, 64,
                                64, 8, 64, 64, 64, 64, 64, 64, 64, 64, 256, 1 << 20, None) == binding.PRHS_EINVAL
    # the wait self-test takes a limit of 1 us .. 1 s
    assert lib.prhs_selftest_wait_timeout(0, None) == binding.PRHS_EINVAL
    assert lib.prhs_selftest_wait_timeout(1000001, None) == binding.PRHS_EINVAL


def test_status_strings(lib):
    from sparse_kv_selection_gb300 import binding
    seen = {binding.status_str(s) for s in range(6)}
    assert len(seen) == 6 and "ok" in seen
