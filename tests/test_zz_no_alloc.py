"""prhs_sparse_attn_noalloc: sparse attention for callers that cannot call
cudaMalloc (and so cannot pass a workspace). It must give the results of
prhs_sparse_attn, call after call, from its fixed in-library scratch.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import oracle.prhs as P
from parity_util import LSE_TOL, OUT_TOL, kv_rows64, q64
from workloads import make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _case(paged):
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload
    S.load()
    wl = make_workload("noalloc", dtype="bf16", B=2, Hq=8, Hkv=2, d=128, t=(900, 2100),
                       paged=paged, block_size=16, n_clusters=20, steps=2, N=128, w=2, seed=4)
    dev = upload(wl)
    kv = S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq, block_table=dev["block_table"])
    cap = 128 * 5
    idx = np.zeros((wl.B, wl.Hq, cap), np.int32)
    n = np.zeros((wl.B, wl.Hq), np.int32)
    for b in range(wl.B):
        for h in range(wl.Hq):
            K, _ = kv_rows64(wl, b, h // wl.G)
            s = P.scores(q64(wl, 0, b, h), K, wl.scale)
            sel = P.top_n(s, 128)
            if h % 2:
                sel = P.dilate(sel, 2, K.shape[0])
            idx[b, h, :len(sel)] = sel
            n[b, h] = len(sel)
    return S, wl, dev, kv, torch.from_numpy(idx).cuda(), torch.from_numpy(n).cuda()


@pytest.mark.parametrize("paged", [False, True])
def test_noalloc_matches_workspace_version_twice(paged):
    S, wl, dev, kv, idx, n = _case(paged)
    ref_out = torch.empty(wl.B, wl.Hq, wl.d, device="cuda")
    ref_lse = torch.empty(wl.B, wl.Hq, device="cuda")
    ws = S.make_workspace(kv, idx.shape[-1])
    S.sparse_attn(kv, dev["q"][0], wl.scale, idx, n, ref_out, ref_lse, ws)
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        S.binding.sparse_attn_noalloc(kv, dev["q"][0], wl.scale, idx, n, out, lse)
        torch.cuda.synchronize()
        assert (out - ref_out).abs().max().item() <= OUT_TOL, call
        assert (lse - ref_lse).abs().max().item() <= LSE_TOL, call
    assert S.last_error() == 0


def test_noalloc_rejects_batches_beyond_its_scratch():
    import sparse_kv_selection_gb300 as S
    from sparse_kv_selection_gb300.binding import PRHS_EINVAL
    Hq, Hkv, t, d = 8192, 1024, 16, 128      # 8192 heads need > 4 MiB of partials
    k = torch.zeros(1, Hkv, t, d, dtype=torch.bfloat16, device="cuda")
    kv = S.KVCache(k, k, torch.tensor([t], dtype=torch.int32, device="cuda"), Hq)
    idx = torch.zeros(1, Hq, 4, dtype=torch.int32, device="cuda")
    n = torch.ones(1, Hq, dtype=torch.int32, device="cuda")
    out = torch.empty(1, Hq, d, device="cuda")
    lse = torch.empty(1, Hq, device="cuda")
    with pytest.raises(S.PrhsError) as e:
        S.binding.sparse_attn_noalloc(kv, torch.zeros(1, Hq, d, dtype=torch.bfloat16,
                                                      device="cuda"), 0.1, idx, n, out, lse)
    assert e.value.status == PRHS_EINVAL and "scratch" in str(e.value)
