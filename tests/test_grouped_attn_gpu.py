"""Sparse attention for grouped query heads (several query heads per KV
head): parity with the fp64 oracle per query head on index sets that overlap
across a group in every way they can (identical, disjoint, nested, one empty
and one whole, dilated runs around shared centres, random), on contiguous
and paged caches of several thousand keys, for groups of 2, 4 and 8, with
two calls in a row on one workspace (the completion tickets left at zero);
a 131072-key cache; and a page id outside the pool (flagged, its rows
skipped)."""
import math

import numpy as np
import pytest

import oracle.prhs as P
from parity_util import LSE_TOL, OUT_TOL, kv_rows64, q64
from workloads import make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _setup(G, paged, t, B=2, Hkv=2, d=128, dtype="bf16", seed=0):
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload
    wl = make_workload("grouped", dtype=dtype, B=B, Hq=Hkv * G, Hkv=Hkv, d=d, t=t, paged=paged,
                       block_size=16, n_clusters=8, steps=2, N=64, w=1, seed=seed)
    dev = upload(wl)
    kv = S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq, block_table=dev["block_table"])
    return S, wl, dev, kv


def _group_sets(rng, G, t, pattern):
    """G index sets over [0, t) with the given overlap pattern."""
    base = np.sort(rng.choice(t, size=min(t, 300), replace=False))
    if pattern == "identical":
        return [base] * G
    if pattern == "disjoint":
        perm = rng.permutation(t)
        k = max(1, t // (2 * G))
        return [np.sort(perm[g * k:(g + 1) * k]) for g in range(G)]
    if pattern == "nested":
        return [base[:max(1, len(base) * (g + 1) // G)] for g in range(G)]
    if pattern == "one_empty_one_all":
        sets = [np.sort(rng.choice(t, size=int(rng.integers(1, t)), replace=False)) for _ in range(G)]
        sets[0] = np.array([], np.int64)
        sets[-1] = np.arange(t)
        return sets
    if pattern == "dilated_runs":   # the decode step's shape: runs around shared centres
        c = np.sort(rng.choice(t, size=40, replace=False))
        return [P.dilate(np.sort(rng.choice(c, size=30, replace=False)), 3, t) for _ in range(G)]
    return [np.sort(rng.choice(t, size=int(rng.integers(0, t + 1)), replace=False)) for _ in range(G)]


PATTERNS = ["identical", "disjoint", "nested", "one_empty_one_all", "dilated_runs", "random"]


def _run_and_check(S, wl, dev, kv, sets, cap, ws, step=0):
    idx = np.zeros((wl.B, wl.Hq, cap), np.int32)
    n = np.zeros((wl.B, wl.Hq), np.int32)
    for (b, h), Sx in sets.items():
        idx[b, h, :len(Sx)] = Sx
        n[b, h] = len(Sx)
    out = torch.full((wl.B, wl.Hq, wl.d), 7.0, device="cuda")
    lse = torch.full((wl.B, wl.Hq), 7.0, device="cuda")
    S.sparse_attn(kv, dev["q"][step], wl.scale, torch.from_numpy(idx).cuda(),
                  torch.from_numpy(n).cuda(), out, lse, ws)
    assert S.last_error() == 0
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for (b, h), Sx in sets.items():
        if len(Sx) == 0:
            assert (o[b, h] == 0).all() and l[b, h] == -math.inf, (b, h)
            continue
        K, V = kv_rows64(wl, b, h // wl.G)
        ro, rl = P.attention(q64(wl, step, b, h), K, V, Sx, wl.scale)
        assert np.abs(o[b, h] - ro).max() <= OUT_TOL, (b, h)
        assert abs(l[b, h] - rl) <= LSE_TOL, (b, h)


@pytest.mark.parametrize("G", [2, 4, 8])
@pytest.mark.parametrize("paged", [False, True])
def test_grouped_overlap_patterns_two_calls(G, paged):
    S, wl, dev, kv = _setup(G, paged, t=(2500, 5200))
    rng = np.random.default_rng(100 + G)
    cap = int(wl.seq_lens.max())
    ws = S.make_workspace(kv, cap)
    for call in range(2):
        sets = {}
        for b in range(wl.B):
            t = int(wl.seq_lens[b])
            for kvh in range(wl.Hkv):
                pat = PATTERNS[(call * 5 + b * wl.Hkv + kvh) % len(PATTERNS)]
                for g, Sx in enumerate(_group_sets(rng, G, t, pat)):
                    sets[(b, kvh * G + g)] = np.asarray(Sx, np.int64)
        _run_and_check(S, wl, dev, kv, sets, cap, ws, step=call)


@pytest.mark.parametrize("dtype,d", [("f32", 128), ("bf16", 64), ("f32", 64)])
def test_grouped_element_types(dtype, d):
    S, wl, dev, kv = _setup(4, False, t=3000, B=1, d=d, dtype=dtype)
    rng = np.random.default_rng(7)
    cap = 3000
    ws = S.make_workspace(kv, cap)
    sets = {}
    for kvh in range(wl.Hkv):
        for g, Sx in enumerate(_group_sets(rng, 4, 3000, "dilated_runs" if kvh else "random")):
            sets[(0, kvh * 4 + g)] = np.asarray(Sx, np.int64)
    _run_and_check(S, wl, dev, kv, sets, cap, ws)


def test_grouped_long_cache():
    """131072 keys, group of 8: sets from 1 key to a whole 4096-key run at
    the end of the cache."""
    S, wl, dev, kv = _setup(8, False, t=131072, B=1, Hkv=1)
    rng = np.random.default_rng(9)
    cap = 4096
    ws = S.make_workspace(kv, cap)
    sets = {}
    for g in range(8):
        k = [1, 17, 300, 4096, 2500, 64, 1000, 3][g]
        sets[(0, g)] = np.sort(rng.choice(131072, size=k, replace=False))
    sets[(0, 3)] = np.arange(131072 - 4096, 131072)   # one whole chunk run at the end
    for rep in range(2):
        _run_and_check(S, wl, dev, kv, sets, cap, ws)


def test_grouped_bad_page_flagged_and_skipped():
    """A page id outside the pool: its rows are flagged and attended by no
    head, the other rows of the sets give the oracle's attention."""
    S, wl, dev, kv = _setup(4, True, t=800, B=1)
    from sparse_kv_selection_gb300.binding import DEV_BAD_BLOCK
    table = dev["block_table"].clone()
    table[0, 3] = 10 ** 6                  # keys 48..63 of sequence 0
    kv_bad = S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq, block_table=table)
    rng = np.random.default_rng(5)
    cap = 800
    idx = np.zeros((1, wl.Hq, cap), np.int32)
    n = np.zeros((1, wl.Hq), np.int32)
    sets = {}
    for h in range(wl.Hq):
        Sx = np.sort(np.union1d(rng.choice(800, size=100, replace=False), np.arange(40, 70)))
        sets[h] = Sx
        idx[0, h, :len(Sx)] = Sx
        n[0, h] = len(Sx)
    out = torch.empty(1, wl.Hq, wl.d, device="cuda")
    lse = torch.empty(1, wl.Hq, device="cuda")
    ws = S.make_workspace(kv_bad, cap)
    S.sparse_attn(kv_bad, dev["q"][0], wl.scale, torch.from_numpy(idx).cuda(),
                  torch.from_numpy(n).cuda(), out, lse, ws)
    assert S.last_error() & DEV_BAD_BLOCK
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for h in range(wl.Hq):
        keep = sets[h][(sets[h] < 48) | (sets[h] >= 64)]
        K, V = kv_rows64(wl, 0, h // wl.G)
        ro, rl = P.attention(q64(wl, 0, 0, h), K, V, keep, wl.scale)
        assert np.abs(o[0, h] - ro).max() <= OUT_TOL and abs(l[0, h] - rl) <= LSE_TOL, h
    # the workspace is clean again: a correct call right after is exact
    _run_and_check(S, wl, dev, kv, {(0, h): sets[h] for h in range(wl.Hq)}, cap, ws)
