"""GPU parity: every C ABI call against the fp64 oracle on the same seeded
inputs (shapes spanning several tiles and a ragged tail, contiguous and
paged caches, MHA and grouped heads, bf16 and fp32)."""
import math

import numpy as np
import pytest

import oracle.prhs as P
from parity_util import (DELTA_TOL, GATE_GAP, LSE_TOL, OUT_TOL, TIE_GAP, check_topn,
                         compare_decode, compare_decode_forced, kv_rows64, q64)
from workloads import make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = {
    "mha_bf16_ragged": dict(dtype="bf16", B=2, Hq=4, Hkv=4, d=128, t=(700, 1500), t_max=1600,
                            n_clusters=12, steps=6, N=96, w=2),
    "gqa4_bf16": dict(dtype="bf16", B=2, Hq=8, Hkv=2, d=128, t=1000, n_clusters=16, steps=6,
                      N=100, w=4),
    "paged_bf16": dict(dtype="bf16", B=3, Hq=4, Hkv=4, d=128, t=(300, 2000), paged=True,
                       block_size=16, n_clusters=lambda tb: tb // 64, steps=6, budget_div=16, w=2),
    "f32_d64_gqa2": dict(dtype="f32", B=1, Hq=2, Hkv=1, d=64, t=517, n_clusters=8, steps=6,
                         N=64, w=2),
    "bf16_d64_gqa8": dict(dtype="bf16", B=1, Hq=8, Hkv=1, d=64, t=900, n_clusters=10, steps=4,
                          N=50, w=1),
    "f32_d128_paged32": dict(dtype="f32", B=2, Hq=2, Hkv=2, d=128, t=(100, 400), paged=True,
                             block_size=32, n_clusters=4, steps=4, N=40, w=3),
    # caches of 4097..8192 keys: sixteen CTAs per head in the score-and-select kernel
    "bf16_long_gqa2": dict(dtype="bf16", B=2, Hq=4, Hkv=2, d=128, t=(5000, 8192), t_max=8192,
                           n_clusters=48, steps=4, N=300, w=2),
    # t_max above 8192: separate scoring, selection and attention launches
    "bf16_9k_mha": dict(dtype="bf16", B=1, Hq=2, Hkv=2, d=128, t=(8500, 9500), t_max=9600,
                        n_clusters=32, steps=4, N=256, w=2),
    # t_max above 8192 with at most one head per SM and no cluster attention
    # (128 heads x 1300 anchors): the decode step scores before the branches
    # fork, then selects and attends the retrieving heads beside the others
    "gqa4_12k_score_first": dict(dtype="bf16", B=4, Hq=32, Hkv=8, d=128, t=(9000, 12000),
                                 t_max=12000, n_clusters=40, steps=4, N=1300, w=2),
    # a cache of one key: every budget covers it (set = {0}, delta = 0)
    "t1_bf16": dict(dtype="bf16", B=2, Hq=2, Hkv=2, d=128, t=1, n_clusters=0, steps=4, N=4, w=2),
    "t1_paged_f32": dict(dtype="f32", B=2, Hq=4, Hkv=1, d=64, t=1, paged=True, block_size=16,
                         n_clusters=0, steps=4, N=1, w=1),
    # caches of 7 keys (less than one 16-key tile), contiguous and paged, grouped
    "t7_paged_gqa4": dict(dtype="bf16", B=2, Hq=8, Hkv=2, d=128, t=7, paged=True, block_size=16,
                          n_clusters=0, steps=4, N=3, w=1),
    "t7_bf16_gqa4": dict(dtype="bf16", B=1, Hq=4, Hkv=1, d=128, t=7, n_clusters=0, steps=4, N=3,
                         w=2),
    # ragged caches of 4 and 7 keys with w = 0 (DirectReuse: the shared set is
    # the anchor's top-N set itself)
    "t4to7_f32_w0": dict(dtype="f32", B=3, Hq=2, Hkv=1, d=64, t=(1, 7), t_max=7, n_clusters=0,
                         steps=4, N=2, w=0),
    "w0_bf16_gqa4": dict(dtype="bf16", B=2, Hq=8, Hkv=2, d=128, t=1200, n_clusters=16, steps=6,
                         N=64, w=0),
    # budget above some caches of a grouped paged batch (lengths 212..387, N = 300)
    "paged_gqa4_n_gt_t": dict(dtype="bf16", B=4, Hq=8, Hkv=2, d=128, t=(5, 400), paged=True,
                              block_size=16, n_clusters=lambda tb: tb // 64, steps=6, N=300, w=2),
}


def _setup(name, seed=0):
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload
    wl = make_workload(name, seed=seed, **CASES[name])
    dev = upload(wl)
    kv = S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq, block_table=dev["block_table"])
    return S, wl, dev, kv


def _heads(wl):
    return [(b, h) for b in range(wl.B) for h in range(wl.Hq)]


@pytest.fixture(autouse=True)
def _clean_error_word():
    import sparse_kv_selection_gb300 as S
    S.last_error()
    yield
    assert S.last_error() == 0, "kernels reported a device data error"


# --------------------------------------------------------------------------- #
# dense attention
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("name", list(CASES))
def test_dense_attn(name):
    S, wl, dev, kv = _setup(name)
    out = torch.empty(wl.B, wl.Hq, wl.d, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, device="cuda")
    ws = S.make_workspace(kv)
    for step in (0, wl.steps - 1):
        S.dense_attn(kv, dev["q"][step], wl.scale, out, lse, ws)
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        for b, h in _heads(wl):
            K, V = kv_rows64(wl, b, h // wl.G)
            ro, rl = P.dense_attention(q64(wl, step, b, h), K, V, wl.scale)
            assert np.abs(o[b, h] - ro).max() <= OUT_TOL
            assert abs(l[b, h] - rl) <= LSE_TOL


# --------------------------------------------------------------------------- #
# sparse attention over oracle-chosen sets
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("name", list(CASES))
def test_sparse_attn_on_oracle_sets(name):
    S, wl, dev, kv = _setup(name)
    rng = np.random.default_rng(5)
    cap = max(1, min(wl.t_max, int(wl.budget.max()) * (2 * wl.w + 1)))
    idx = np.zeros((wl.B, wl.Hq, cap), np.int32)
    n = np.zeros((wl.B, wl.Hq), np.int32)
    sets = {}
    for b, h in _heads(wl):
        K, V = kv_rows64(wl, b, h // wl.G)
        t = K.shape[0]
        s = P.scores(q64(wl, 1, b, h), K, wl.scale)
        kind = (b * wl.Hq + h) % 3
        if kind == 0:
            Sx = P.top_n(s, int(wl.budget[b]))
        elif kind == 1:
            Sx = P.dilate(P.top_n(s, int(wl.budget[b])), wl.w, t)
        else:
            Sx = np.sort(rng.choice(t, size=min(t, cap, int(rng.integers(1, 300))), replace=False))
        sets[(b, h)] = Sx
        idx[b, h, :len(Sx)] = Sx
        n[b, h] = len(Sx)
    out = torch.empty(wl.B, wl.Hq, wl.d, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, device="cuda")
    ws = S.make_workspace(kv, cap)
    S.sparse_attn(kv, dev["q"][1], wl.scale, torch.from_numpy(idx).cuda(),
                  torch.from_numpy(n).cuda(), out, lse, ws)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for b, h in _heads(wl):
        K, V = kv_rows64(wl, b, h // wl.G)
        ro, rl = P.attention(q64(wl, 1, b, h), K, V, sets[(b, h)], wl.scale)
        assert np.abs(o[b, h] - ro).max() <= OUT_TOL, (b, h)
        assert abs(l[b, h] - rl) <= LSE_TOL, (b, h)


@pytest.mark.parametrize("B,Hq,t,live,nmax", [
    (2, 4, 1500, 1, 1400),     # one head with rows: each CTA takes part of that head
    (2, 4, 1500, 8, 1400),     # every head, long sets: CTAs aligned to heads
    (8, 32, 300, 256, 40),     # many heads with short sets: CTAs straddle heads
    (65, 32, 64, 2080, 20),    # more heads than the head-aligned split handles
])
def test_sparse_attn_split_modes(B, Hq, t, live, nmax):
    """Both ways of cutting the rows over CTAs, and the merge of split heads."""
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload
    wl = make_workload("split", dtype="bf16", B=B, Hq=Hq, Hkv=Hq, d=128, t=t, n_clusters=2,
                       steps=1, N=8, w=1, seed=3)
    dev = upload(wl)
    kv = S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq)
    rng = np.random.default_rng(11)
    cap = nmax
    idx = np.zeros((B, Hq, cap), np.int32)
    n = np.zeros((B, Hq), np.int32)
    sets = {}
    for u in range(B * Hq):
        b, h = divmod(u, Hq)
        if u >= live:
            continue
        k = int(rng.integers(1, min(nmax, t) + 1))
        Sx = np.sort(rng.choice(t, size=k, replace=False))
        sets[(b, h)] = Sx
        idx[b, h, :k] = Sx
        n[b, h] = k
    out = torch.full((B, Hq, wl.d), 7.0, device="cuda")
    lse = torch.full((B, Hq), 7.0, device="cuda")
    ws = S.make_workspace(kv, cap)
    for rep in range(2):  # tickets must be back at zero for the second call
        S.sparse_attn(kv, dev["q"][0], wl.scale, torch.from_numpy(idx).cuda(),
                      torch.from_numpy(n).cuda(), out, lse, ws)
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        for u in range(B * Hq):
            b, h = divmod(u, Hq)
            if (b, h) not in sets:
                assert (o[b, h] == 0).all() and l[b, h] == -math.inf, (b, h)
                continue
            K, V = kv_rows64(wl, b, h)
            ro, rl = P.attention(q64(wl, 0, b, h), K, V, sets[(b, h)], wl.scale)
            assert np.abs(o[b, h] - ro).max() <= OUT_TOL, (rep, b, h)
            assert abs(l[b, h] - rl) <= LSE_TOL, (rep, b, h)


def test_sparse_attn_edge_sets():
    """Empty set, single key, every key, last key, repeated calls."""
    S, wl, dev, kv = _setup("mha_bf16_ragged")
    cap = wl.t_max
    idx = np.zeros((wl.B, wl.Hq, cap), np.int32)
    n = np.zeros((wl.B, wl.Hq), np.int32)
    t0 = int(wl.seq_lens[0])
    t1 = int(wl.seq_lens[1])
    cases = {(0, 0): np.array([], np.int64), (0, 1): np.array([7]), (0, 2): np.arange(t0),
             (0, 3): np.array([t0 - 1]), (1, 0): np.arange(t1), (1, 1): np.arange(0, t1, 97),
             (1, 2): np.array([0, t1 - 1]), (1, 3): np.arange(t1 - 33, t1)}
    for (b, h), Sx in cases.items():
        idx[b, h, :len(Sx)] = Sx
        n[b, h] = len(Sx)
    out = torch.empty(wl.B, wl.Hq, wl.d, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, device="cuda")
    ws = S.make_workspace(kv, cap)
    for rep in range(2):  # the completion tickets must be left at zero
        S.sparse_attn(kv, dev["q"][0], wl.scale, torch.from_numpy(idx).cuda(),
                      torch.from_numpy(n).cuda(), out, lse, ws)
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        assert (o[0, 0] == 0).all() and l[0, 0] == -math.inf
        for (b, h), Sx in cases.items():
            if len(Sx) == 0:
                continue
            K, V = kv_rows64(wl, b, h)
            ro, rl = P.attention(q64(wl, 0, b, h), K, V, Sx, wl.scale)
            assert np.abs(o[b, h] - ro).max() <= OUT_TOL and abs(l[b, h] - rl) <= LSE_TOL


def test_sparse_attn_flags_bad_index():
    """Entries outside [0, t_b) are skipped and reported, never read."""
    S, wl, dev, kv = _setup("gqa4_bf16")
    cap = 16
    idx = np.tile(np.arange(cap, dtype=np.int32), (wl.B, wl.Hq, 1))
    n = np.full((wl.B, wl.Hq), cap, np.int32)
    idx[1, 3, 5] = 10 ** 6
    idx[0, 0, 0] = -3
    out = torch.empty(wl.B, wl.Hq, wl.d, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, device="cuda")
    ws = S.make_workspace(kv, cap)
    S.sparse_attn(kv, dev["q"][0], wl.scale, torch.from_numpy(idx).cuda(),
                  torch.from_numpy(n).cuda(), out, lse, ws)
    from sparse_kv_selection_gb300.binding import DEV_BAD_INDEX
    assert S.last_error() & DEV_BAD_INDEX
    o = out.cpu().numpy()
    K, V = kv_rows64(wl, 1, 3 // wl.G)
    keep = np.array([i for i in range(cap) if i != 5])
    ro, _ = P.attention(q64(wl, 0, 1, 3), K, V, keep, wl.scale)
    assert np.abs(o[1, 3] - ro).max() <= OUT_TOL


# --------------------------------------------------------------------------- #
# top-N selection and dropped mass
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("name", list(CASES))
def test_score_select(name):
    S, wl, dev, kv = _setup(name)
    N = int(wl.budget.max())
    cap = max(1, min(N, wl.t_max))
    idx = torch.full((wl.B, wl.Hq, cap), -7, dtype=torch.int32, device="cuda")
    n_sel = torch.empty(wl.B, wl.Hq, dtype=torch.int32, device="cuda")
    delta = torch.empty(wl.B, wl.Hq, device="cuda")
    aidx = torch.full_like(idx, -9)
    an = torch.zeros_like(n_sel)
    qa = torch.zeros_like(dev["q"][0])
    ws = S.make_workspace(kv, cap)
    nb = dev["budget"] if wl.params and len(set(wl.budget.tolist())) > 1 else None
    S.score_select(kv, dev["q"][2], wl.scale, N, idx, n_sel, delta, ws, n_budget=nb,
                   anchor_idx=aidx, anchor_n=an, q_anchor=qa)
    gi, gn, gd = idx.cpu().numpy(), n_sel.cpu().numpy(), delta.cpu().numpy()
    ga = aidx.cpu().numpy()
    assert (an.cpu().numpy() == gn).all()
    for b, h in _heads(wl):
        assert (ga[b, h, :gn[b, h]] == gi[b, h, :gn[b, h]]).all()
    assert torch.equal(qa, dev["q"][2])
    ties = 0
    for b, h in _heads(wl):
        K, _ = kv_rows64(wl, b, h // wl.G)
        s = P.scores(q64(wl, 2, b, h), K, wl.scale)
        Nb = int(wl.budget[b]) if nb is not None else N
        Nb_eff = min(Nb, s.size)
        assert gn[b, h] == Nb_eff
        ties += check_topn(gi[b, h, :gn[b, h]], s, Nb)
        assert abs(gd[b, h] - P.dropped_mass(s, P.top_n(s, Nb))) <= DELTA_TOL
        assert (gi[b, h, gn[b, h]:] == -7).all()
    print(f"{name}: near-tie positions left uncompared: {ties}")


@pytest.mark.parametrize("t,dup_end,Ns", [
    (700, 400, (1, 2, 150, 301, 302, 650)),
    # 8192 keys: the logits are split over a cluster of CTAs, ties cross slices
    (8192, 6000, (1, 500, 3000, 5901, 5902, 7000)),
])
def test_score_select_exact_ties_lowest_index(t, dup_end, Ns):
    """Duplicated key rows give bit-identical logits: the lowest indices win."""
    import sparse_kv_selection_gb300 as S
    d = 128
    rng = np.random.default_rng(3)
    K = rng.normal(size=(t, d)).astype(np.float32)
    K[100:dup_end] = K[50]      # identical rows: index 50 and 100..dup_end-1
    q = (K[50] * 0.5 + rng.normal(size=d) * 0.1).astype(np.float32)
    for N in Ns:
        kt = torch.from_numpy(K).reshape(1, 1, t, d).cuda()
        kv = S.KVCache(kt, kt, torch.tensor([t], dtype=torch.int32).cuda(), 1)
        idx = torch.empty(1, 1, N, dtype=torch.int32, device="cuda")
        n_sel = torch.empty(1, 1, dtype=torch.int32, device="cuda")
        delta = torch.empty(1, 1, device="cuda")
        ws = S.make_workspace(kv, N)
        S.score_select(kv, torch.from_numpy(q).reshape(1, 1, d).cuda(), 1 / math.sqrt(d), N, idx,
                       n_sel, delta, ws)
        s = P.scores(q.astype(np.float64), K.astype(np.float64), 1 / math.sqrt(d))
        ref = P.top_n(s, N)
        got = idx.cpu().numpy()[0, 0]
        tied = np.abs(s - s[50]) < TIE_GAP
        # tied rows are bit-identical on both sides: compare exactly unless an
        # untied key sits within the near-tie band of the N-th logit
        s_n = np.sort(s)[::-1][N - 1]
        other_near = (np.abs(s - s_n) < TIE_GAP) & ~tied
        if not other_near.any():
            assert got.tolist() == ref.tolist(), N


def test_score_select_head_skip_and_full_budget():
    S, wl, dev, kv = _setup("gqa4_bf16")
    cap = wl.t_max
    idx = torch.full((wl.B, wl.Hq, cap), -5, dtype=torch.int32, device="cuda")
    n_sel = torch.full((wl.B, wl.Hq), -5, dtype=torch.int32, device="cuda")
    delta = torch.full((wl.B, wl.Hq), -5.0, device="cuda")
    skip = torch.zeros(wl.B, wl.Hq, dtype=torch.uint8, device="cuda")
    skip[0, 1] = 1
    skip[1, 4:8] = 1   # a whole KV group
    ws = S.make_workspace(kv, cap)
    S.score_select(kv, dev["q"][0], wl.scale, 10 ** 6, idx, n_sel, delta, ws, head_skip=skip)
    gi, gn, gd = idx.cpu().numpy(), n_sel.cpu().numpy(), delta.cpu().numpy()
    sk = skip.cpu().numpy().astype(bool)
    assert (gi[sk] == -5).all() and (gn[sk] == -5).all() and (gd[sk] == -5).all()
    t = wl.t_max
    for b, h in _heads(wl):
        if not sk[b, h]:
            assert gn[b, h] == t and gd[b, h] == 0.0 and (gi[b, h] == np.arange(t)).all()


@pytest.mark.parametrize("paged", [False, True])
def test_score_select_one_head_per_kv_head_long(paged):
    """prhs_score then prhs_select on caches above 8192 keys with one query
    head per KV head: ragged lengths from 9000 to 40000 keys, contiguous and
    paged (one TMA box per page), a third of the heads skipped; the sets and
    dropped masses of the scored heads against the oracle."""
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload
    wl = make_workload("mha_long", dtype="bf16", B=2, Hq=3, Hkv=3, d=128, t=(9000, 40000),
                       paged=paged, block_size=16, n_clusters=40, steps=1, N=700, w=1)
    dev = upload(wl)
    kv = S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq, block_table=dev["block_table"])
    N = 700
    skip = np.zeros((wl.B, wl.Hq), np.uint8)
    skip[0, 1] = skip[1, 0] = 1
    idx = torch.full((wl.B, wl.Hq, N), -1, dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(wl.B, wl.Hq, dtype=torch.int32, device="cuda")
    delta = torch.zeros(wl.B, wl.Hq, device="cuda")
    ws = S.make_workspace(kv, N)
    S.binding.score(kv, dev["q"][0], wl.scale, ws, head_skip=torch.from_numpy(skip).cuda())
    S.binding.select(kv, dev["q"][0], N, idx, n_sel, delta, ws, head_skip=torch.from_numpy(skip).cuda())
    assert S.last_error() == 0
    gi, gn, gd = idx.cpu().numpy(), n_sel.cpu().numpy(), delta.cpu().numpy()
    for b, h in _heads(wl):
        if skip[b, h]:
            continue
        K, _ = kv_rows64(wl, b, h)
        sc = P.scores(q64(wl, 0, b, h), K, wl.scale)
        gset = gi[b, h, :gn[b, h]]
        check_topn(gset, sc, N)
        assert abs(gd[b, h] - P.dropped_mass(sc, gset)) <= DELTA_TOL, (b, h)


@pytest.mark.parametrize("t,N", [(70001, 1500), (49153, 3), (200003, 777)])
def test_score_select_long_cache(t, N):
    """Long caches: logits split over a cluster of CTAs, and (200003 keys,
    beyond eight shared-memory slices) streamed by one CTA from L2."""
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload
    wl = make_workload("long", dtype="bf16", B=1, Hq=2, Hkv=1, d=128, t=t, n_clusters=40,
                       sinks=4, steps=1, N=N, w=1)
    dev = upload(wl)
    kv = S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq)
    idx = torch.empty(1, 2, N, dtype=torch.int32, device="cuda")
    n_sel = torch.empty(1, 2, dtype=torch.int32, device="cuda")
    delta = torch.empty(1, 2, device="cuda")
    ws = S.make_workspace(kv, N)
    S.score_select(kv, dev["q"][0], wl.scale, N, idx, n_sel, delta, ws)
    K, _ = kv_rows64(wl, 0, 0)
    for h in range(2):
        s = P.scores(q64(wl, 0, 0, h), K, wl.scale)
        check_topn(idx.cpu().numpy()[0, h], s, N)
        assert abs(delta.cpu().numpy()[0, h] - P.dropped_mass(s, P.top_n(s, N))) <= DELTA_TOL


@pytest.mark.parametrize("t,N,Hq,Hkv,paged", [(70001, 1500, 2, 1, False), (131072, 4096, 8, 2, False),
                                               (200003, 777, 2, 1, False), (40000, 2500, 4, 4, True)])
def test_retrieve_long_cache(t, N, Hq, Hkv, paged):
    """prhs_retrieve past the one-launch limit: scoring, selection, then an
    attention launch that weights the selected V rows by the logits the
    scoring left in the workspace. Set (up to near-ties), delta, out and lse
    of every retrieving head against the oracle; a skipped head untouched."""
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload
    wl = make_workload("long", dtype="bf16", B=1, Hq=Hq, Hkv=Hkv, d=128, t=t, n_clusters=40,
                       sinks=4, steps=1, N=N, w=1, paged=paged, block_size=16)
    dev = upload(wl)
    kv = S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq, block_table=dev["block_table"])
    i32 = dict(dtype=torch.int32, device="cuda")
    idx = torch.full((1, Hq, N), -7, **i32)
    n_sel = torch.full((1, Hq), -7, **i32)
    delta = torch.full((1, Hq), -7.0, device="cuda")
    out = torch.full((1, Hq, 128), -7.0, device="cuda")
    lse = torch.full((1, Hq), -7.0, device="cuda")
    skip = torch.zeros(1, Hq, dtype=torch.uint8, device="cuda")
    skip[0, Hq - 1] = 1
    ws = S.make_workspace(kv, N)
    c0 = S.binding.launch_count()
    S.retrieve(kv, dev["q"][0], wl.scale, N, idx, n_sel, delta, out, lse, ws, head_skip=skip)
    assert S.binding.launch_count() - c0 == 3   # scoring, selection, attention
    assert S.last_error() == 0
    gi, gn, gd, go, gl = [x.cpu().numpy() for x in (idx, n_sel, delta, out, lse)]
    for h in range(Hq):
        if h == Hq - 1:
            assert gn[0, h] == -7 and (go[0, h] == -7.0).all() and gl[0, h] == -7.0
            continue
        K, V = kv_rows64(wl, 0, h // wl.G)
        qv = q64(wl, 0, 0, h)
        sc = P.scores(qv, K, wl.scale)
        gset = gi[0, h, :gn[0, h]]
        check_topn(gset, sc, N)
        assert abs(gd[0, h] - P.dropped_mass(sc, gset)) <= DELTA_TOL, h
        ro, rl = P.attention(qv, K, V, gset, wl.scale)
        assert np.abs(go[0, h] - ro).max() <= OUT_TOL and abs(gl[0, h] - rl) <= LSE_TOL, h


@pytest.mark.parametrize("t", [4096, 12000, 50000])
def test_retrieve_geometric_logits_radix_fallback(t):
    """Logits in a geometric progression (2^0 ... 2^-99, many copies of each,
    above them a hundred values in (1, 1.8]): value bins over the range leave the small
    ones in one bin round after round, so every selection form ends in its
    radix fallback: the one-launch retrieval (4096 keys), the one-CTA
    selection (12000) and the cluster selection (50000). With q = e1, scale
    1 and bf16-exact key values the logits are exact on both sides, so the
    set (ties by lowest index) must equal the oracle's exactly."""
    import sparse_kv_selection_gb300 as S
    from workloads import bf16_bits_from_f32
    from workloads.torch_io import tensor_of
    rng = np.random.default_rng(t)
    H, d, J = 2, 128, 100
    copies = (t - 96) // J
    n_big = t - J * copies
    kf = np.zeros((1, H, t, d), np.float32)
    vf = rng.normal(size=(1, H, t, d)).astype(np.float32)
    for h in range(H):
        # the large values 1 + k/128 (exact in bf16) keep the small keys' weights
        # within a factor e^-1.8 of the largest, so delta and out test them too
        vals = np.concatenate([np.repeat(2.0 ** -np.arange(J), copies), 1.0 + (1.0 + np.arange(n_big)) / 128])
        kf[0, h, :, 0] = vals[rng.permutation(t)]
    qf = np.zeros((1, H, d), np.float32)
    qf[..., 0] = 1.0
    kb, vb, qb = bf16_bits_from_f32(kf), bf16_bits_from_f32(vf), bf16_bits_from_f32(qf)
    k, v, q = tensor_of(kb, "bf16", "cuda"), tensor_of(vb, "bf16", "cuda"), tensor_of(qb, "bf16", "cuda")
    kv = S.KVCache(k, v, torch.tensor([t], dtype=torch.int32, device="cuda"), H)
    N = n_big + copies * 50 + copies // 2   # the threshold inside the ties of 2^-50
    i32 = dict(dtype=torch.int32, device="cuda")
    idx = torch.full((1, H, N), -7, **i32)
    n_sel = torch.full((1, H), -7, **i32)
    delta = torch.zeros(1, H, device="cuda")
    out = torch.zeros(1, H, d, device="cuda")
    lse = torch.zeros(1, H, device="cuda")
    ws = S.make_workspace(kv, N)
    S.retrieve(kv, q[0], 1.0, N, idx, n_sel, delta, out, lse, ws)
    assert S.last_error() == 0
    gi, gn, gd, go, gl = [x.cpu().numpy() for x in (idx, n_sel, delta, out, lse)]
    for h in range(H):
        K, V = P.widen(kb[0, h], "bf16"), P.widen(vb[0, h], "bf16")
        sc = P.scores(P.widen(qb[0, h], "bf16"), K, 1.0)
        ref = P.top_n(sc, N)
        assert gn[0, h] == N
        assert (gi[0, h] == ref).all(), (h, np.flatnonzero(gi[0, h] != ref)[:5])
        assert abs(gd[0, h] - P.dropped_mass(sc, ref)) <= DELTA_TOL
        ro, rl = P.attention(P.widen(qb[0, h], "bf16"), K, V, ref, 1.0)
        assert np.abs(go[0, h] - ro).max() <= OUT_TOL and abs(gl[0, h] - rl) <= LSE_TOL, h


# --------------------------------------------------------------------------- #
# CIS gate and dilation
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("n_sink,window,n_den", [(0, 0, 0), (4, 64, 0), (4, 64, 2)])
def test_cis_dilate_cluster(n_sink, window, n_den):
    """Few heads with long anchor rows: the gate's dilation split over a
    cluster of CTAs per head (4096 entries, 4 CTAs of 1024; budgeted dilation
    keeps one CTA). A full row, a row of 1500 entries (the last two CTAs
    empty) and a row of 3000 with runs of adjacent anchors across the CTAs'
    boundaries and anchors inside the forced window, against the oracle's
    (budgeted) dilation joined with the forced keys."""
    import sparse_kv_selection_gb300 as S
    from workloads import bf16_bits_from_f32
    from workloads.torch_io import tensor_of
    rng = np.random.default_rng(5)
    B, H, t, acap, w, d = 1, 3, 40000, 4096, 3, 128
    cap = min(t, acap * (2 * w + 1) + n_sink + window)
    k = torch.zeros(B, H, t, d, dtype=torch.bfloat16, device="cuda")
    kv = S.KVCache(k, k, torch.tensor([t], dtype=torch.int32, device="cuda"), H)
    q = rng.normal(size=(B, H, d)).astype(np.float32)
    qa = q + 0.05 * rng.normal(size=(B, H, d)).astype(np.float32)   # cosine near 0.999: reuse
    an = np.array([[4096, 1500, 3000]], np.int32)
    aidx = np.zeros((B, H, acap), np.int32)
    aidx[0, 0] = np.sort(rng.choice(t, size=4096, replace=False))
    aidx[0, 1, :1500] = np.sort(rng.choice(t, size=1500, replace=False))
    third = set(rng.choice(t - 200, size=2900, replace=False).tolist())
    third = sorted(third)[:2900]
    third = np.array(third, np.int64)
    third[1015:1035] = third[1015] + np.arange(20)           # a run across entry 1024
    third = np.unique(np.concatenate([third, np.arange(t - 100, t)]))[:3000]
    an[0, 2] = len(third)
    aidx[0, 2, :len(third)] = np.sort(third)
    idx = torch.full((B, H, cap), -4, dtype=torch.int32, device="cuda")
    n_sel = torch.full((B, H), -4, dtype=torch.int32, device="cuda")
    reuse = torch.full((B, H), 9, dtype=torch.uint8, device="cuda")
    S.cis_dilate(kv, torch.from_numpy(aidx).cuda(), torch.from_numpy(an).cuda(),
                 tensor_of(bf16_bits_from_f32(q), "bf16", "cuda"),
                 tensor_of(bf16_bits_from_f32(qa), "bf16", "cuda"), w, 0.8, idx, n_sel, reuse,
                 n_sink=n_sink, window=window, n_den=n_den)
    assert S.last_error() == 0
    gi, gn, gr = idx.cpu().numpy(), n_sel.cpu().numpy(), reuse.cpu().numpy()
    for h in range(H):
        assert gr[0, h] == 1, h
        anc = aidx[0, h, :an[0, h]]
        shared = P.dilate(anc, w, t) if n_den == 0 else P.dilate_budget(anc, w, t, len(anc) // n_den)
        ref = np.union1d(P.forced_set(t, n_sink, window), shared)
        assert gn[0, h] == len(ref), (h, gn[0, h], len(ref))
        assert (gi[0, h, :gn[0, h]] == ref).all(), h


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_cis_dilate(dtype, d):
    import sparse_kv_selection_gb300 as S
    from workloads import bf16_bits_from_f32
    from workloads.torch_io import tensor_of
    rng = np.random.default_rng(11)
    B, H, t, acap, w = 3, 8, 333, 40, 3
    cap = min(t, acap * (2 * w + 1))
    k = torch.zeros(B, H, t, d, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                    device="cuda")
    lens = np.array([333, 57, 200], np.int32)
    kv = S.KVCache(k, k, torch.from_numpy(lens).cuda(), H)
    q = rng.normal(size=(B, H, d))
    target = np.linspace(0.5, 0.99, B * H).reshape(B, H)
    target[0, 0], target[0, 1] = 0.8, 0.80001
    orth = rng.normal(size=(B, H, d))
    orth -= (orth * q).sum(-1, keepdims=True) / (q * q).sum(-1, keepdims=True) * q
    qa = (target[..., None] * q / np.linalg.norm(q, axis=-1, keepdims=True)
          + np.sqrt(1 - target[..., None] ** 2) * orth / np.linalg.norm(orth, axis=-1, keepdims=True))
    qa[2, 7] = 0.0                       # zero-norm anchor query: never shares
    store = (lambda x: x.astype(np.float32)) if dtype == "f32" else bf16_bits_from_f32
    qs, qas = store(q.astype(np.float32)), store(qa.astype(np.float32))
    an = rng.integers(0, acap + 1, size=(B, H)).astype(np.int32)
    an[1, 2] = 0                         # no anchor yet: never shares
    aidx = np.zeros((B, H, acap), np.int32)
    for b in range(B):
        for h in range(H):
            n_ = min(an[b, h], lens[b])
            an[b, h] = n_
            aidx[b, h, :n_] = np.sort(rng.choice(lens[b], size=n_, replace=False))
    aidx[0, 3, :an[0, 3]] = np.arange(lens[0] - an[0, 3], lens[0])   # runs into the end
    idx = torch.full((B, H, cap), -4, dtype=torch.int32, device="cuda")
    n_sel = torch.full((B, H), -4, dtype=torch.int32, device="cuda")
    reuse = torch.full((B, H), 9, dtype=torch.uint8, device="cuda")
    S.cis_dilate(kv, torch.from_numpy(aidx).cuda(), torch.from_numpy(an).cuda(),
                 tensor_of(qs, dtype, "cuda"), tensor_of(qas, dtype, "cuda"), w, 0.8, idx, n_sel,
                 reuse)
    gi, gn, gr = idx.cpu().numpy(), n_sel.cpu().numpy(), reuse.cpu().numpy()
    for b in range(B):
        for h in range(H):
            qv, qav = P.widen(qs[b, h], dtype), P.widen(qas[b, h], dtype)
            c, want = P.cis_gate(qv, qav, 0.8)
            want = want and an[b, h] > 0
            if c is not None and abs(c - 0.8) < GATE_GAP:
                continue
            assert bool(gr[b, h]) == want, (b, h, c)
            if want:
                ref = P.dilate(aidx[b, h, :an[b, h]], w, int(lens[b]))
                assert gn[b, h] == len(ref) and gi[b, h, :gn[b, h]].tolist() == ref.tolist()
            else:
                assert gn[b, h] == -4 and (gi[b, h] == -4).all()


@pytest.mark.parametrize("w,n_den,n_sink,window", [(2, 1, 0, 0), (2, 2, 0, 0), (3, 5, 0, 0), (1, 3, 0, 0),
                                                    (4, 2, 0, 0), (0, 2, 0, 0), (2, 3, 4, 16),
                                                    (3, 1, 2, 0), (2, 4, 0, 9)])
def test_cis_dilate_budget(w, n_den, n_sink, window):
    """Budgeted dilation (Fig. 9a): every reusing head's set against the
    oracle's dilate_budget with m = floor(anchor_n / n_den), united with
    the forced keys; anchor rows of every size, some running into either
    end of the cache, some over 1024 entries (several passes of the kernel)."""
    import sparse_kv_selection_gb300 as S
    rng = np.random.default_rng(31 + w + 7 * n_den)
    B, H, d, acap = 2, 6, 64, 1500
    lens = np.array([3000, 700], np.int32)
    t_max = int(lens.max())
    cap = min(t_max, acap * (2 * w + 1) + n_sink + window)
    k = torch.zeros(B, H, t_max, d, device="cuda")
    kv = S.KVCache(k, k, torch.from_numpy(lens).cuda(), H)
    q = torch.from_numpy(rng.normal(size=(B, H, d)).astype(np.float32)).cuda()
    an = np.zeros((B, H), np.int32)
    aidx = np.zeros((B, H, acap), np.int32)
    sizes = [1, 7, 300, 1100, 1500, 40]
    for b in range(B):
        t = int(lens[b])
        lo, hi = min(n_sink, t), max(min(n_sink, t), t - window)   # anchors avoid the forced keys
        for h in range(H):
            n_ = min(sizes[h], hi - lo, acap)
            an[b, h] = n_
            if h == 5:      # runs into both ends of the middle range
                row = np.concatenate([np.arange(lo, lo + n_ // 2), np.arange(hi - (n_ - n_ // 2), hi)])
            else:
                row = np.sort(lo + rng.choice(hi - lo, size=n_, replace=False))
            aidx[b, h, :n_] = row
    idx = torch.full((B, H, cap), -4, dtype=torch.int32, device="cuda")
    n_sel = torch.full((B, H), -4, dtype=torch.int32, device="cuda")
    reuse = torch.zeros((B, H), dtype=torch.uint8, device="cuda")
    S.cis_dilate(kv, torch.from_numpy(aidx).cuda(), torch.from_numpy(an).cuda(), q, q, w, 0.8, idx,
                 n_sel, reuse, n_sink=n_sink, window=window, n_den=n_den)
    assert S.last_error() == 0
    gi, gn = idx.cpu().numpy(), n_sel.cpu().numpy()
    assert reuse.cpu().numpy().all()
    for b in range(B):
        t = int(lens[b])
        for h in range(H):
            A = aidx[b, h, :an[b, h]].astype(np.int64)
            want = np.union1d(P.forced_set(t, n_sink, window),
                              P.dilate_budget(A, w, t, len(A) // n_den))
            assert gn[b, h] == len(want), (b, h, gn[b, h], len(want))
            assert gi[b, h, :gn[b, h]].tolist() == want.tolist(), (b, h)


@pytest.mark.parametrize("name,n_den", [("mha_bf16_ragged", 2), ("gqa4_bf16", 4), ("paged_bf16", 1),
                                        ("f32_d64_gqa2", 3)])
def test_decode_budgeted_dilation(name, n_den):
    """Decode with budgeted dilation against the oracle, free-running and
    teacher-forced."""
    S, wl, dev, kv = _setup(name)
    compared, r = compare_decode(wl, dev, kv, _heads(wl), n_den=n_den)
    assert compared >= len(_heads(wl)) * wl.steps // 2 and r[1:].any()
    compared = compare_decode_forced(wl, dev, kv, _heads(wl), n_den=n_den)
    assert compared >= len(_heads(wl)) * wl.steps - 2, compared


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
@pytest.mark.parametrize("gap", [1e-3, 2e-4, 5e-5, 1e-6, 1e-9, 1e-11])
def test_cis_gate_near_threshold(dtype, d, gap):
    """tau placed `gap` below or above each head's float64 cosine: gaps past
    1e-4 are decided from the fp32 sums, nearer ones by the float64 formula;
    every decision must be the oracle's."""
    import sparse_kv_selection_gb300 as S
    from workloads import bf16_bits_from_f32
    from workloads.torch_io import tensor_of
    rng = np.random.default_rng(17)
    B, H, t, acap, w = 1, 16, 64, 4, 1
    k = torch.zeros(B, H, t, d, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                    device="cuda")
    kv = S.KVCache(k, k, torch.full((B,), t, dtype=torch.int32, device="cuda"), H)
    store = (lambda x: x.astype(np.float32)) if dtype == "f32" else bf16_bits_from_f32
    q = rng.normal(size=(B, H, d)).astype(np.float32)
    qa = (q + 0.6 * rng.normal(size=(B, H, d))).astype(np.float32)
    qs, qas = store(q), store(qa)
    cos = np.array([[P.cosine(P.widen(qs[0, h], dtype), P.widen(qas[0, h], dtype))
                     for h in range(H)]])
    an = np.full((B, H), acap, np.int32)
    aidx = np.tile(np.arange(0, 4 * acap, 4, dtype=np.int32), (B, H, 1))
    for sign in (-1.0, 1.0):
        for h in range(H):
            tau = float(cos[0, h] + sign * gap)
            reuse = torch.full((B, H), 9, dtype=torch.uint8, device="cuda")
            idx = torch.zeros((B, H, t), dtype=torch.int32, device="cuda")
            n_sel = torch.zeros((B, H), dtype=torch.int32, device="cuda")
            S.cis_dilate(kv, torch.from_numpy(aidx).cuda(), torch.from_numpy(an).cuda(),
                         tensor_of(qs, dtype, "cuda"), tensor_of(qas, dtype, "cuda"), w, tau, idx,
                         n_sel, reuse)
            c, want = P.cis_gate(P.widen(qs[0, h], dtype), P.widen(qas[0, h], dtype), tau)
            assert bool(reuse[0, h].item()) == want == (sign < 0), (h, sign, c, tau)


# --------------------------------------------------------------------------- #
# whole decode loop
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("max_run", [1, 2, 3])
def test_decode_max_run_matches_oracle(max_run):
    """CIS block size s as a bound on consecutive reuses (Tables IV/V/VIII)."""
    S, wl, dev, kv = _setup("gqa4_bf16")
    compared, r = compare_decode(wl, dev, kv, _heads(wl), max_run=max_run)
    assert compared >= len(_heads(wl)) * wl.steps // 2
    if max_run == 1:
        assert not r.any()
    else:  # no head reuses more than max_run - 1 times in a row
        run = np.zeros(r.shape[1:], int)
        for s in range(r.shape[0]):
            run = np.where(r[s] != 0, run + 1, 0)
            assert (run <= max_run - 1).all()


@pytest.mark.parametrize("name", list(CASES))
def test_decode_matches_oracle(name):
    S, wl, dev, kv = _setup(name)
    compared, r = compare_decode(wl, dev, kv, _heads(wl))
    assert compared >= len(_heads(wl)) * wl.steps // 2
    assert r[1:].any() or wl.steps < 3   # some head reused its anchor


# --------------------------------------------------------------------------- #
# the split entry points and graph capture of the decode step
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_step_ties_flat_and_budgets(dtype):
    """First decode step (every head retrieves) on caches whose logits tie
    heavily (keys drawn from 7 rows), are all equal, or are fewer than the
    budget, and with a zero budget: the set must be the oracle's exactly,
    ties going to the lowest index."""
    import sparse_kv_selection_gb300 as S
    from workloads import bf16_bits_from_f32
    from workloads.torch_io import tensor_of
    rng = np.random.default_rng(23)
    B, H, d, tmax = 4, 2, 128, 1500
    lens = np.array([1500, 300, 1000, 800], np.int32)
    budget = np.array([100, 400, 0, 257], np.int32)
    store = (lambda x: x.astype(np.float32)) if dtype == "f32" else bf16_bits_from_f32
    base = rng.normal(size=(H, 7, d)).astype(np.float32)
    K = np.zeros((B, H, tmax, d), np.float32)
    K[0] = base[:, np.arange(tmax) % 7]                  # 7 distinct logits per head
    K[1] = rng.normal(size=(H, 1, d)).astype(np.float32)  # budget above the length
    K[2] = rng.normal(size=(H, tmax, d))                  # zero budget
    K[3] = base[:, :1]                                    # one logit value: flat
    V = rng.normal(size=(B, H, tmax, d)).astype(np.float32)
    q = rng.normal(size=(B, H, d)).astype(np.float32)
    Ks, Vs, qs = store(K), store(V), store(q)
    kv = S.KVCache(tensor_of(Ks, dtype, "cuda"), tensor_of(Vs, dtype, "cuda"),
                   torch.from_numpy(lens).cuda(), H)
    scale = d ** -0.5
    dec = S.SparseDecoder(kv, n_budget=torch.from_numpy(budget), w=1, tau=0.8, scale=scale)
    o, l, dl, r, n = dec.alloc_outputs(1)
    dec.step(tensor_of(qs, dtype, "cuda"), o[0], l[0], dl[0], r[0], n[0])
    gi = dec.idx.cpu().numpy()
    o, l, dl, n = o[0].cpu().numpy(), l[0].cpu().numpy(), dl[0].cpu().numpy(), n[0].cpu().numpy()
    ai, an = dec.anchor_idx.cpu().numpy(), dec.anchor_n.cpu().numpy()
    assert S.last_error() == 0
    for b in range(B):
        for h in range(H):
            t = int(lens[b])
            Kb = P.widen(Ks[b, h, :t], dtype)
            Vb = P.widen(Vs[b, h, :t], dtype)
            qv = P.widen(qs[b, h], dtype)
            if budget[b] == 0:
                assert n[b, h] == 0 and an[b, h] == 0 and dl[b, h] == 1.0
                assert (o[b, h] == 0).all() and l[b, h] == -math.inf
                continue
            sc = P.scores(qv, Kb, scale)
            Sx = P.top_n(sc, int(budget[b]))
            assert n[b, h] == len(Sx) == an[b, h], (b, h)
            assert gi[b, h, :len(Sx)].tolist() == Sx.tolist(), (b, h)
            assert ai[b, h, :len(Sx)].tolist() == Sx.tolist(), (b, h)
            assert abs(dl[b, h] - P.dropped_mass(sc, Sx)) <= DELTA_TOL, (b, h)
            ro, rl = P.attention(qv, Kb, Vb, Sx, scale)
            assert np.abs(o[b, h] - ro).max() <= OUT_TOL and abs(l[b, h] - rl) <= LSE_TOL, (b, h)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("max_run", [0, 3])
def test_decode_teacher_forced(name, max_run):
    S, wl, dev, kv = _setup(name)
    compared = compare_decode_forced(wl, dev, kv, _heads(wl), max_run=max_run)
    assert compared >= len(_heads(wl)) * wl.steps - 2, compared


@pytest.mark.parametrize("name", ["mha_bf16_ragged", "gqa4_bf16", "paged_bf16", "f32_d64_gqa2"])
def test_set_mass_matches_oracle(name):
    """Dropped mass of given sets (the reuse-step diagnostic): top-N sets,
    their dilations, random sets, the empty set and the whole cache."""
    S, wl, dev, kv = _setup(name)
    rng = np.random.default_rng(29)
    cap = wl.t_max
    idx = np.zeros((wl.B, wl.Hq, cap), np.int32)
    n = np.zeros((wl.B, wl.Hq), np.int32)
    sets = {}
    for b, h in _heads(wl):
        K, _ = kv_rows64(wl, b, h // wl.G)
        t = K.shape[0]
        sc = P.scores(q64(wl, 2, b, h), K, wl.scale)
        kind = (b * wl.Hq + h) % 5
        if kind == 0:
            Sx = P.top_n(sc, int(wl.budget[b]))
        elif kind == 1:
            Sx = P.dilate(P.top_n(sc, int(wl.budget[b])), wl.w, t)
        elif kind == 2:
            Sx = np.sort(rng.choice(t, size=int(rng.integers(1, t)), replace=False))
        elif kind == 3:
            Sx = np.zeros(0, np.int64)
        else:
            Sx = np.arange(t)
        sets[(b, h)] = Sx
        idx[b, h, :len(Sx)] = Sx
        n[b, h] = len(Sx)
    delta = torch.full((wl.B, wl.Hq), -1.0, device="cuda")
    ws = S.make_workspace(kv, cap)
    S.set_mass(kv, dev["q"][2], wl.scale, torch.from_numpy(idx).cuda(), torch.from_numpy(n).cuda(),
               delta, ws)
    dl = delta.cpu().numpy()
    for b, h in _heads(wl):
        K, _ = kv_rows64(wl, b, h // wl.G)
        want = P.dropped_mass(P.scores(q64(wl, 2, b, h), K, wl.scale), sets[(b, h)])
        assert abs(dl[b, h] - want) <= DELTA_TOL, (b, h, dl[b, h], want)


@pytest.mark.parametrize("name", ["gqa4_bf16", "mha_bf16_ragged", "paged_bf16", "f32_d64_gqa2",
                                  "bf16_long_gqa2"])
def test_score_then_select_and_score_select(name):
    """prhs_score followed by prhs_select, and prhs_score_select (one launch
    computing the logits in shared memory when the cache is short), each
    against the oracle: the top-N set up to near-ties and the dropped mass."""
    S, wl, dev, kv = _setup(name)
    nb = dev["budget"] if len(set(wl.budget.tolist())) > 1 else None
    N = 0 if nb is not None else int(wl.budget[0])   # N is not read with per-sequence budgets
    cap = int(wl.budget.max())
    for split in (False, True):
        idx = torch.full((wl.B, wl.Hq, cap), -1, dtype=torch.int32, device="cuda")
        n_sel = torch.zeros(wl.B, wl.Hq, dtype=torch.int32, device="cuda")
        delta = torch.zeros(wl.B, wl.Hq, device="cuda")
        ws = S.make_workspace(kv, cap)
        if split:
            S.binding.score(kv, dev["q"][3], wl.scale, ws)
            S.binding.select(kv, dev["q"][3], N, idx, n_sel, delta, ws, n_budget=nb)
        else:
            S.score_select(kv, dev["q"][3], wl.scale, N, idx, n_sel, delta, ws, n_budget=nb)
        assert S.last_error() == 0
        gi, gn, gd = idx.cpu().numpy(), n_sel.cpu().numpy(), delta.cpu().numpy()
        for b, h in _heads(wl):
            K, _ = kv_rows64(wl, b, h // wl.G)
            sc = P.scores(q64(wl, 3, b, h), K, wl.scale)
            gset = gi[b, h, :gn[b, h]]
            check_topn(gset, sc, int(wl.budget[b]))
            assert abs(gd[b, h] - P.dropped_mass(sc, gset)) <= DELTA_TOL, (split, b, h)


@pytest.mark.parametrize("name", ["mha_bf16_ragged", "paged_bf16"])
def test_decode_step_in_cuda_graph_matches_eager(name):
    """prhs_decode_step forks onto a side stream; captured in a CUDA graph and
    replayed, it must give the eager results bit for bit."""
    S, wl, dev, kv = _setup(name)
    nb = dev["budget"] if len(set(wl.budget.tolist())) > 1 else None
    N = None if nb is not None else int(wl.budget[0])

    def run(graph):
        dec = S.SparseDecoder(kv, N=N, n_budget=nb, w=wl.w, tau=wl.tau, scale=wl.scale)
        outs = dec.alloc_outputs(wl.steps)
        stream = torch.cuda.Stream()
        if not graph:
            with torch.cuda.stream(stream):
                dec.run(dev["q"], outs)
        else:
            with torch.cuda.stream(stream):   # eager warm-up resolves per-device state
                dec.run(dev["q"], dec.alloc_outputs(wl.steps))
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                dec.reset()
                dec.run(dev["q"], outs)
            g.replay()
        torch.cuda.synchronize()
        return [x.cpu() for x in outs]

    eager, graphed = run(False), run(True)
    for a, b in zip(eager, graphed):
        assert torch.equal(a.nan_to_num(), b.nan_to_num())


def test_decode_step_max_heads_and_empty_cache():
    """The largest batch the library takes (B * Hq = 16384 query heads) through
    one decode step, with some sequences' caches empty: sampled heads against
    the oracle, empty caches give an empty set, out = 0, lse = -inf, delta = 0."""
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload
    B, Hq = 512, 32
    wl = make_workload("maxheads", dtype="bf16", B=B, Hq=Hq, Hkv=Hq, d=64, t=(20, 48), t_max=48,
                       n_clusters=2, width=(2, 4), steps=1, N=6, w=1, seed=13)
    dev = upload(wl)
    lens = wl.seq_lens.copy()
    lens[::97] = 0                                    # a few empty caches
    kv = S.KVCache(dev["k"], dev["v"], torch.from_numpy(lens).cuda(), Hq)
    dec = S.SparseDecoder(kv, N=6, w=1, tau=wl.tau, scale=wl.scale)
    o, l, dl, r, n = dec.alloc_outputs(1)
    dec.step(dev["q"][0], o[0], l[0], dl[0], r[0], n[0])
    gi = dec.idx.cpu().numpy()
    o, l, dl, n = o[0].cpu().numpy(), l[0].cpu().numpy(), dl[0].cpu().numpy(), n[0].cpu().numpy()
    assert S.last_error() == 0
    rng = np.random.default_rng(3)
    heads = [(int(b), int(h)) for b, h in zip(rng.integers(0, B, 48), rng.integers(0, Hq, 48))]
    heads += [(0, 0), (97, 5), (B - 1, Hq - 1)]
    for b, h in heads:
        t = int(lens[b])
        if t == 0:
            assert n[b, h] == 0 and dl[b, h] == 0.0 and (o[b, h] == 0).all() and l[b, h] == -math.inf
            continue
        K, V = kv_rows64(wl, b, h)
        K, V = K[:t], V[:t]
        qv = q64(wl, 0, b, h)
        sc = P.scores(qv, K, wl.scale)
        gset = gi[b, h, :n[b, h]]
        check_topn(gset, sc, 6)
        assert abs(dl[b, h] - P.dropped_mass(sc, gset)) <= DELTA_TOL, (b, h)
        ro, rl = P.attention(qv, K, V, gset, wl.scale)
        assert np.abs(o[b, h] - ro).max() <= OUT_TOL and abs(l[b, h] - rl) <= LSE_TOL, (b, h)


def test_launch_counts():
    """Kernels per call, read from the library's launch counter: prhs_score_select
    is one launch on a short cache and two (score, select) on a long one; a
    decode step adds the gate, the two attention branches, and the compose and
    set-mass launches when keys are forced."""
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload

    def count(fn):
        c0 = S.binding.launch_count()
        fn()
        torch.cuda.synchronize()
        return S.binding.launch_count() - c0

    for t, fused in ((1000, True), (8192, True), (9000, False)):
        wl = make_workload("lc", dtype="bf16", B=1, Hq=2, Hkv=2, d=128, t=t, n_clusters=8, steps=1,
                           N=64, w=1, seed=5)
        dev = upload(wl)
        kv = S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq)
        idx = torch.zeros(1, 2, 64, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, 2, dtype=torch.int32, device="cuda")
        dl = torch.zeros(1, 2, device="cuda")
        ws = S.make_workspace(kv, 64 * 3 + 16)
        assert count(lambda: S.score_select(kv, dev["q"][0], wl.scale, 64, idx, n, dl, ws)) == (1 if fused else 2)
        o = torch.zeros(1, 2, 128, device="cuda")
        lse = torch.zeros(1, 2, device="cuda")
        # retrieval: one launch on a short cache, else score, select and attention
        assert count(lambda: S.retrieve(kv, dev["q"][0], wl.scale, 64, idx, n, dl, o, lse, ws)) == (1 if fused else 3)
        ss = 1 if fused else 2
        for n_sink, window in ((0, 0), (2, 8)):
            dec = S.SparseDecoder(kv, N=64, w=1, tau=wl.tau, scale=wl.scale, n_sink=n_sink, window=window)
            # gate and side attention, then the retrieval: one launch, or score (+ select),
            # compose and set mass for forced keys, and attention
            want = 3 if fused and not n_sink else 2 + ss + (2 if n_sink else 0) + 1
            assert count(lambda: dec.step(dev["q"][0])) == want, (t, n_sink)
        assert S.last_error() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_retrieve(name):
    """prhs_retrieve against the oracle: for the heads not flagged, the top-N
    set (up to near-ties), delta and the attention over the set; flagged
    heads' rows untouched."""
    S, wl, dev, kv = _setup(name)
    nb = dev["budget"] if len(set(wl.budget.tolist())) > 1 else None
    N = 0 if nb is not None else int(wl.budget[0])
    cap = int(wl.budget.max())
    g = torch.Generator().manual_seed(7)
    skip = (torch.rand(wl.B, wl.Hq, generator=g) < 0.4).to(torch.uint8)
    skip.view(-1)[0] = 0
    idx = torch.full((wl.B, wl.Hq, cap), -7, dtype=torch.int32, device="cuda")
    n_sel = torch.full((wl.B, wl.Hq), -7, dtype=torch.int32, device="cuda")
    delta = torch.full((wl.B, wl.Hq), -7.0, device="cuda")
    out = torch.full((wl.B, wl.Hq, wl.d), -7.0, device="cuda")
    lse = torch.full((wl.B, wl.Hq), -7.0, device="cuda")
    ws = S.make_workspace(kv, cap)
    S.retrieve(kv, dev["q"][2], wl.scale, N, idx, n_sel, delta, out, lse, ws, n_budget=nb,
               head_skip=skip.cuda())
    assert S.last_error() == 0
    gi, gn, gd, go, gl = [x.cpu().numpy() for x in (idx, n_sel, delta, out, lse)]
    sk = skip.numpy()
    for b, h in _heads(wl):
        if sk[b, h]:
            assert gn[b, h] == -7 and gd[b, h] == -7.0 and (go[b, h] == -7.0).all() and gl[b, h] == -7.0
            assert (gi[b, h] == -7).all()
            continue
        K, V = kv_rows64(wl, b, h // wl.G)
        qv = q64(wl, 2, b, h)
        sc = P.scores(qv, K, wl.scale)
        gset = gi[b, h, :gn[b, h]]
        check_topn(gset, sc, int(wl.budget[b]))
        assert abs(gd[b, h] - P.dropped_mass(sc, gset)) <= DELTA_TOL, (b, h)
        ro, rl = P.attention(qv, K, V, gset, wl.scale)
        assert np.abs(go[b, h] - ro).max() <= OUT_TOL and abs(gl[b, h] - rl) <= LSE_TOL, (b, h)


@pytest.mark.parametrize("t,N,budget_zero", [(300, 400, False), (300, 300, False), (300, 64, True),
                                             (6000, 6000, False)])
def test_retrieve_whole_and_empty_sets(t, N, budget_zero):
    """A budget of at least t keeps every key (delta = 0, attention over the
    whole cache); a zero budget and an empty cache give the empty set,
    out = 0 and lse = -inf."""
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload
    wl = make_workload("whole", dtype="bf16", B=3, Hq=2, Hkv=1, d=128, t=t, n_clusters=6, steps=1,
                       N=N, w=1, seed=11)
    dev = upload(wl)
    lens = torch.from_numpy(wl.seq_lens.copy()).cuda()
    lens[2] = 0                                        # an empty cache
    kv = S.KVCache(dev["k"], dev["v"], lens, wl.Hq)
    nb = torch.tensor([N, 0 if budget_zero else N, N], dtype=torch.int32, device="cuda")
    cap = min(N, t)
    idx = torch.zeros(3, 2, cap, dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(3, 2, dtype=torch.int32, device="cuda")
    delta = torch.full((3, 2), -1.0, device="cuda")
    out = torch.full((3, 2, 128), 5.0, device="cuda")
    lse = torch.zeros(3, 2, device="cuda")
    ws = S.make_workspace(kv, cap)
    S.retrieve(kv, dev["q"][0], wl.scale, 0, idx, n_sel, delta, out, lse, ws, n_budget=nb)
    assert S.last_error() == 0
    gi, gn, gd, go, gl = [x.cpu().numpy() for x in (idx, n_sel, delta, out, lse)]
    for b in range(3):
        for h in range(2):
            tb = int(lens[b])
            nbud = int(nb[b])
            if tb == 0 or nbud == 0:
                assert gn[b, h] == 0 and (go[b, h] == 0).all() and gl[b, h] == -math.inf
                assert gd[b, h] == (0.0 if tb == 0 else 1.0)
                continue
            K, V = kv_rows64(wl, b, 0)
            qv = q64(wl, 0, b, h)
            sc = P.scores(qv, K, wl.scale)
            gset = gi[b, h, :gn[b, h]]
            if nbud >= tb:
                assert gset.tolist() == list(range(tb)) and gd[b, h] == 0.0
            else:
                check_topn(gset, sc, nbud)
                assert abs(gd[b, h] - P.dropped_mass(sc, gset)) <= DELTA_TOL
            ro, rl = P.attention(qv, K, V, gset, wl.scale)
            assert np.abs(go[b, h] - ro).max() <= OUT_TOL and abs(gl[b, h] - rl) <= LSE_TOL, (b, h)


@pytest.mark.parametrize("name,n_sink,window", [("gqa4_bf16", 0, 0), ("mha_bf16_ragged", 4, 32),
                                                ("bf16_9k_mha", 4, 64), ("paged_bf16", 2, 16)])
def test_retrieve_anchors_and_forced_keys(name, n_sink, window):
    """prhs_retrieve with the anchor buffers and forced keys: the attended set
    is the forced keys with the top N of the keys between them, delta its
    dropped mass and out/lse the attention over it; the anchor row holds the
    ranked part only, anchor_n its size and q_anchor the query."""
    S, wl, dev, kv = _setup(name)
    N = int(wl.budget.min())
    nb = None
    if len(set(wl.budget.tolist())) > 1:
        nb = dev["budget"]
    cap = int(wl.budget.max()) + n_sink + window
    acap = int(wl.budget.max())
    i32 = dict(dtype=torch.int32, device="cuda")
    idx = torch.full((wl.B, wl.Hq, cap), -1, **i32)
    n_sel = torch.zeros(wl.B, wl.Hq, **i32)
    delta = torch.zeros(wl.B, wl.Hq, device="cuda")
    out = torch.zeros(wl.B, wl.Hq, wl.d, device="cuda")
    lse = torch.zeros(wl.B, wl.Hq, device="cuda")
    aidx = torch.full((wl.B, wl.Hq, acap), -1, **i32)
    an = torch.zeros(wl.B, wl.Hq, **i32)
    qa = torch.zeros_like(dev["q"][1])
    ws = S.make_workspace(kv, cap)
    S.retrieve(kv, dev["q"][1], wl.scale, 0 if nb is not None else N, idx, n_sel, delta, out, lse, ws,
               n_budget=nb, anchor_idx=aidx, anchor_n=an, q_anchor=qa, n_sink=n_sink, window=window)
    assert S.last_error() == 0
    gi, gn, gd, go, gl, ga, gan = [x.cpu().numpy() for x in (idx, n_sel, delta, out, lse, aidx, an)]
    assert torch.equal(qa, dev["q"][1])
    for b, h in _heads(wl):
        t = int(wl.seq_lens[b])
        K, V = kv_rows64(wl, b, h // wl.G)
        qv = q64(wl, 1, b, h)
        sc = P.scores(qv, K, wl.scale)
        nbud = int(wl.budget[b])
        ranked = ga[b, h, :gan[b, h]]
        forced = P.forced_set(t, n_sink, window)
        mid = t - len(forced)
        assert len(ranked) == min(nbud, mid)
        if len(ranked) < mid:  # the ranked part against the middle keys' top N, up to near-ties
            lo = min(n_sink, t)
            check_topn(ranked - lo, sc[lo:lo + mid], nbud)
        gset = gi[b, h, :gn[b, h]]
        want = np.union1d(forced, ranked)
        assert gset.tolist() == want.tolist(), (b, h)
        assert abs(gd[b, h] - P.dropped_mass(sc, gset)) <= DELTA_TOL, (b, h)
        ro, rl = P.attention(qv, K, V, gset, wl.scale)
        assert np.abs(go[b, h] - ro).max() <= OUT_TOL and abs(gl[b, h] - rl) <= LSE_TOL, (b, h)
