"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each ``check_*`` helper reads the oracle functions through the module object
at call time, so the mutation tests at the bottom can plant a plausible
mistake in the oracle and confirm that some pin catches it.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle.prhs as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


# --------------------------------------------------------------------------- #
# pin helpers
# --------------------------------------------------------------------------- #
def check_softmax_hand():
    g = _read_golden("softmax_hand.txt")
    s = np.log(np.array(g["logits_exp"]))
    assert np.allclose(P.softmax(s), g["weights"], rtol=0, atol=1e-15)
    assert abs(P.logsumexp(s) - math.log(g["lse_exp"][0])) < 1e-14
    S = P.top_n(s, int(g["N"][0]))
    assert S.tolist() == [int(x) for x in g["topN"]]
    assert abs(P.dropped_mass(s, S) - g["delta"][0]) < 1e-15


def check_softmax_invariants(rng):
    s = rng.normal(size=257) * 5
    A = P.softmax(s)
    assert abs(A.sum() - 1.0) < 1e-12 and (A >= 0).all()
    assert np.allclose(P.softmax(s + 123.0), A, rtol=1e-12, atol=0)   # shift invariance
    # the largest logit gets the largest weight
    assert A.argmax() == s.argmax()


def check_topn_bruteforce(rng):
    """delta(top-N) is the minimum over every size-N subset (t <= 12)."""
    for t in (1, 5, 9, 12):
        for trial in range(4):
            s = rng.normal(size=t) * 2
            if trial == 3:
                s = np.round(s)                  # force ties
            for N in range(1, t + 1):
                S = P.top_n(s, N)
                assert len(S) == N and np.all(np.diff(S) > 0)
                d = P.dropped_mass(s, S)
                best = min(P.dropped_mass(s, np.array(c)) for c in
                           itertools.combinations(range(t), N))
                assert d <= best + 1e-15
                # ties go to the lowest index: among the optimal subsets it is the
                # lexicographically smallest one once sorted by descending logit
                optimal = [c for c in itertools.combinations(range(t), N)
                           if P.dropped_mass(s, np.array(c)) <= best + 1e-15]
                if trial == 3:
                    thr = np.sort(s)[::-1][N - 1]
                    above = set(np.nonzero(s > thr)[0])
                    ties = sorted(np.nonzero(s == thr)[0])
                    expect = sorted(above | set(ties[:N - len(above)]))
                    assert S.tolist() == expect
                    assert tuple(expect) in optimal


def check_topn_ties():
    s = np.array([1.0, 3.0, 3.0, 2.0, 3.0])
    assert P.top_n(s, 2).tolist() == [1, 2]
    assert P.top_n(s, 4).tolist() == [1, 2, 3, 4]
    assert P.top_n(np.zeros(7), 3).tolist() == [0, 1, 2]
    assert P.top_n(np.array([0.0, -0.0, 0.0]), 1).tolist() == [0]
    assert P.top_n(s, 5).tolist() == [0, 1, 2, 3, 4]
    assert P.top_n(s, 9).tolist() == [0, 1, 2, 3, 4]


def check_delta_properties(rng):
    s = rng.normal(size=300) * 3
    t = s.size
    assert P.dropped_mass(s, np.arange(t)) == 0.0
    assert abs(P.dropped_mass(s, np.array([], np.int64)) - 1.0) < 1e-12
    prev = 1.0
    for N in (1, 10, 50, 150, 299, 300):
        d = P.dropped_mass(s, P.top_n(s, N))
        assert 0.0 <= d <= 1.0 and d <= prev + 1e-15
        prev = d
    # delta = 1 - exp(lse_S - lse_full), with lse_S from the attention routine
    K = rng.normal(size=(t, 16))
    V = rng.normal(size=(t, 16))
    q = rng.normal(size=16)
    sc = P.scores(q, K, 0.25)
    S = P.top_n(sc, 40)
    _, lse_S = P.attention(q, K, V, S, 0.25)
    _, lse_F = P.dense_attention(q, K, V, 0.25)
    assert abs(P.dropped_mass(sc, S) - (1.0 - math.exp(lse_S - lse_F))) < 1e-12


def check_attention_identities(rng):
    t, d = 200, 32
    K = rng.normal(size=(t, d))
    V = rng.normal(size=(t, d))
    q = rng.normal(size=d)
    scale = 1 / math.sqrt(d)
    o_all, l_all = P.attention(q, K, V, np.arange(t), scale)
    o_d, l_d = P.dense_attention(q, K, V, scale)
    assert np.allclose(o_all, o_d, atol=1e-14) and abs(l_all - l_d) < 1e-14
    # convex split: o_full = (1 - delta) o_S + delta o_Sc; lse_full = logaddexp
    sc = P.scores(q, K, scale)
    S = P.top_n(sc, 37)
    Sc = np.setdiff1d(np.arange(t), S)
    oS, lS = P.attention(q, K, V, S, scale)
    oC, lC = P.attention(q, K, V, Sc, scale)
    delta = P.dropped_mass(sc, S)
    assert np.allclose(o_d, (1 - delta) * oS + delta * oC, atol=1e-13)
    assert abs(l_d - np.logaddexp(lS, lC)) < 1e-13
    # equal keys -> uniform weights -> mean of V; lse = s + log t
    Ke = np.tile(rng.normal(size=d), (t, 1))
    oe, le = P.dense_attention(q, Ke, V, scale)
    assert np.allclose(oe, V.mean(0), atol=1e-13)
    assert abs(le - (scale * Ke[0] @ q + math.log(t))) < 1e-12
    # one dominant key -> its value row
    Kd = K.copy()
    Kd[17] = 200.0 * q / np.linalg.norm(q)
    od, _ = P.dense_attention(q, Kd, V, scale)
    assert np.allclose(od, V[17], atol=1e-9)


def check_attention_vs_torch_sdpa(rng):
    torch = pytest.importorskip("torch")
    B, H, t, d = 2, 3, 97, 64
    q = rng.normal(size=(B, H, 1, d))
    K = rng.normal(size=(B, H, t, d))
    V = rng.normal(size=(B, H, t, d))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(K), torch.from_numpy(V)).numpy()
    for b in range(B):
        for h in range(H):
            o, _ = P.dense_attention(q[b, h, 0], K[b, h], V[b, h], 1 / math.sqrt(d))
            assert np.allclose(o, ref[b, h, 0], atol=1e-12)
    # restricted to a subset = SDPA with a boolean mask
    S = np.array([3, 4, 5, 40, 41, 90])
    mask = np.zeros((1, 1, 1, t), bool)
    mask[..., S] = True
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(K), torch.from_numpy(V),
        attn_mask=torch.from_numpy(mask)).numpy()
    o, _ = P.attention(q[1, 2, 0], K[1, 2], V[1, 2], S, 1 / math.sqrt(d))
    assert np.allclose(o, ref[1, 2, 0], atol=1e-12)


def check_dilation_golden():
    g = _read_golden("fig4_dilation.txt")
    out = P.dilate(np.array(g["input"], np.int64), int(g["w"][0]), int(g["t"][0]))
    assert out.tolist() == [int(x) for x in g["expected"]]


def check_dilation_bruteforce(rng):
    for trial in range(60):
        t = int(rng.integers(1, 80))
        n = int(rng.integers(0, t + 1))
        w = int(rng.integers(0, 6))
        S = np.sort(rng.choice(t, size=n, replace=False))
        out = P.dilate(S, w, t)
        ref = sorted({j for i in S for j in range(i - w, i + w + 1) if 0 <= j < t})
        assert out.tolist() == ref
        assert set(S.tolist()) <= set(out.tolist())
        assert len(out) <= min(t, n * (2 * w + 1))
        if w == 0:
            assert out.tolist() == S.tolist()
    # a contiguous run [a, b] -> [max(0, a - w), min(t - 1, b + w)]
    assert P.dilate(np.arange(1, 4), 3, 10).tolist() == list(range(0, 7))
    assert P.dilate(np.arange(7, 10), 2, 10).tolist() == list(range(5, 10))


def check_cosine_gate(rng):
    scipy_dist = pytest.importorskip("scipy.spatial.distance")
    for _ in range(20):
        a, b = rng.normal(size=64), rng.normal(size=64)
        assert abs(P.cosine(a, b) - (1 - scipy_dist.cosine(a, b))) < 1e-13
    q = rng.normal(size=32)
    assert P.cis_gate(q, q, 0.8)[1] and abs(P.cosine(q, q) - 1) < 1e-15
    c, r = P.cis_gate(q, -q, 0.8)
    assert not r and abs(c + 1) < 1e-15
    assert P.cis_gate(np.zeros(4), np.ones(4), -2.0) == (None, False)
    # boundary: cosine exactly equal to tau triggers sharing (">=")
    assert P.cis_gate(np.array([1.0, 0.0]), np.array([0.8, 0.6]), 0.8)[1]
    assert not P.cis_gate(np.array([1.0, 0.0]), np.array([0.6, 0.8]), 0.8)[1]


def check_decode_schedule(rng):
    t, d, N, w = 120, 16, 10, 1
    K = rng.normal(size=(t, d))
    V = rng.normal(size=(t, d))
    qs = rng.normal(size=(6, d))
    sc = 1 / math.sqrt(d)
    # tau above 1: every step retrieves its own top-N
    rec = P.decode_head(qs, K, V, N, w, 1.5, sc)
    for q, r in zip(qs, rec):
        assert not r.reuse
        assert r.S.tolist() == P.top_n(P.scores(q, K, sc), N).tolist()
        assert abs(r.delta - r.delta_used) < 1e-15
    # tau below -1: step 0 retrieves, later steps share its dilated set
    rec = P.decode_head(qs, K, V, N, w, -1.5, sc)
    S0 = P.top_n(P.scores(qs[0], K, sc), N)
    assert not rec[0].reuse and rec[0].S.tolist() == S0.tolist()
    for r in rec[1:]:
        assert r.reuse and r.S.tolist() == P.dilate(S0, w, t).tolist()
        assert r.anchor_S.tolist() == S0.tolist()
    # attended output of each step equals attention over the attended set
    for q, r in zip(qs, rec):
        o, l = P.attention(q, K, V, r.S, sc)
        assert np.allclose(o, r.out) and abs(l - r.lse) < 1e-14


def check_max_run(rng):
    t, d, N, w = 90, 16, 8, 1
    K = rng.normal(size=(t, d))
    V = rng.normal(size=(t, d))
    qs = rng.normal(size=(7, d))
    sc = 1 / math.sqrt(d)
    # s = 1: every query retrieves even with every gate open
    assert not any(r.reuse for r in P.decode_head(qs, K, V, N, w, -1.5, sc, max_run=1))
    # s = 2 with every gate open: retrieve, reuse, retrieve, reuse, ...
    pat = [r.reuse for r in P.decode_head(qs, K, V, N, w, -1.5, sc, max_run=2)]
    assert pat == [False, True, False, True, False, True, False]
    # s = 3: two reuses per retrieval; a retrieval resets the count
    pat = [r.reuse for r in P.decode_head(qs, K, V, N, w, -1.5, sc, max_run=3)]
    assert pat == [False, True, True, False, True, True, False]
    # unbounded equals a bound longer than the sequence
    a = [r.reuse for r in P.decode_head(qs, K, V, N, w, 0.2, sc)]
    b = [r.reuse for r in P.decode_head(qs, K, V, N, w, 0.2, sc, max_run=50)]
    assert a == b


def check_gate_target_hand():
    """Four queries whose schedule differs by which query each is gated
    against: the anchor (the last query that retrieved), not the previous
    query, and the anchor moves on every retrieval. The expected flags and
    sets are derived by hand in tests/golden/cis_schedule_hand.txt."""
    g = _read_golden("cis_schedule_hand.txt")
    a = np.radians(g["key_angles_deg"])
    K = g["key_norm"][0] * np.stack([np.cos(a), np.sin(a)], axis=1)
    b = np.radians(g["query_angles_deg"])
    qs = np.stack([np.cos(b), np.sin(b)], axis=1)
    V = np.arange(2 * len(a), dtype=np.float64).reshape(len(a), 2)
    rec = P.decode_head(qs, K, V, int(g["N"][0]), int(g["w"][0]), g["tau"][0], 1.0)
    assert [int(r.reuse) for r in rec] == [int(x) for x in g["reuse"]]
    for s, r in enumerate(rec):
        assert r.S.tolist() == [int(x) for x in g[f"S{s}"]], s
        assert r.anchor_S.tolist() == [int(x) for x in g[f"anchor{s}"]], s
        if not r.reuse:   # a one-key set attends exactly that key's value row
            assert np.allclose(r.out, V[r.S[0]], atol=0)


def _hand_gqa_workload():
    """Hq = 8 query heads over Hkv = 2 KV heads (group 4), t = 4, d = 2:
    KV head 0's dominant key (along e1) is key 0, KV head 1's is key 3, and
    every query is e1. Under the grouped layout query heads 0-3 read KV head 0
    and heads 4-7 read KV head 1, so their top-1 sets are {0} x4 then {3} x4."""
    from workloads import Workload
    K = np.zeros((1, 2, 4, 2), np.float32)
    K[0, 0] = [[5, 0], [1, 0], [0, 1], [-1, 0]]
    K[0, 1] = [[-1, 0], [0, 1], [1, 0], [5, 0]]
    V = np.zeros_like(K)
    V[0, 0, :, 0] = [10, 11, 12, 13]
    V[0, 1, :, 0] = [20, 21, 22, 23]
    q = np.zeros((1, 1, 8, 2), np.float32)
    q[..., 0] = 1.0
    return Workload(name="hand_gqa", dtype="f32", B=1, Hq=8, Hkv=2, d=2,
                    seq_lens=np.array([4], np.int32), t_max=4, paged=False, block_size=16,
                    block_table=None, K=K, V=V, q=q, budget=np.array([1], np.int32), w=0,
                    tau=0.8, scale=1.0, steps=1, seed=0)


def check_head_map_hand():
    res = P.decode_workload(_hand_gqa_workload())
    sets = [res[(0, h)][0].S.tolist() for h in range(8)]
    assert sets == [[0]] * 4 + [[3]] * 4, sets
    outs = [res[(0, h)][0].out[0] for h in range(8)]
    assert outs == [10.0] * 4 + [23.0] * 4, outs


def check_dilate_budget_hand():
    g = _read_golden("budget_dilation_hand.txt")
    ints = lambda k: [int(x) for x in g[k]]
    for case, ms in (("a", (0, 1, 3, 4, 5, 8)), ("b", (3,)), ("c", (2,))):
        S = np.array(ints(f"{case}_S"), np.int64)
        w, t = int(g[f"{case}_w"][0]), int(g[f"{case}_t"][0])
        for m in ms:
            assert P.dilate_budget(S, w, t, m).tolist() == ints(f"{case}_m{m}"), (case, m)
    # more than every candidate: the full +-w dilation
    S = np.array(ints("a_S"), np.int64)
    assert P.dilate_budget(S, 2, 30, 10 ** 6).tolist() == P.dilate(S, 2, 30).tolist()


def check_dilate_budget_bruteforce(rng):
    """Invariants against a distance computed by brute force: S kept, only
    +-w neighbours added, min(m, candidates) of them, each added position
    nearer (lower at equal distance) than every candidate left out, and the
    sets nested in m."""
    for trial in range(80):
        t = int(rng.integers(1, 60))
        n = int(rng.integers(0, min(t, 12) + 1))
        w = int(rng.integers(0, 5))
        S = np.sort(rng.choice(t, size=n, replace=False))
        full = set(P.dilate(S, w, t).tolist())
        cand = sorted(full - set(S.tolist()))
        prev = set(S.tolist())
        for m in range(0, len(cand) + 2):
            out = P.dilate_budget(S, w, t, m).tolist()
            assert out == sorted(set(out)) and set(S.tolist()) <= set(out) <= full
            added = set(out) - set(S.tolist())
            assert len(added) == min(m, len(cand))
            key = lambda p: (min(abs(p - a) for a in S.tolist()), p)
            left = set(cand) - added
            if added and left:
                assert max(key(p) for p in added) < min(key(p) for p in left)
            assert prev <= set(out)
            prev = set(out)


def check_decode_budget(rng):
    """A reusing query attends the anchor set with floor(|anchor| / n_den)
    dilated positions (every gate open, so every later query reuses)."""
    t, d, N, w = 150, 16, 12, 2
    K = rng.normal(size=(t, d))
    V = rng.normal(size=(t, d))
    qs = rng.normal(size=(4, d))
    sc = 1 / math.sqrt(d)
    for n_den in (1, 3, 5, 100):
        rec = P.decode_head(qs, K, V, N, w, -1.5, sc, n_den=n_den)
        S0 = rec[0].S
        assert len(S0) == N
        for r in rec[1:]:
            assert r.reuse
            assert len(r.S) == N + min(N // n_den, len(P.dilate(S0, w, t)) - N)
            assert set(S0.tolist()) <= set(r.S.tolist()) <= set(P.dilate(S0, w, t).tolist())
    full = P.decode_head(qs, K, V, N, w, -1.5, sc)
    assert all(a.S.tolist() == b.S.tolist() for a, b in zip(full, P.decode_head(qs, K, V, N, w, -1.5, sc, n_den=0)))


def check_key_gate_hand():
    """The "Key" similarity design (Table IX) on a growing cache: the gate
    compares the key each query appends with the anchor's appended key.
    d = 2, t0 = 4 visible keys, four queries. Every query is e1 (gating on
    queries would reuse at every step after the first); the appended keys
    point at 0, 30, 90 and 110 degrees: cos(30, 0) = 0.866 -> reuse;
    cos(90, 0) = 0 -> retrieve, the anchor becomes query 2 (key at 90);
    cos(110, 90) = 0.94 -> reuse. Flags: retrieve, reuse, retrieve, reuse."""
    t0 = 4
    ang = np.radians([0.0, 30.0, 90.0, 110.0])
    K = np.zeros((t0 + 4, 2))
    K[:t0] = [[1.0, 0.0], [0.0, 1.0], [-1.0, 0.0], [0.0, -1.0]]
    K[t0:] = np.stack([np.cos(ang), np.sin(ang)], axis=1)
    V = np.arange(2 * (t0 + 4), dtype=np.float64).reshape(t0 + 4, 2)
    qs = np.tile([1.0, 0.0], (4, 1))
    rec = P.decode_head_grow(qs, K, V, t0, 2, 1, 0.8, 1.0, 0, 0, gate="key")
    assert [r.reuse for r in rec] == [False, True, False, True]
    byq = P.decode_head_grow(qs, K, V, t0, 2, 1, 0.8, 1.0, 0, 0, gate="query")
    assert [r.reuse for r in byq] == [False, True, True, True]


def check_widen():
    bits = np.array([0x3F80, 0xC020, 0x0000, 0x8000, 0x7F7F], np.uint16)
    v = P.widen(bits, "bf16")
    assert v[0] == 1.0 and v[1] == -2.5 and v[2] == 0.0 and v[4] == 3.3895313892515355e38
    assert P.widen(np.array([0.1], np.float32), "f32")[0] == float(np.float32(0.1))


def check_forced_set():
    """Sinks and window clipped to [0, t): hand cases."""
    assert P.forced_set(10, 2, 3).tolist() == [0, 1, 7, 8, 9]
    assert P.forced_set(3, 2, 3).tolist() == [0, 1, 2]
    assert P.forced_set(10, 0, 0).tolist() == []
    assert P.forced_set(10, 12, 0).tolist() == list(range(10))
    assert P.forced_set(10, 0, 1).tolist() == [9]
    assert P.forced_set(0, 2, 3).tolist() == []


def check_top_n_between(rng):
    """The N best keys outside the forced set: brute force over subsets of
    the middle keys (the lowest-index subset among the optimal ones)."""
    for t in (5, 8, 11):
        for n_sink, window in ((0, 0), (1, 2), (2, 3), (4, 4)):
            s = rng.normal(size=t) * 2
            s[rng.integers(0, t)] = s[rng.integers(0, t)]  # a tie
            mid = [i for i in range(t) if i >= n_sink and i < t - window]
            for N in range(1, len(mid) + 2):
                got = P.top_n_between(s, N, n_sink, window).tolist()
                if N >= len(mid):
                    assert got == mid
                    continue
                best = None
                for sub in itertools.combinations(mid, N):
                    key = (-np.exp(s[list(sub)]).sum(), sub)
                    if best is None or key < best:
                        best = key
                # equal sums only at exact ties: compare the kept mass
                assert abs(np.exp(s[got]).sum() + best[0]) < 1e-12, (t, n_sink, window, N)
                assert set(got).isdisjoint(P.forced_set(t, n_sink, window).tolist())


def check_decode_grow(rng):
    """Growing-cache decode: the forced keys are always attended, retrieving
    steps keep |F| + min(N, |middle|) keys and no N-subset of the middle
    drops less mass, reuse steps attend F with the dilated anchor, the
    anchor never holds forced keys; the first step with no forced keys is
    decode_head's on the visible rows; a budget covering the cache is dense."""
    d, t0, steps, w = 8, 9, 6, 1
    K = rng.normal(size=(t0 + steps, d))
    V = rng.normal(size=(t0 + steps, d))
    qs = rng.normal(size=(steps, d))
    qs[1:] = qs[0] + 0.05 * rng.normal(size=(steps - 1, d))    # reuse after step 0
    qs[3] = -qs[0]                                              # then retrieve again
    for n_sink, window, N in ((2, 2, 3), (1, 3, 2), (0, 0, 4)):
        rec = P.decode_head_grow(qs, K, V, t0, N, w, 0.8, d ** -0.5, n_sink, window,
                                 keep_scores=True)
        assert [r.reuse for r in rec][:4] == [False, True, True, False]
        for st, r in enumerate(rec):
            t = t0 + st + 1
            F = P.forced_set(t, n_sink, window)
            assert np.all(np.diff(r.S) > 0) and r.S.min() >= 0 and r.S.max() < t
            assert set(F.tolist()) <= set(r.S.tolist())
            assert set(r.anchor_S.tolist()).isdisjoint(F.tolist()) or (n_sink == 0 and window == 0)
            if r.reuse:
                want = np.union1d(F, P.dilate(r.anchor_S, w, t))
                assert r.S.tolist() == want.tolist()
            else:
                mid = [i for i in range(t) if i >= n_sink and i < t - window]
                assert len(r.S) == len(F) + min(N, len(mid))
                for sub in itertools.combinations(mid, min(N, len(mid))):
                    alt = np.union1d(F, list(sub)).astype(np.int64)
                    assert r.delta <= P.dropped_mass(r.scores, alt) + 1e-12
        if n_sink == 0 and window == 0:
            first = P.decode_head(qs[:1], K[:t0 + 1], V[:t0 + 1], N, w, 0.8, d ** -0.5)[0]
            assert rec[0].S.tolist() == first.S.tolist()
            assert np.allclose(rec[0].out, first.out, atol=1e-14) and abs(rec[0].lse - first.lse) < 1e-14
    big = P.decode_head_grow(qs[:1], K, V, t0, 100, w, 0.8, d ** -0.5, 2, 2)[0]
    do, dl = P.dense_attention(qs[0], K[:t0 + 1], V[:t0 + 1], d ** -0.5)
    assert big.S.tolist() == list(range(t0 + 1)) and big.delta == 0.0
    assert np.allclose(big.out, do, atol=1e-14) and abs(big.lse - dl) < 1e-14


# --------------------------------------------------------------------------- #
# tests
# --------------------------------------------------------------------------- #
@pytest.fixture
def rng():
    return np.random.default_rng(1234)


def test_softmax_hand():
    check_softmax_hand()


def test_softmax_invariants(rng):
    check_softmax_invariants(rng)


def test_topn_bruteforce(rng):
    check_topn_bruteforce(rng)


def test_topn_ties():
    check_topn_ties()


def test_delta_properties(rng):
    check_delta_properties(rng)


def test_attention_identities(rng):
    check_attention_identities(rng)


def test_attention_vs_torch_sdpa(rng):
    check_attention_vs_torch_sdpa(rng)


def test_dilation_golden():
    check_dilation_golden()


def test_dilation_bruteforce(rng):
    check_dilation_bruteforce(rng)


def test_cosine_gate(rng):
    check_cosine_gate(rng)


def test_decode_schedule(rng):
    check_decode_schedule(rng)


def test_widen():
    check_widen()


def test_max_run(rng):
    check_max_run(rng)


# --------------------------------------------------------------------------- #
# planted mistakes: each must be caught by at least one pin
# --------------------------------------------------------------------------- #
def _caught(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def test_mutation_topn_highest_index_ties(monkeypatch, rng):
    def bad(s, N):
        s = np.asarray(s, np.float64)
        if N >= s.size:
            return np.arange(s.size)
        order = np.argsort(-s[::-1], kind="stable")
        return np.sort(s.size - 1 - order[:N])
    monkeypatch.setattr(P, "top_n", bad)
    assert _caught(check_topn_ties)


def test_mutation_topn_off_by_one(monkeypatch, rng):
    good = P.top_n
    monkeypatch.setattr(P, "top_n", lambda s, N: good(s, max(N - 1, 0)) if N < len(s) else good(s, N))
    assert _caught(check_softmax_hand) and _caught(check_topn_bruteforce, rng)


def test_mutation_delta_retained(monkeypatch):
    good = P.dropped_mass
    monkeypatch.setattr(P, "dropped_mass", lambda s, S: 1.0 - good(s, S))
    assert _caught(check_softmax_hand)


def test_mutation_scores_missing_scale(monkeypatch, rng):
    monkeypatch.setattr(P, "scores", lambda q, K, scale: np.asarray(K) @ np.asarray(q))
    assert _caught(check_delta_properties, rng)


def test_mutation_attention_unnormalised(monkeypatch, rng):
    good = P.attention

    def bad(q, K, V, S, scale):
        o, l = good(q, K, V, S, scale)
        return o * len(S), l
    monkeypatch.setattr(P, "attention", bad)
    assert _caught(check_attention_identities, rng)


def test_mutation_attention_transposed_value(monkeypatch, rng):
    """Weights applied to K instead of V must fail the SDPA pin."""
    good = P.attention
    monkeypatch.setattr(P, "attention", lambda q, K, V, S, scale: good(q, K, K, S, scale))
    assert _caught(check_attention_vs_torch_sdpa, rng)


def test_mutation_dilation_radius(monkeypatch):
    good = P.dilate
    monkeypatch.setattr(P, "dilate", lambda S, w, t: good(S, max(w - 1, 0), t))
    assert _caught(check_dilation_golden)


def test_mutation_dilation_no_clip(monkeypatch, rng):
    def bad(S, w, t):
        return np.array(sorted({j for i in S for j in range(i - w, i + w + 1) if j >= 0}))
    monkeypatch.setattr(P, "dilate", bad)
    assert _caught(check_dilation_bruteforce, rng)


def test_mutation_gate_strict(monkeypatch):
    good = P.cosine

    def bad(q, qa, tau):
        c = good(q, qa)
        return c, (c is not None and c > tau)
    monkeypatch.setattr(P, "cis_gate", bad)
    assert _caught(check_cosine_gate, np.random.default_rng(0))


def test_mutation_max_run_off_by_one(monkeypatch, rng):
    good = P.decode_head

    def bad(q_steps, K, V, N, w, tau, scale, keep_scores=False, max_run=0):
        return good(q_steps, K, V, N, w, tau, scale, keep_scores, max_run + 1 if max_run else 0)
    monkeypatch.setattr(P, "decode_head", bad)
    assert _caught(check_max_run, rng)


def test_mutation_gate_sign(monkeypatch):
    good = P.cosine
    monkeypatch.setattr(P, "cosine", lambda q, qa: None if good(q, qa) is None else -good(q, qa))
    assert _caught(check_cosine_gate, np.random.default_rng(0))


def test_forced_set():
    check_forced_set()


def test_top_n_between(rng):
    check_top_n_between(rng)


def test_decode_grow(rng):
    check_decode_grow(rng)


def test_mutation_window_off_by_one(monkeypatch, rng):
    orig = P.forced_set
    monkeypatch.setattr(P, "forced_set", lambda t, n, wdw: orig(t, n, wdw + 1))
    assert _caught(check_forced_set)


def test_mutation_forced_keys_ranked(monkeypatch, rng):
    monkeypatch.setattr(P, "top_n_between", lambda s, N, n, wdw: P.top_n(s, N))
    assert _caught(check_top_n_between, rng)


def test_mutation_anchor_holds_forced(monkeypatch, rng):
    orig = P.top_n_between
    monkeypatch.setattr(P, "top_n_between",
                        lambda s, N, n, wdw: np.union1d(orig(s, N, n, wdw), P.forced_set(len(s), n, wdw)))
    assert _caught(check_decode_grow, rng)


def test_gate_target_hand():
    check_gate_target_hand()


def test_head_map_hand():
    check_head_map_hand()


def _schedule_variant(gate_previous=False, keep_first_anchor_query=False):
    """decode_head with one planted mistake in its schedule: gating against
    the previous query instead of the anchor, or never moving the anchor
    query after the first retrieval."""
    def bad(q_steps, K, V, N, w, tau, scale, keep_scores=False, max_run=0):
        K = np.asarray(K, np.float64)
        V = np.asarray(V, np.float64)
        t = K.shape[0]
        anchor_S = anchor_q = prev_q = None
        rec = []
        for q in np.asarray(q_steps, np.float64):
            ref_q = prev_q if gate_previous else anchor_q
            c, reuse = (None, False) if anchor_S is None else P.cis_gate(q, ref_q, tau)
            s = P.scores(q, K, scale)
            delta = None
            if reuse:
                S = P.dilate(anchor_S, w, t)
            else:
                S = P.top_n(s, N)
                delta = P.dropped_mass(s, S)
                anchor_S = S
                if anchor_q is None or not keep_first_anchor_query:
                    anchor_q = q
            prev_q = q
            out, lse = P.attention(q, K, V, S, scale)
            rec.append(P.HeadStep(reuse=reuse, cos=c, S=S, anchor_S=anchor_S, delta=delta,
                                  delta_used=P.dropped_mass(s, S), s_nth=None, out=out, lse=lse))
        return rec
    return bad


def test_mutation_gate_against_previous_query(monkeypatch):
    monkeypatch.setattr(P, "decode_head", _schedule_variant(gate_previous=True))
    assert _caught(check_gate_target_hand)


def test_mutation_anchor_query_not_moved(monkeypatch):
    monkeypatch.setattr(P, "decode_head", _schedule_variant(keep_first_anchor_query=True))
    assert _caught(check_gate_target_hand)


def test_schedule_variant_without_mistake_passes(monkeypatch):
    """The hand-written variant above is itself correct when no mistake is
    planted, so the two mutation tests fail for the planted reason only."""
    monkeypatch.setattr(P, "decode_head", _schedule_variant())
    check_gate_target_hand()


def test_mutation_head_map_modulo(monkeypatch):
    """Query head h reading KV head h % Hkv (interleaved grouping) instead of
    h // G (consecutive grouping)."""
    def bad(wl, heads=None, steps=None, keep_scores=False, max_run=0):
        heads = [(b, h) for b in range(wl.B) for h in range(wl.Hq)] if heads is None else heads
        res = {}
        for b, hq in heads:
            kvh = hq % wl.Hkv
            K = P.widen(wl.logical_rows("K", b, kvh), wl.dtype)
            V = P.widen(wl.logical_rows("V", b, kvh), wl.dtype)
            qs = P.widen(wl.q[:wl.steps, b, hq], wl.dtype)
            res[(b, hq)] = P.decode_head(qs, K, V, int(wl.budget[b]), wl.w, wl.tau, wl.scale)
        return res
    monkeypatch.setattr(P, "decode_workload", bad)
    assert _caught(check_head_map_hand)


def test_dilate_budget_hand():
    check_dilate_budget_hand()


def test_dilate_budget_bruteforce(rng):
    check_dilate_budget_bruteforce(rng)


def test_decode_budget(rng):
    check_decode_budget(rng)


def test_key_gate_hand():
    check_key_gate_hand()


def test_mutation_budget_farthest_first(monkeypatch):
    """Adding the farthest neighbours first must fail the hand cases."""
    def bad(S, w, t, m):
        S = np.asarray(S, np.int64)
        cand = sorted(set(P.dilate(S, w, t).tolist()) - set(S.tolist()),
                      key=lambda p: (-min(abs(p - a) for a in S.tolist()), p))
        return np.sort(np.concatenate([S, np.asarray(cand[:max(0, m)], np.int64)]))
    monkeypatch.setattr(P, "dilate_budget", bad)
    assert _caught(check_dilate_budget_hand)


def test_mutation_budget_highest_position_first(monkeypatch):
    def bad(S, w, t, m):
        S = np.asarray(S, np.int64)
        cand = sorted(set(P.dilate(S, w, t).tolist()) - set(S.tolist()),
                      key=lambda p: (min(abs(p - a) for a in S.tolist()), -p))
        return np.sort(np.concatenate([S, np.asarray(cand[:max(0, m)], np.int64)]))
    monkeypatch.setattr(P, "dilate_budget", bad)
    assert _caught(check_dilate_budget_hand)


def test_mutation_key_gate_uses_query(monkeypatch):
    """Gating on the queries while asked for keys must fail the hand case."""
    good = P.decode_head_grow

    def bad(*args, gate="query", **kw):
        return good(*args, gate="query", **kw)
    monkeypatch.setattr(P, "decode_head_grow", bad)
    assert _caught(check_key_gate_hand)


def test_mutation_budget_from_budget_not_anchor(monkeypatch, rng):
    """m taken from a fixed 2 N instead of the anchor's size must fail."""
    good = P.shared_set
    monkeypatch.setattr(P, "shared_set",
                        lambda a, w, t, n_den: good(a, w, t, n_den) if n_den <= 0 else
                        P.dilate_budget(a, w, t, 2 * len(a) // n_den))
    assert _caught(check_decode_budget, rng)
