"""fp64 restatement of the PrHS decode path (test infrastructure only).

Source throughout: "Near-Oracle KV Selection via Pre-hoc Sparsity for
Long-Context Inference" (arXiv 2602.08329), abstract, Table I (notation),
Fig. 2, Fig. 4, Fig. 8, Fig. 9, Table VIII. The pages print no formula; each
function states the plain definition it takes and the reading behind it.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


# --------------------------------------------------------------------------- #
# input decoding
# --------------------------------------------------------------------------- #
def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored float32 values or bfloat16 bit patterns -> exact float64."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    bits = np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- #
# attention weights (Table I: A(.), K, q, d)
# --------------------------------------------------------------------------- #
def scores(q: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """Attention logits s_i = scale * <q, k_i> for every cached key i.

    Table I names the attention weight A(.) over the KV cache; the scaled dot
    product with scale = 1/sqrt(d) is the standard transformer logit (reading:
    no positional rotation is applied, the synthetic keys are post-position).
    """
    return scale * (np.asarray(K, np.float64) @ np.asarray(q, np.float64))


def softmax(s: np.ndarray) -> np.ndarray:
    """A_i = exp(s_i - m) / sum_j exp(s_j - m), m = max_j s_j (Table I, A(.))."""
    s = np.asarray(s, np.float64)
    e = np.exp(s - s.max())
    return e / e.sum()


def logsumexp(s: np.ndarray) -> float:
    """Natural-log partition function: m + log sum_i exp(s_i - m)."""
    s = np.asarray(s, np.float64)
    m = s.max()
    return float(m + np.log(np.exp(s - m).sum()))


# --------------------------------------------------------------------------- #
# top-N oracle selector and dropped mass (abstract; Table I S, S_t, N, tau, delta)
# --------------------------------------------------------------------------- #
def top_n(s: np.ndarray, N: int) -> np.ndarray:
    """Index set S_t of the N largest logits, returned in ascending order.

    The abstract's "top-k oracle" keeps the N (Table I: KV budget N) keys with
    the largest attention weights; ranking by the logit gives the same order
    as ranking by A_i. Reading: ties go to the lowest index; N >= t keeps all.
    """
    s = np.asarray(s, np.float64)
    t = s.shape[0]
    if N >= t:
        return np.arange(t, dtype=np.int64)
    order = np.argsort(-s, kind="stable")     # stable: equal logits keep index order
    return np.sort(order[:N])


def dropped_mass(s: np.ndarray, S: np.ndarray) -> float:
    """delta(S) = sum of the attention weights A_i of the keys i not in S.

    Abstract: "the attention mass of discarded entries"; Table I: tau(.) the
    retained mass and delta(.) = 1 - tau(.) the dropped mass. Summed over
    the complement directly (not as 1 - tau) so small masses keep precision.
    """
    A = softmax(s)
    keep = np.zeros(A.shape[0], bool)
    keep[np.asarray(S, np.int64)] = True
    return float(A[~keep].sum())


# --------------------------------------------------------------------------- #
# critical-index-set reuse (Fig. 2, Fig. 4, Fig. 8, Table VIII)
# --------------------------------------------------------------------------- #
def cosine(q: np.ndarray, qa: np.ndarray) -> float | None:
    """Cosine similarity <q, qa> / (|q| |qa|); None when either norm is 0."""
    q = np.asarray(q, np.float64)
    qa = np.asarray(qa, np.float64)
    den = np.sqrt(q @ q) * np.sqrt(qa @ qa)
    if den == 0.0:
        return None
    return float((q @ qa) / den)


def cis_gate(q: np.ndarray, qa: np.ndarray, tau: float) -> tuple[float | None, bool]:
    """Share the anchor's critical-index set iff sim(q, q_a) >= tau.

    Fig. 8 defines triggering as sim(q, q') >= tau; Fig. 2 and Table VIII use
    tau = 0.8. Reading: a zero-norm query never shares.
    """
    c = cosine(q, qa)
    return c, (c is not None and c >= tau)


def dilate(S: np.ndarray, w: int, t: int) -> np.ndarray:
    """Dilated set: union over i in S of [i - w, i + w], clipped to [0, t).

    Fig. 4 ("Critical-index set (CIS) dilation") widens the shared set around
    its indices so that neighbouring keys of a cluster are covered for later
    queries; Table VIII's radius r (r = 2 raises the average processed tokens
    from 131 to 167) is read as this +/- w. Result sorted, without repeats,
    not truncated back to N.
    """
    mask = np.zeros(t, bool)
    for i in np.asarray(S, np.int64):
        mask[max(0, i - w):min(t, i + w + 1)] = True
    return np.nonzero(mask)[0].astype(np.int64)


def dilate_budget(S: np.ndarray, w: int, t: int, m: int) -> np.ndarray:
    """Budgeted dilation: S and at most m of its +/- w neighbours.

    Fig. 9a varies the "dilation strength" m = floor(k / n_den) (a smaller
    n_den dilates more). Reading: k is the size of the shared set S and m
    the number of positions dilation may add to it; the candidates are the
    positions of dilate(S, w, t) not in S, taken nearest to S first and, at
    equal distance, lowest position first. m >= all candidates gives
    dilate(S, w, t); m = 0 gives S itself (direct reuse). Result ascending.
    """
    S = np.asarray(S, np.int64)
    full = dilate(S, w, t)
    inS = np.zeros(t, bool)
    inS[S] = True
    cand = [p for p in full.tolist() if not inS[p]]
    if S.size:
        dist = {p: int(np.min(np.abs(S - p))) for p in cand}
    else:
        dist = {}
    cand.sort(key=lambda p: (dist[p], p))
    keep = cand[:max(0, m)]
    return np.sort(np.concatenate([S, np.asarray(keep, np.int64)])).astype(np.int64)


# --------------------------------------------------------------------------- #
# attention over a selected set (abstract; Table V caption, sparse kernel)
# --------------------------------------------------------------------------- #
def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, S: np.ndarray,
              scale: float) -> tuple[np.ndarray, float]:
    """Exact softmax attention restricted to the keys in S.

    out = sum_{i in S} p_i v_i with p_i = exp(s_i - lse_S) and
    lse_S = log sum_{i in S} exp(s_i) (weights renormalised over S).
    """
    S = np.asarray(S, np.int64)
    s = scale * (np.asarray(K, np.float64)[S] @ np.asarray(q, np.float64))
    m = s.max()
    p = np.exp(s - m)
    l = p.sum()
    out = (p @ np.asarray(V, np.float64)[S]) / l
    return out, float(m + np.log(l))


def dense_attention(q, K, V, scale):
    """Attention over every cached key (the dense baseline of Table IV)."""
    return attention(q, K, V, np.arange(np.asarray(K).shape[0]), scale)


# --------------------------------------------------------------------------- #
# multi-step decode with CIS reuse
# --------------------------------------------------------------------------- #
@dataclass
class HeadStep:
    reuse: bool                 # this step shared the anchor's set
    cos: float | None           # sim(q_s, q_anchor); None on step 0 / zero norm
    S: np.ndarray               # index set attended at this step (ascending)
    anchor_S: np.ndarray        # anchor's undilated top-N set after this step
    delta: float | None         # dropped mass of the fresh top-N set (fresh steps)
    delta_used: float           # dropped mass of S under the current query
    s_nth: float | None         # N-th largest logit (fresh steps, N < t)
    out: np.ndarray             # attention output over S
    lse: float
    scores: np.ndarray | None = None


def shared_set(anchor_S: np.ndarray, w: int, t: int, n_den: int) -> np.ndarray:
    """The set a reusing query attends: the anchor's set dilated by +/- w
    (Fig. 4, Table VIII), or with n_den > 0 the budgeted dilation of Fig. 9a
    with m = floor(|anchor set| / n_den) added positions."""
    if n_den > 0:
        return dilate_budget(anchor_S, w, t, len(anchor_S) // n_den)
    return dilate(anchor_S, w, t)


def decode_head(q_steps: np.ndarray, K: np.ndarray, V: np.ndarray, N: int, w: int,
                tau: float, scale: float, keep_scores: bool = False,
                max_run: int = 0, n_den: int = 0) -> list[HeadStep]:
    """One head through a sequence of decode queries with CIS reuse.

    Reading of Fig. 4 ("critical tokens from query 405 are shared to queries
    406 and 407") and Fig. 8 (pairs (q, q') for which sharing triggers): the
    first query retrieves; a later query whose similarity to the last
    retrieving query (the anchor) is >= tau attends the anchor's top-N set
    dilated by +/- w; otherwise it retrieves and becomes the new anchor.
    Dilation is applied to the anchor set once, never compounded.

    max_run > 0 reads the CIS block size s of Tables IV, V and VIII ("CIS-8",
    "CIS-16") as the most consecutive queries one retrieval may serve: after
    s - 1 reuses the next query retrieves whatever its similarity. 0 = no
    bound. Parity unpinned beyond its two limits (s = 1 always retrieves;
    s = 2 with every gate open alternates), which the tests check.

    n_den > 0 bounds the dilation (shared_set, Fig. 9a).
    """
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    t = K.shape[0]
    anchor_S = None
    anchor_q = None
    rec = []
    age = 0  # reuses since the anchor retrieved
    for q in np.asarray(q_steps, np.float64):
        c, reuse = (None, False) if anchor_S is None else cis_gate(q, anchor_q, tau)
        if max_run > 0 and age >= max_run - 1:
            reuse = False
        age = age + 1 if reuse else 0
        s = scores(q, K, scale)
        delta = s_nth = None
        if reuse:
            S = shared_set(anchor_S, w, t, n_den)
        else:
            S = top_n(s, N)
            delta = dropped_mass(s, S)
            if N < t:
                s_nth = float(np.sort(s)[::-1][N - 1])
            anchor_S, anchor_q = S, q
        out, lse = attention(q, K, V, S, scale)
        rec.append(HeadStep(reuse=reuse, cos=c, S=S, anchor_S=anchor_S, delta=delta,
                            delta_used=dropped_mass(s, S), s_nth=s_nth, out=out, lse=lse,
                            scores=s if keep_scores else None))
    return rec


def decode_workload(wl, heads=None, steps=None, keep_scores=False, max_run=0, n_den=0):
    """Run decode_head over (b, query head) pairs of a ``workloads.Workload``.

    Query head hq reads KV head hq // (Hq / Hkv) (consecutive grouping, the
    usual grouped-query layout). Returns {(b, hq): [HeadStep, ...]}.
    """
    G = wl.Hq // wl.Hkv
    heads = [(b, h) for b in range(wl.B) for h in range(wl.Hq)] if heads is None else heads
    nsteps = wl.steps if steps is None else steps
    res = {}
    cache = {}
    for b, hq in heads:
        kvh = hq // G
        if (b, kvh) not in cache:
            cache = {(b, kvh): (widen(wl.logical_rows("K", b, kvh), wl.dtype),
                                widen(wl.logical_rows("V", b, kvh), wl.dtype))}
        K, V = cache[(b, kvh)]
        qs = widen(wl.q[:nsteps, b, hq], wl.dtype)
        res[(b, hq)] = decode_head(qs, K, V, int(wl.budget[b]), wl.w, wl.tau, wl.scale,
                                   keep_scores=keep_scores, max_run=max_run, n_den=n_den)
    return res


# --------------------------------------------------------------------------- #
# growing cache with forced sinks and local window (Fig. 11)
# --------------------------------------------------------------------------- #
def forced_set(t: int, n_sink: int, window: int) -> np.ndarray:
    """Keys every query attends whatever its scores: the first n_sink keys
    (attention sinks) and the last `window` keys (the local window), clipped
    to [0, t), ascending without repeats.

    Reading of Fig. 11 (sink and recent positions carry attention mass for
    every query) as a deterministic set added to the selected one.
    """
    keep = np.zeros(t, bool)
    keep[:min(max(n_sink, 0), t)] = True
    keep[max(0, t - max(window, 0)):] = True
    return np.nonzero(keep)[0].astype(np.int64)


def top_n_between(s: np.ndarray, N: int, n_sink: int, window: int) -> np.ndarray:
    """The N largest logits among the keys outside the forced set (lowest
    index on ties), ascending: top_n over the middle range [n_sink, t - window)."""
    t = np.asarray(s).shape[0]
    lo, hi = min(max(n_sink, 0), t), max(min(max(n_sink, 0), t), t - max(window, 0))
    return lo + top_n(np.asarray(s)[lo:hi], N)


def decode_head_grow(q_steps: np.ndarray, K: np.ndarray, V: np.ndarray, t0: int, N: int, w: int,
                     tau: float, scale: float, n_sink: int, window: int,
                     keep_scores: bool = False, max_run: int = 0, n_den: int = 0,
                     gate: str = "query") -> list[HeadStep]:
    """decode_head on a cache that gains one key per query, with a forced set.

    Query s sees the first t_s = t0 + s + 1 rows of K and V (the current
    token's key and value are appended before it attends). A retrieving
    query attends forced_set(t_s) together with top_n_between(N); its anchor
    is the top-N part. A reusing query attends forced_set(t_s) together with
    the anchor's set dilated by +/- w and clipped to [0, t_s). delta is the
    dropped mass of the attended set on retrieving queries. With n_sink =
    window = 0 and a fixed cache this is decode_head.

    gate = "key" is the "Key" similarity design of Table IX: the gate
    compares the current token's key (row t_s - 1, appended at this step)
    with the key the anchor query's token appended, instead of the two
    queries. n_den > 0 bounds the dilation as in decode_head.
    """
    if gate not in ("query", "key"):
        raise ValueError(gate)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    anchor_S = anchor_q = None
    rec = []
    age = 0
    for step, q in enumerate(np.asarray(q_steps, np.float64)):
        t = t0 + step + 1
        Kt, Vt = K[:t], V[:t]
        g = q if gate == "query" else K[t - 1]   # the vector this step is gated on
        c, reuse = (None, False) if anchor_S is None else cis_gate(g, anchor_q, tau)
        if max_run > 0 and age >= max_run - 1:
            reuse = False
        age = age + 1 if reuse else 0
        s = scores(q, Kt, scale)
        F = forced_set(t, n_sink, window)
        delta = s_nth = None
        if reuse:
            S = np.union1d(F, shared_set(anchor_S, w, t, n_den)).astype(np.int64)
        else:
            T = top_n_between(s, N, n_sink, window)
            S = np.union1d(F, T).astype(np.int64)
            delta = dropped_mass(s, S)
            anchor_S, anchor_q = T, g
        out, lse = attention(q, Kt, Vt, S, scale)
        rec.append(HeadStep(reuse=reuse, cos=c, S=S, anchor_S=anchor_S, delta=delta,
                            delta_used=dropped_mass(s, S), s_nth=s_nth, out=out, lse=lse,
                            scores=s if keep_scores else None))
    return rec
