"""Helpers shared by the GPU parity tests (comparison rules, uploads)."""
from __future__ import annotations

import numpy as np

import oracle.prhs as P

# Tolerances: attention outputs max-abs 2e-3 (bf16 inputs, fp32 accumulation);
# dropped mass and log-sum-exp 1e-4; index sets exact outside near-ties,
# where a near-tie is a key whose float64 logit lies within 1e-4 of the N-th
# largest; cosine gates within 1e-12 of tau are not compared (the GPU gate is
# float64 too, only the summation order differs).
OUT_TOL = 2e-3
LSE_TOL = 1e-4
DELTA_TOL = 1e-4
TIE_GAP = 1e-4
GATE_GAP = 1e-12


def check_topn(gpu_set: np.ndarray, s: np.ndarray, N: int) -> int:
    """Assert a GPU top-N set agrees with the float64 logits; return the
    number of near-tie positions that were left uncompared."""
    t = s.size
    gpu_set = np.asarray(gpu_set, np.int64)
    if N >= t:
        assert gpu_set.tolist() == list(range(t))
        return 0
    assert gpu_set.size == N, (gpu_set.size, N)
    assert np.all(np.diff(gpu_set) > 0), "set must be ascending without repeats"
    assert gpu_set.min() >= 0 and gpu_set.max() < t
    ref = P.top_n(s, N)
    s_n = np.sort(s)[::-1][N - 1]
    near = np.abs(s - s_n) < TIE_GAP
    far = ~near
    in_gpu = np.zeros(t, bool)
    in_gpu[gpu_set] = True
    in_ref = np.zeros(t, bool)
    in_ref[ref] = True
    assert (in_gpu[far] == in_ref[far]).all(), "index sets differ away from near-ties"
    return int(near.sum()) if (in_gpu != in_ref).any() else 0


def kv_rows64(wl, b, kvh):
    return (P.widen(wl.logical_rows("K", b, kvh), wl.dtype),
            P.widen(wl.logical_rows("V", b, kvh), wl.dtype))


def q64(wl, step, b, hq):
    return P.widen(wl.q[step, b, hq], wl.dtype)


def compare_decode(wl, dev, kv, heads, steps=None, N=None, max_run=0, n_den=0):
    """Decode on the device query by query and compare sampled heads with
    oracle.decode_head: reuse flags, the attended set, its size, delta, out
    and lse. A retrieving step whose set differs from the oracle's only at
    near-ties is accepted (check_topn) and ends the comparison of that head,
    since later sets may legitimately differ; so does a gate within
    GATE_GAP of tau. Returns (steps compared, reuse flags [S][B][Hq])."""
    import torch

    import sparse_kv_selection_gb300 as S
    steps = wl.steps if steps is None else steps
    nb = dev["budget"] if len(set(wl.budget.tolist())) > 1 else None
    dec = S.SparseDecoder(kv, N=int(wl.budget[0]) if nb is None else None, n_budget=nb, w=wl.w,
                          tau=wl.tau, scale=wl.scale, max_run=max_run, n_den=n_den)
    o, l, dl, r, n = dec.alloc_outputs(steps)
    dl.fill_(float("nan"))
    bi = torch.tensor([b for b, _ in heads], device="cuda")
    hi = torch.tensor([h for _, h in heads], device="cuda")
    gpu_sets = []
    for s in range(steps):
        dec.step(dev["q"][s], o[s], l[s], dl[s], r[s], n[s])
        gpu_sets.append((dec.idx[bi, hi].cpu().numpy(), n[s][bi, hi].cpu().numpy()))
    o, l, dl, r, n = [x.cpu().numpy() for x in (o, l, dl, r, n)]
    ref = P.decode_workload(wl, heads=heads, steps=steps, keep_scores=True, max_run=max_run,
                            n_den=n_den)
    compared = 0
    for k, ((b, h), recs) in enumerate(ref.items()):
        for s, rec in enumerate(recs):
            if rec.cos is not None and abs(rec.cos - wl.tau) < GATE_GAP:
                break
            assert bool(r[s, b, h]) == rec.reuse, (b, h, s)
            g_idx, g_n = gpu_sets[s]
            gset = g_idx[k, :g_n[k]]
            same = gset.size == rec.S.size and (gset == rec.S).all()
            if not rec.reuse:
                assert abs(dl[s, b, h] - rec.delta) <= DELTA_TOL, (b, h, s)
            else:
                assert same, ("dilated set differs", b, h, s)
            if same:
                want_o, want_l = rec.out, rec.lse
            else:
                # a retrieving set that differs only at near-ties: the attention
                # is checked on the GPU's own set, then this head stops
                check_topn(gset, rec.scores, int(wl.budget[b]))
                K, V = kv_rows64(wl, b, h // wl.G)
                want_o, want_l = P.attention(q64(wl, s, b, h), K, V, gset, wl.scale)
            assert np.abs(o[s, b, h] - want_o).max() <= OUT_TOL, (b, h, s)
            assert abs(l[s, b, h] - want_l) <= LSE_TOL, (b, h, s)
            compared += 1
            if not same:
                break
            assert n[s, b, h] == len(rec.S), (b, h, s)
    return compared, r


def compare_decode_forced(wl, dev, kv, heads, steps=None, max_run=0, n_den=0):
    """Teacher-forced decode: before every query the sampled heads get the
    oracle's anchor state (its undilated set, the anchor query, the reuse
    count), so a near-tie at one query cannot carry over to the next and
    every (head, query) pair is compared. A retrieving set that differs from
    the oracle's only at near-ties is accepted; the attention is then checked
    against the oracle on the GPU's own set. Returns the pairs compared."""
    import torch

    import sparse_kv_selection_gb300 as S
    steps = wl.steps if steps is None else steps
    nb = dev["budget"] if len(set(wl.budget.tolist())) > 1 else None
    dec = S.SparseDecoder(kv, N=int(wl.budget[0]) if nb is None else None, n_budget=nb, w=wl.w,
                          tau=wl.tau, scale=wl.scale, max_run=max_run, n_den=n_den)
    ref = P.decode_workload(wl, heads=heads, steps=steps, keep_scores=True, max_run=max_run,
                            n_den=n_den)
    o, l, dl, r, n = dec.alloc_outputs(1)
    compared = 0
    for s in range(steps):
        for (b, h), recs in ref.items():
            if s == 0:
                dec.anchor_n[b, h] = 0
                dec.anchor_age[b, h] = 0
                continue
            A = recs[s - 1].anchor_S
            last = max(j for j in range(s) if not recs[j].reuse)  # the anchor's query
            dec.anchor_idx[b, h, :len(A)] = torch.from_numpy(A.astype(np.int32)).cuda()
            dec.anchor_n[b, h] = len(A)
            dec.anchor_age[b, h] = s - 1 - last
            dec.q_anchor[b, h] = dev["q"][last, b, h]
        dl.fill_(float("nan"))
        dec.step(dev["q"][s], o[0], l[0], dl[0], r[0], n[0])
        oo, ll, dd, rr, nn = [x[0].cpu().numpy() for x in (o, l, dl, r, n)]
        gidx = dec.idx.cpu().numpy()
        for (b, h), recs in ref.items():
            rec = recs[s]
            if rec.cos is not None and abs(rec.cos - wl.tau) < GATE_GAP:
                continue
            assert bool(rr[b, h]) == rec.reuse, (b, h, s)
            gset = gidx[b, h, :nn[b, h]]
            if rec.reuse:
                assert gset.tolist() == rec.S.tolist(), ("dilated set differs", b, h, s)
                want_o, want_l = rec.out, rec.lse
            else:
                assert abs(dd[b, h] - rec.delta) <= DELTA_TOL, (b, h, s)
                if gset.size == rec.S.size and (gset == rec.S).all():
                    want_o, want_l = rec.out, rec.lse
                else:
                    check_topn(gset, rec.scores, int(wl.budget[b]))
                    K, V = kv_rows64(wl, b, h // wl.G)
                    want_o, want_l = P.attention(q64(wl, s, b, h), K, V, gset, wl.scale)
            assert np.abs(oo[b, h] - want_o).max() <= OUT_TOL, (b, h, s)
            assert abs(ll[b, h] - want_l) <= LSE_TOL, (b, h, s)
            compared += 1
    return compared
