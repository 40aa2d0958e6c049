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
