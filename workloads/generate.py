"""Seeded synthetic long-context decode workloads.

The pages measure on GSM8K, CoQA, LongBench v2 and WikiText2 with trained
LLaMA/Mistral/Qwen/GLM weights. None of that is used here. These generators
stand in for them by copying the shapes (LLaMA2-7B: 32 heads of d=128;
Mistral-7B: 32 query / 8 KV heads) and the structure the pages show:

* critical indices form small contiguous clusters of keys
  (Near-Oracle KV Selection via Pre-hoc Sparsity, Fig. 2 and Fig. 11);
* consecutive decode queries of one head are highly similar
  (same page, Fig. 2 "cosine similarity > 0.8" and Fig. 10);
* attention sinks at the first positions (Fig. 11 "deterministic sink").

Recipe (one KV head ``h`` of sequence ``b``):

* every K and V element is N(0, 1);
* ``n_clusters`` disjoint runs of consecutive positions, widths uniform in
  ``width``, placed uniformly; cluster ``c`` gets a random unit direction
  ``u_c`` and its keys get ``+boost * u_c``;
* optional sinks: positions ``0..sinks-1`` get ``+sink_boost * u_sink``;
* each query head picks one cluster ``c*`` of its KV head and draws an
  AR(1) sequence ``a_0 ~ N(0, I)``, ``a_{s+1} = rho*a_s + sigma*eps_s``; the
  decode query is ``q_s = a_s + beta * u_{c*}`` with ``beta = sqrt(d)``.

Values are drawn in float32 and then stored either as float32 or rounded to
bfloat16 (round to nearest even), so both consumers see identical bits.

Random streams: numpy's counter-based Philox generator, one independent
SeedSequence child per (seed, tensor tag, sequence, chunk), so the arrays do
not depend on the number of threads used to fill them.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_CHUNK = 1 << 22          # elements per independent random substream
_TAG = {"K": 1, "V": 2, "clusters": 3, "queries": 4, "lengths": 5, "table": 6, "sink": 7}


# --------------------------------------------------------------------------- #
# storage formats
# --------------------------------------------------------------------------- #
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits."""
    # finite inputs only: the sum below stays under 2**32 for every finite float
    src = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(src.shape, np.uint16)
    flat_in, flat_out = src.reshape(-1).view(np.uint32), out.reshape(-1)
    n = flat_in.size

    def conv(c: int) -> None:
        u = flat_in[c * _CHUNK:(c + 1) * _CHUNK]
        r = (u >> 16) & 1
        r += 0x7FFF
        r += u
        r >>= 16
        flat_out[c * _CHUNK:(c + 1) * _CHUNK] = r

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            conv(c)
    else:
        with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(conv, range(nchunks)))
    return out


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- #
# random streams
# --------------------------------------------------------------------------- #
def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence(list(key))))


def _normals(n: int, *key: int) -> np.ndarray:
    """n float32 N(0,1) draws, chunked into independent substreams."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        _rng(*key, c).standard_normal(out=out[lo:hi], dtype=np.float32)

    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def _unit_vectors(n: int, d: int, *key: int) -> np.ndarray:
    v = _rng(*key).standard_normal((n, d))
    v /= np.linalg.norm(v, axis=1, keepdims=True)
    return v.astype(np.float32)


# --------------------------------------------------------------------------- #
# workload container
# --------------------------------------------------------------------------- #
@dataclass
class Workload:
    name: str
    dtype: str                    # "f32" or "bf16": storage type of K, V and q
    B: int
    Hq: int
    Hkv: int
    d: int
    seq_lens: np.ndarray          # int32 [B]
    t_max: int                    # contiguous row stride, or max_blocks*block_size when paged
    paged: bool
    block_size: int
    block_table: np.ndarray | None  # int32 [B][max_blocks] when paged
    K: np.ndarray                 # contiguous [B][Hkv][t_max][d] or paged [nblk][Hkv][bs][d]
    V: np.ndarray
    q: np.ndarray                 # [steps][B][Hq][d]
    budget: np.ndarray            # int32 [B]: KV budget N of each sequence
    w: int
    tau: float
    scale: float
    steps: int
    seed: int
    clusters: list = field(default_factory=list)   # [(b, h)] -> int32 [n][2] (start, width)
    target_cluster: np.ndarray | None = None       # int32 [B][Hq]
    params: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def max_blocks(self) -> int:
        return 0 if self.block_table is None else self.block_table.shape[1]

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def to_f32(self, a: np.ndarray) -> np.ndarray:
        return a.astype(np.float32) if self.dtype == "f32" else f32_from_bf16_bits(a)

    def logical_rows(self, which: str, b: int, h: int) -> np.ndarray:
        """Rows 0..t_b-1 of K or V for sequence b, KV head h, in storage format."""
        src = self.K if which == "K" else self.V
        t = int(self.seq_lens[b])
        if not self.paged:
            return src[b, h, :t]
        nb = (t + self.block_size - 1) // self.block_size
        blocks = src[self.block_table[b, :nb], h]          # [nb][bs][d]
        return blocks.reshape(nb * self.block_size, self.d)[:t]

    def kv_bytes(self) -> int:
        return self.K.nbytes + self.V.nbytes


def _place_clusters(t: int, lo: int, n: int, width: tuple[int, int], rng) -> np.ndarray:
    """n disjoint runs of consecutive positions inside [lo, t)."""
    span = t - lo
    widths = rng.integers(width[0], width[1] + 1, size=n)
    while n > 0 and widths.sum() > span // 2:          # keep clusters sparse
        n -= 1
        widths = widths[:n]
    if n == 0:
        return np.zeros((0, 2), np.int32)
    free = span - int(widths.sum())
    cuts = np.sort(rng.integers(0, free + 1, size=n))
    gaps = np.diff(np.concatenate([[0], cuts]))
    starts = lo + np.cumsum(gaps) + np.concatenate([[0], np.cumsum(widths)[:-1]])
    return np.stack([starts, widths], axis=1).astype(np.int32)


def make_workload(name: str = "custom", *, dtype: str = "bf16", B: int = 1, Hq: int = 1,
                  Hkv: int = 1, d: int = 128, t=4096, paged: bool = False,
                  block_size: int = 16, n_clusters=8, width=(4, 16), boost: float = 3.0,
                  sinks: int = 0, sink_boost: float = 4.0, steps: int = 4, N=None,
                  budget_div: int | None = None, w: int = 2, tau: float = 0.8,
                  rho: float = 0.9, sigma: float = 0.44, beta: float | None = None,
                  seed: int = 0, t_max: int | None = None) -> Workload:
    """Draw one seeded workload.

    ``t`` is a cache length, or ``(lo, hi)`` for lengths uniform in [lo, hi].
    ``n_clusters`` is an int or a callable of the sequence length.
    The KV budget is ``N`` or, with ``budget_div``, ``t_b // budget_div``.
    """
    assert dtype in ("f32", "bf16") and Hq % Hkv == 0
    G = Hq // Hkv
    if isinstance(t, tuple):
        lens = _rng(seed, _TAG["lengths"]).integers(t[0], t[1] + 1, size=B)
    else:
        lens = np.full(B, int(t))
    seq_lens = lens.astype(np.int32)
    if paged:
        tm = int(math.ceil(seq_lens.max() / block_size) * block_size)
    else:
        tm = int(t_max if t_max is not None else seq_lens.max())
        assert tm >= seq_lens.max()
    if budget_div is not None:
        budget = np.maximum(1, seq_lens // budget_div).astype(np.int32)
    else:
        budget = np.full(B, int(N), np.int32)
    beta = math.sqrt(d) if beta is None else beta

    store = (lambda x: x.astype(np.float32)) if dtype == "f32" else bf16_bits_from_f32
    sdt = np.float32 if dtype == "f32" else np.uint16

    # ---- paging ----
    if paged:
        nblk_b = (seq_lens + block_size - 1) // block_size
        nblk = int(nblk_b.sum())
        perm = _rng(seed, _TAG["table"]).permutation(nblk).astype(np.int32)
        max_blocks = int(nblk_b.max())
        table = np.zeros((B, max_blocks), np.int32)
        off = 0
        for b in range(B):
            table[b, :nblk_b[b]] = perm[off:off + nblk_b[b]]
            off += nblk_b[b]
        K = np.zeros((nblk, Hkv, block_size, d), sdt)
        V = np.zeros((nblk, Hkv, block_size, d), sdt)
    else:
        table = None
        K = np.zeros((B, Hkv, tm, d), sdt)
        V = np.zeros((B, Hkv, tm, d), sdt)

    clusters = []
    dirs = {}
    for b in range(B):
        tb = int(seq_lens[b])
        kf = _normals(Hkv * tb * d, seed, _TAG["K"], b).reshape(Hkv, tb, d)
        vf = _normals(Hkv * tb * d, seed, _TAG["V"], b).reshape(Hkv, tb, d)
        crng = _rng(seed, _TAG["clusters"], b)
        nc = n_clusters(tb) if callable(n_clusters) else int(n_clusters)
        for h in range(Hkv):
            cl = _place_clusters(tb, sinks, nc, width, crng)
            u = _unit_vectors(max(len(cl), 1), d, seed, _TAG["clusters"], b, h)
            for c, (s0, wd) in enumerate(cl):
                kf[h, s0:s0 + wd] += boost * u[c]
            if sinks:
                us = _unit_vectors(1, d, seed, _TAG["sink"], b, h)[0]
                kf[h, :sinks] += sink_boost * us
            clusters.append(cl)
            dirs[(b, h)] = u
        ks, vs = store(kf), store(vf)
        if paged:
            nb = int(nblk_b[b])
            pad = nb * block_size - tb
            kp = np.concatenate([ks, np.zeros((Hkv, pad, d), sdt)], axis=1)
            vp = np.concatenate([vs, np.zeros((Hkv, pad, d), sdt)], axis=1)
            K[table[b, :nb]] = kp.reshape(Hkv, nb, block_size, d).transpose(1, 0, 2, 3)
            V[table[b, :nb]] = vp.reshape(Hkv, nb, block_size, d).transpose(1, 0, 2, 3)
        else:
            K[b, :, :tb] = ks
            V[b, :, :tb] = vs

    # ---- queries: AR(1) around a planted cluster direction ----
    qrng = _rng(seed, _TAG["queries"])
    target = np.zeros((B, Hq), np.int32)
    qf = np.zeros((steps, B, Hq, d), np.float32)
    for b in range(B):
        for hq in range(Hq):
            h = hq // G
            ncl = len(clusters[b * Hkv + h])
            c = int(qrng.integers(0, max(ncl, 1)))
            target[b, hq] = c if ncl else -1
            bias = beta * dirs[(b, h)][c] if ncl else np.zeros(d, np.float32)
            a = qrng.standard_normal(d)
            for s in range(steps):
                qf[s, b, hq] = a + bias
                a = rho * a + sigma * qrng.standard_normal(d)
    q = store(qf)

    return Workload(name=name, dtype=dtype, B=B, Hq=Hq, Hkv=Hkv, d=d, seq_lens=seq_lens,
                    t_max=tm, paged=paged, block_size=block_size, block_table=table,
                    K=K, V=V, q=q, budget=budget, w=w, tau=tau, scale=1.0 / math.sqrt(d),
                    steps=steps, seed=seed, clusters=clusters, target_cluster=target,
                    params=dict(n_clusters=n_clusters if not callable(n_clusters) else "t/64",
                                width=width, boost=boost, sinks=sinks, sink_boost=sink_boost,
                                rho=rho, sigma=sigma, beta=beta))


# --------------------------------------------------------------------------- #
# the five decode workloads
# --------------------------------------------------------------------------- #
PRESETS = {
    # 1 layer, batch 1, one head, d=64, fp32 cache of 512 keys, 8 clusters, 16 queries
    "tiny": dict(dtype="f32", B=1, Hq=1, Hkv=1, d=64, t=512, n_clusters=8, steps=16,
                 N=64, w=2),
    # LLaMA2-7B decode layer: 32 MHA heads, d=128, bf16 cache of 4096 keys, N/t = 1/8
    "llama2_7b_mha": dict(dtype="bf16", B=1, Hq=32, Hkv=32, d=128, t=4096, n_clusters=64,
                          steps=64, N=512, w=2),
    # Mistral-7B GQA decode: batch 4, 32 query / 8 KV heads, 32768 keys, N/t = 1/16
    "mistral_7b_gqa": dict(dtype="bf16", B=4, Hq=32, Hkv=8, d=128, t=32768, n_clusters=256,
                           steps=32, N=2048, w=4),
    # paged serving: batch 32 of LLaMA-7B shape, lengths in [2048, 16384], 16-token pages
    "paged_serving": dict(dtype="bf16", B=32, Hq=32, Hkv=32, d=128, t=(2048, 16384),
                          paged=True, block_size=16, n_clusters=lambda tb: tb // 64,
                          steps=16, budget_div=16, w=2),
    # long context: 131072 keys, 32 query / 8 KV heads, 4 sinks, N/t = 1/32
    "long_context": dict(dtype="bf16", B=1, Hq=32, Hkv=8, d=128, t=131072, n_clusters=1024,
                         sinks=4, sink_boost=4.0, steps=16, N=4096, w=4),
}


def preset(name: str, seed: int = 0, **override) -> Workload:
    kw = dict(PRESETS[name])
    kw.update(override)
    return make_workload(name, seed=seed, **kw)
