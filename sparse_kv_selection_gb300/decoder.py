"""Multi-step sparse decode with critical-index-set reuse.

Holds the per-head CIS anchor (its undilated top-N set and its query) on the
device and calls ``prhs_decode_step`` once per decode query: heads whose
query is similar enough to their anchor attend the anchor set dilated by
+/- w, the others retrieve a fresh top-N set and become the new anchor
("Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference",
Fig. 4 and Fig. 8). With n_sink / window every query also attends the first
and the last keys of its cache (Fig. 11), and ``append`` grows the cache by
one key per sequence before the next query. Buffers are allocated once; a
step launches the gate, scoring, selection and two attention kernels (two
more with forced keys) and never synchronises with the host.
"""
from __future__ import annotations

import torch

from . import binding as _b


class SparseDecoder:
    def __init__(self, kv: _b.KVCache, *, N: int | None = None, n_budget=None, w: int = 2,
                 tau: float = 0.8, scale: float | None = None, max_run: int = 0, n_sink: int = 0,
                 window: int = 0, n_den: int = 0, stream=None):
        dev = kv.k.device
        self.kv, self.w, self.tau = kv, int(w), float(tau)
        self.scale = scale if scale is not None else kv.desc.d ** -0.5
        self.N = int(N) if N is not None else 0
        self.n_budget = None if n_budget is None else n_budget.to(device=dev, dtype=torch.int32)
        nmax = self.N if n_budget is None else int(n_budget.max())
        tmax = kv.t_max
        self.anchor_cap = max(1, min(nmax, tmax))
        self.n_sink, self.window = int(n_sink), int(window)
        self.n_den = int(n_den)  # > 0: budgeted dilation (Fig. 9a)
        self.cap = max(1, min(tmax, self.anchor_cap * (2 * self.w + 1) + self.n_sink + self.window))
        B, Hq, d = kv.B, kv.Hq, kv.desc.d
        qdt = kv.k.dtype
        i32 = dict(device=dev, dtype=torch.int32)
        self.anchor_idx = torch.zeros(B, Hq, self.anchor_cap, **i32)
        self.anchor_n = torch.zeros(B, Hq, **i32)
        self.max_run = int(max_run)
        self.anchor_age = torch.zeros(B, Hq, **i32)
        self.q_anchor = torch.zeros(B, Hq, d, device=dev, dtype=qdt)
        self.idx = torch.zeros(B, Hq, self.cap, **i32)
        self.n_sel = torch.zeros(B, Hq, **i32)
        self.reuse = torch.zeros(B, Hq, device=dev, dtype=torch.uint8)
        self.delta = torch.zeros(B, Hq, device=dev, dtype=torch.float32)
        self.out = torch.zeros(B, Hq, d, device=dev, dtype=torch.float32)
        self.lse = torch.zeros(B, Hq, device=dev, dtype=torch.float32)
        self.ws = _b.make_workspace(kv, self.cap, stream)
        self.stream = stream

    def reset(self) -> None:
        """Forget every anchor: the next step retrieves for all heads."""
        self.anchor_n.zero_()
        self.anchor_age.zero_()

    def step(self, q: torch.Tensor, out=None, lse=None, delta=None, reuse=None, n_sel=None,
             gate=None) -> None:
        """One decode query per head (q [B][Hq][d] on the device). Results go
        to the given [B][Hq](...) views, else to the decoder's own buffers.
        delta is written for retrieving heads only. gate ([B][Hq][d], optional):
        the vectors the reuse gate compares in place of q (the "Key"
        similarity design: the key each sequence appended, per query head)."""
        _b.decode_step(self.kv, q, self.scale, self.N, self.w, self.tau, self.anchor_idx,
                       self.anchor_n, self.q_anchor, self.idx,
                       self.n_sel if n_sel is None else n_sel,
                       self.reuse if reuse is None else reuse,
                       self.delta if delta is None else delta,
                       self.out if out is None else out,
                       self.lse if lse is None else lse,
                       self.ws, n_budget=self.n_budget, max_run=self.max_run,
                       anchor_age=self.anchor_age, n_sink=self.n_sink, window=self.window,
                       n_den=self.n_den, gate=gate, stream=self.stream)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor) -> None:
        """Grow the cache by one key per sequence ([B][Hkv][d] device rows,
        the cache's element type) before the next query attends."""
        _b.append_kv(self.kv, k_new, v_new, stream=self.stream)

    def run(self, q_steps: torch.Tensor, outs=None):
        """Decode a [S][B][Hq][d] device sequence; returns stacked per-step
        (out, lse, delta, reuse, n_sel) device tensors (written into ``outs``
        when given). delta is NaN on steps where a head reused its anchor."""
        S = q_steps.shape[0]
        if outs is None:
            outs = self.alloc_outputs(S)
        o, l, dl, r, n = outs
        dl.fill_(float("nan"))
        for s in range(S):
            self.step(q_steps[s], o[s], l[s], dl[s], r[s], n[s])
        return outs

    def alloc_outputs(self, S: int, device=None, pin: bool = False):
        B, Hq, d = self.kv.B, self.kv.Hq, self.kv.desc.d
        dev = self.kv.k.device if device is None else device
        kw = dict(device=dev)
        if pin:
            kw = dict(device="cpu", pin_memory=True)
        return (torch.empty(S, B, Hq, d, dtype=torch.float32, **kw),
                torch.empty(S, B, Hq, dtype=torch.float32, **kw),
                torch.empty(S, B, Hq, dtype=torch.float32, **kw),
                torch.empty(S, B, Hq, dtype=torch.uint8, **kw),
                torch.empty(S, B, Hq, dtype=torch.int32, **kw))

    def run_host(self, q_host: torch.Tensor, q_dev: torch.Tensor, dev_outs, host_outs):
        """End-to-end decode from pinned host queries to pinned host results:
        host->device copy of the queries, the device decode loop, and a
        device->host copy of out, lse, delta, reuse and n_sel."""
        q_dev.copy_(q_host, non_blocking=True)
        self.reset()
        self.run(q_dev, dev_outs)
        for h, d in zip(host_outs, dev_outs):
            h.copy_(d, non_blocking=True)
