"""Failure detection on the GPU without a fault, and decode steps issued
concurrently on several streams.

The bounded waits of the TMA pipelines are exercised by a self-test kernel
whose mbarrier nothing arrives on: the wait must run out after the short
limit the host chose, set the timeout bit of the device error word and
return, leaving the context usable for the next call.
"""
import threading
import time

import numpy as np
import pytest

import oracle.prhs as P
from parity_util import LSE_TOL, OUT_TOL, kv_rows64, q64
from workloads import make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPE = dict(dtype="bf16", B=2, Hq=4, Hkv=4, d=128, t=(700, 1500), t_max=1600, n_clusters=12,
             steps=8, N=96, w=2)


def _cache(seed):
    import sparse_kv_selection_gb300 as S
    from workloads.torch_io import upload
    wl = make_workload("streams", seed=seed, **SHAPE)
    dev = upload(wl)
    return wl, dev, S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq)


def test_bounded_wait_runs_out_and_context_survives():
    import sparse_kv_selection_gb300 as S
    from sparse_kv_selection_gb300.binding import DEV_TIMEOUT
    S.last_error()
    for limit_us in (2000, 20000):
        t0 = time.perf_counter()
        S.binding.selftest_wait_timeout(limit_us)
        bits = S.last_error()
        elapsed = time.perf_counter() - t0
        assert bits & DEV_TIMEOUT, bits
        assert elapsed >= limit_us * 1e-6 and elapsed < 5.0, elapsed
    assert S.last_error() == 0   # the word was cleared by the read above
    # the context is still usable: a sparse attention call right after is exact
    wl, dev, kv = _cache(0)
    cap = 64
    idx = np.tile(np.arange(0, 2 * cap, 2, dtype=np.int32), (wl.B, wl.Hq, 1))
    n = np.full((wl.B, wl.Hq), cap, np.int32)
    out = torch.empty(wl.B, wl.Hq, wl.d, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, device="cuda")
    ws = S.make_workspace(kv, cap)
    S.sparse_attn(kv, dev["q"][0], wl.scale, torch.from_numpy(idx).cuda(),
                  torch.from_numpy(n).cuda(), out, lse, ws)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert S.last_error() == 0
    for b in range(wl.B):
        for h in range(wl.Hq):
            K, V = kv_rows64(wl, b, h)
            ro, rl = P.attention(q64(wl, 0, b, h), K, V, idx[b, h], wl.scale)
            assert np.abs(o[b, h] - ro).max() <= OUT_TOL and abs(l[b, h] - rl) <= LSE_TOL


def test_decode_steps_on_two_streams_from_two_threads():
    """Two decoders, each with its own workspace and caller stream, driven by
    two host threads at once: every output must equal the one the same
    decoder gives when it runs alone."""
    import sparse_kv_selection_gb300 as S
    caches = [_cache(0), _cache(1)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]

    def decoder(i):
        wl, dev, kv = caches[i]
        return S.SparseDecoder(kv, N=int(wl.budget[0]), w=wl.w, tau=wl.tau, scale=wl.scale,
                               stream=streams[i])

    decs = [decoder(0), decoder(1)]

    def run(i, outs):
        with torch.cuda.stream(streams[i]):
            decs[i].reset()
            decs[i].run(caches[i][1]["q"], outs)

    alone = []
    for i in range(2):
        outs = decs[i].alloc_outputs(SHAPE["steps"])
        run(i, outs)
        torch.cuda.synchronize()
        alone.append([x.cpu() for x in outs])
    assert S.last_error() == 0
    for rep in range(6):
        outs = [decs[i].alloc_outputs(SHAPE["steps"]) for i in range(2)]
        threads = [threading.Thread(target=run, args=(i, outs[i])) for i in range(2)]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        torch.cuda.synchronize()
        assert S.last_error() == 0
        for i in range(2):
            for a, b in zip(alone[i], outs[i]):
                assert torch.equal(a.nan_to_num(), b.cpu().nan_to_num()), (rep, i)
