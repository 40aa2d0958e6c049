"""Parity at the full sizes of the five decode workloads, in the launch
configuration the benchmark uses (prhs_decode_step per query, the library's
own grids), on sampled heads the fp64 oracle decodes one by one."""
import numpy as np
import pytest

from parity_util import LSE_TOL, OUT_TOL, compare_decode, compare_decode_forced, kv_rows64, q64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SAMPLES = {
    "tiny": [(0, 0)],
    "llama2_7b_mha": [(0, h) for h in (0, 5, 11, 16, 22, 31)],
    "mistral_7b_gqa": [(0, 0), (1, 7), (2, 18), (3, 31)],
    "paged_serving": "lengths",   # shortest, longest and middle sequences
    "long_context": [(0, 0), (0, 13), (0, 30)],
}


def _load(name):
    import sparse_kv_selection_gb300 as S
    from workloads import preset
    from workloads.torch_io import upload
    wl = preset(name, seed=0)
    dev = upload(wl)
    kv = S.KVCache(dev["k"], dev["v"], dev["seq_lens"], wl.Hq, block_table=dev["block_table"])
    heads = SAMPLES[name]
    if heads == "lengths":
        order = np.argsort(wl.seq_lens)
        heads = [(int(order[0]), 3), (int(order[-1]), 17), (int(order[len(order) // 2]), 29)]
    return S, wl, dev, kv, heads


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_size_decode(name):
    S, wl, dev, kv, heads = _load(name)
    compared, r = compare_decode(wl, dev, kv, heads)
    assert compared >= len(heads), "too few steps compared"
    assert S.last_error() == 0
    print(f"{name}: compared {compared} (head, step) pairs of {len(heads) * wl.steps}; "
          f"reuse fraction {r.mean():.3f}")


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_size_decode_teacher_forced(name):
    S, wl, dev, kv, heads = _load(name)
    compared = compare_decode_forced(wl, dev, kv, heads)
    assert compared >= len(heads) * wl.steps - 2, compared


@pytest.mark.parametrize("name", ["llama2_7b_mha", "mistral_7b_gqa", "paged_serving"])
def test_full_size_dense(name):
    import oracle.prhs as P
    S, wl, dev, kv, heads = _load(name)
    out = torch.empty(wl.B, wl.Hq, wl.d, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, device="cuda")
    ws = S.make_workspace(kv)
    S.dense_attn(kv, dev["q"][0], wl.scale, out, lse, ws)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for b, h in heads:
        K, V = kv_rows64(wl, b, h // wl.G)
        ro, rl = P.dense_attention(q64(wl, 0, b, h), K, V, wl.scale)
        assert np.abs(o[b, h] - ro).max() <= OUT_TOL and abs(l[b, h] - rl) <= LSE_TOL
    assert S.last_error() == 0
