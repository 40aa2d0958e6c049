"""The seeded generators: determinism, layout and the structure they promise."""
import numpy as np

from workloads import make_workload, preset, bf16_bits_from_f32, f32_from_bf16_bits


def test_bf16_round_nearest_even():
    x = np.array([1.0, 1.00390625, 1.005859375, 1.0117188, -2.5, 0.0], np.float32)
    # 1 + 2^-8 is a tie -> even (1.0); 1 + 1.5*2^-8 rounds up to 1 + 2^-7
    assert f32_from_bf16_bits(bf16_bits_from_f32(x)).tolist()[:3] == [1.0, 1.0, 1.0078125]
    torch = __import__("pytest").importorskip("torch")
    y = np.random.default_rng(0).normal(size=4096).astype(np.float32) * 100
    ref = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (ref == bf16_bits_from_f32(y)).all()


def test_deterministic():
    a = make_workload(B=2, Hq=4, Hkv=2, d=32, t=300, steps=3, N=20, seed=7)
    b = make_workload(B=2, Hq=4, Hkv=2, d=32, t=300, steps=3, N=20, seed=7)
    c = make_workload(B=2, Hq=4, Hkv=2, d=32, t=300, steps=3, N=20, seed=8)
    assert (a.K == b.K).all() and (a.V == b.V).all() and (a.q == b.q).all()
    assert not (a.K == c.K).all()


def test_paged_layout_matches_contiguous():
    kw = dict(B=3, Hq=4, Hkv=2, d=32, t=(40, 200), steps=2, budget_div=8, seed=3)
    p = make_workload(paged=True, block_size=16, **kw)
    c = make_workload(paged=False, **kw)
    assert (p.seq_lens == c.seq_lens).all()
    for b in range(3):
        nb = -(-int(p.seq_lens[b]) // 16)
        assert len(set(p.block_table[b, :nb].tolist())) == nb
        for h in range(2):
            assert (p.logical_rows("K", b, h) == c.logical_rows("K", b, h)).all()
            assert (p.logical_rows("V", b, h) == c.logical_rows("V", b, h)).all()
    # every physical block is used by exactly one (sequence, page)
    used = np.concatenate([p.block_table[b, :-(-int(p.seq_lens[b]) // 16)] for b in range(3)])
    assert sorted(used.tolist()) == list(range(p.K.shape[0]))
    assert (p.budget == p.seq_lens // 8).all()


def test_clusters_disjoint_and_boosted():
    w = make_workload(dtype="f32", B=1, Hq=1, Hkv=1, d=64, t=512, n_clusters=8, steps=2, N=64)
    cl = w.clusters[0]
    assert len(cl) == 8
    ends = cl[:, 0] + cl[:, 1]
    assert (cl[1:, 0] >= ends[:-1]).all() and ends[-1] <= 512 and (cl[:, 1] >= 4).all()
    assert (cl[:, 1] <= 16).all()


def test_sinks_kept_clear_of_clusters():
    w = make_workload(B=1, Hq=2, Hkv=1, d=32, t=600, n_clusters=10, sinks=4, steps=2, N=32)
    assert (w.clusters[0][:, 0] >= 4).all()


def test_query_similarity_llama_shape():
    """Consecutive queries of a head have mean cosine >= 0.8 (Fig. 10 regime)."""
    w = make_workload(B=1, Hq=32, Hkv=32, d=128, t=64, n_clusters=4, steps=64, N=8)
    q = f32_from_bf16_bits(w.q).astype(np.float64)
    c = (q[1:] * q[:-1]).sum(-1) / np.linalg.norm(q[1:], axis=-1) / np.linalg.norm(q[:-1], axis=-1)
    assert c.mean() >= 0.8


def test_presets_shapes_small():
    w = preset("tiny")
    assert w.K.shape == (1, 1, 512, 64) and w.K.dtype == np.float32 and w.q.shape == (16, 1, 1, 64)
    assert int(w.budget[0]) == 64 and w.w == 2
