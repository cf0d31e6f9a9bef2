"""The seeded input generator (CPU only)."""
import numpy as np

from sparse_attention_kv_qsa_gb300 import workloads as w


def test_pcg32_matches_published_demo():
    # first outputs of pcg32 seeded with (initstate=42, initseq=54) in the
    # PCG reference distribution's demo
    want = [0xA15C02B7, 0x7B47F409, 0xBA1D3330, 0x83D2F293, 0xBFA4784B, 0xCBED606E]
    assert [int(x) for x in w.u32(42, 54, 6)] == want
    assert w.pcg32_reference(42, 54, 6) == want


def test_c_generator_equals_scalar_reference():
    for seed, stream in ((w.SEED_BASE, 1), (w.SEED_BASE + 3, 2), (12345, 6)):
        assert np.array_equal(w.u32(seed, stream, 4000),
                              np.array(w.pcg32_reference(seed, stream, 4000), dtype=np.uint32))


def test_distributions():
    z = w.normal64(1, 1, 400000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    t = w.student_t3_32(1, 2, 400000).astype(np.float64)
    assert abs(np.median(t)) < 0.01
    # unit variance (heavy tail: loose bound); the kurtosis is large
    assert 0.85 < t.var() < 1.15 and np.mean(t ** 4) > 5
    i8 = w.int8_127(1, 3, 200000)
    assert i8.min() == -127 and i8.max() == 127
    u = w.uniform(1, 4, 100000)
    assert u.min() >= 0 and u.max() < 1


def test_workload_shapes_and_capacity():
    W = w.mid()
    assert W.q.shape == (256, 4, 128) and W.kblk.shape == (65538, 128)
    assert not np.isnan(W.kblk[:W.active]).any() and np.isnan(W.kblk[W.active:]).all()
    D = w.decode(4, 262144)
    assert D.active == 65536 and D.kq8.shape == (65538, 128)
    sc = D.kscale[:D.active].view(np.float16).astype(np.float64)
    assert sc.min() >= 0.9e-3 and sc.max() <= 1.01e-1
    assert np.isnan(D.kscale[D.active:].view(np.float16)).all()
    L = w.long()
    assert L.meta["needles"].shape == (256, 16) and len(np.unique(L.meta["needles"])) == 4096


def test_deterministic():
    a, b = w.tiny(), w.tiny()
    assert np.array_equal(a.q, b.q) and np.array_equal(a.kblk, b.kblk)
    assert not np.array_equal(w.tiny(0).q, w.tiny(5).q)


def test_attention_case():
    """The attention recipe: deterministic, k - pad distinct ascending block
    ids in range then -1 padding, int8 cells on [-127, 127], binary16 scales
    positive, finite and within [1e-3, 1e-1] after rounding."""
    A = w.attn_case(5, 4099 * 4 + 3, 60, pad=7)
    B = w.attn_case(5, 4099 * 4 + 3, 60, pad=7)
    for x, y in ((A.q, B.q), (A.kc, B.kc), (A.vc, B.vc), (A.ks, B.ks), (A.vs, B.vs), (A.ids, B.ids)):
        assert np.array_equal(x, y)
    nblocks = (A.ncells + 3) // 4
    assert A.ids.shape == (5, 60) and np.all(A.ids[:, 53:] == -1)
    for row in A.ids[:, :53]:
        assert np.all(np.diff(row) > 0) and row.min() >= 0 and row.max() < nblocks
    assert A.kc.shape == (A.ncells, 128) and A.kc.min() >= -127 and A.kc.max() <= 127
    for sc in (A.ks, A.vs):
        f = sc.view(np.float16).astype(np.float64)
        assert np.all(np.isfinite(f)) and f.min() >= 0.999e-3 and f.max() <= 1.001e-1
    assert not np.array_equal(A.kc, A.vc)            # K and V come from different streams
    # all blocks of a small pool, in a seeded order, ascending
    S = w.attn_case(2, 17, 5)
    assert np.array_equal(S.ids, np.tile(np.arange(5, dtype=np.int32), (2, 1)))
