"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every workload is seeded and synthetic; the oracle computes every expected
value on the host. Score gate: 1e-6 of each row's largest |score|; ids:
bit-exact against the oracle's top-k of the GPU's own fp32 scores, and the
near-tie rule against the FP64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import qsa_cases
import sparse_attention_kv_qsa_gb300 as qsa
from sparse_attention_kv_qsa_gb300 import workloads as w

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def to_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def gpu_scores(W, dev, scorer="default"):
    q = to_dev(W.q, dev)
    if W.kblk is not None:
        kb = to_dev(W.kblk, dev)
        if scorer == "ffma":
            s = qsa.block_scores_ffma(q, W.active, kblk=kb)
        else:
            s = qsa.block_scores(q, kb, W.active)
    else:
        kq = to_dev(W.kq8, dev)
        ks = to_dev(W.kscale.view(np.int16), dev)
        if scorer == "ffma":
            s = qsa.block_scores_ffma(q, W.active, kblk_q8=kq, kscale_f16=ks)
        else:
            s = qsa.block_scores_q8(q, kq, ks, W.active)
    return s


def oracle_scores(o, W):
    if W.kblk is not None:
        return o.scores(W.q, W.kblk, W.active)
    return o.scores_q8(W.q, W.kq8, W.kscale, W.active)


def check_select(o, W, s_dev, k=None, S_ref=None):
    k = W.k if k is None else k
    ids = qsa.block_topk(s_dev, k).cpu().numpy()
    S_gpu = s_dev.cpu().numpy()
    S_ref = oracle_scores(o, W) if S_ref is None else S_ref
    parity.check_scores(S_gpu, S_ref)
    assert np.array_equal(ids, o.topk_f32(S_gpu, k)), "ids differ from the exact top-k of the GPU scores"
    parity.check_ids_near_tie(ids, S_ref, o.topk_f64(S_ref, k), k)
    return S_gpu, S_ref, ids


SCORERS = ["default", "ffma"]


@pytest.mark.parametrize("scorer", SCORERS)
def test_tiny_planted_ties(dev, o, scorer):
    W = qsa_cases.tiny_with_ties(o)
    S_gpu, S_ref, ids = check_select(o, W, gpu_scores(W, dev, scorer))
    want = o.topk_f64(S_ref, W.k)
    for i, g in enumerate(W.meta["tie_groups"]):
        assert np.all(S_gpu[i][g] == S_gpu[i][g[0]]), "identical keys scored differently"
        assert [b in ids[i] for b in g] == [b in want[i] for b in g]


@pytest.mark.parametrize("scorer", SCORERS)
@pytest.mark.parametrize("nq,active,max_blocks", [
    (8, 1024, 1024), (5, 1003, 1100), (1, 17, 17), (130, 4099, 4101), (256, 8192, 65538), (3, 65536, 65538),
    (200, 5003, 5003), (255, 129, 130)])
def test_integer_inputs_bit_exact(dev, o, scorer, nq, active, max_blocks):
    W = w.integer_valued(nq, active, max_blocks)
    S_gpu = gpu_scores(W, dev, scorer).cpu().numpy()
    S_ref = o.scores(W.q, W.kblk, W.active)
    assert np.array_equal(S_gpu.astype(np.float64), S_ref)


@pytest.mark.parametrize("scorer", SCORERS)
def test_mid_skewed(dev, o, scorer):
    W = w.mid()
    check_select(o, W, gpu_scores(W, dev, scorer))


def test_long_needles(dev, o):
    W = qsa_cases.long_with_needles(o)
    _, _, ids = check_select(o, W, gpu_scores(W, dev))
    for i in range(W.nq):
        assert set(W.meta["needles"][i]) <= set(ids[i]), f"query {i} lost a needle"


@pytest.mark.parametrize("scorer", SCORERS)
def test_full_capacity_k_sweep(dev, o, scorer):
    W = w.full()
    s = gpu_scores(W, dev, scorer)
    S_ref = o.scores(W.q, W.kblk, W.active)
    for k in (512, 64, 256, 1024):
        check_select(o, W, s, k=k, S_ref=S_ref)


@pytest.mark.parametrize("scorer", SCORERS)
@pytest.mark.parametrize("nq", [1, 4])
@pytest.mark.parametrize("cells", [2048, 16384, 65536, 262144])
def test_decode_int8_keys(dev, o, scorer, nq, cells):
    W = w.decode(nq, cells)
    check_select(o, W, gpu_scores(W, dev, scorer))


@pytest.mark.parametrize("scorer", SCORERS)
@pytest.mark.parametrize("nq,active,k", [(3, 4099, 100), (129, 777, 5), (2, 131, 130), (200, 20000, 300)])
def test_int8_ragged(dev, o, scorer, nq, active, k):
    W = w.int8_case(nq, active, k, max_blocks=active + 3)
    check_select(o, W, gpu_scores(W, dev, scorer))


def _wide_magnitudes(W, seed=11):
    """Query rows and key rows rescaled by 10^u, u uniform in [-15, 15] per
    row (far outside the binary16 range the tensor-core scorer's operand
    parts use), plus one query row dominated by a single element, one zero
    key and one key with a single nonzero element."""
    u = w.uniform(seed, 91, W.nq)
    q = (W.q.astype(np.float64) * (10.0 ** (30.0 * u - 15.0))[:, None, None]).astype(np.float32)
    q[0, :, 0] = 1e12
    W.q = q
    if W.kblk is not None:
        v = w.uniform(seed, 92, W.active)
        kb = W.kblk.copy()
        kb[:W.active] = (kb[:W.active].astype(np.float64) * (10.0 ** (30.0 * v - 15.0))[:, None]).astype(np.float32)
        kb[min(5, W.active - 1)] = 0.0
        if W.active > 7:
            kb[7] = 0.0
            kb[7, 3] = 2.5e-20
        W.kblk = kb
    return W


@pytest.mark.parametrize("nq,active,k", [(160, 4099, 64), (256, 65536, 512), (7, 1000, 17)])
def test_wide_magnitude_ranges(dev, o, nq, active, k):
    W = _wide_magnitudes(w.normal_case(nq, active, k, max_blocks=active + 2))
    check_select(o, W, gpu_scores(W, dev))


@pytest.mark.parametrize("nq,active,k", [(160, 4099, 64), (4, 2048, 32)])
def test_wide_query_magnitudes_int8_keys(dev, o, nq, active, k):
    W = _wide_magnitudes(w.int8_case(nq, active, k, max_blocks=active + 2))
    check_select(o, W, gpu_scores(W, dev))


@pytest.mark.parametrize("nq,active", [(1, 1), (2, 63), (3, 4099), (4, 65536), (1, 70001)])
def test_small_nq_fp32_keys(dev, o, nq, active):
    """nq <= 4 takes the CUDA-core row scorer (grid over key rows)."""
    W = w.normal_case(nq=nq, active=active, k=min(64, active))
    check_select(o, W, gpu_scores(W, dev))


@pytest.mark.parametrize("nq,active", [(2, 517), (3, 65535), (4, 1)])
def test_small_nq_int8_keys(dev, o, nq, active):
    W = w.int8_case(nq, active, min(50, active), max_blocks=active + 1)
    check_select(o, W, gpu_scores(W, dev))


def _tie_heavy(nq, active, seed):
    u = w.u32(seed, 11, nq * active).reshape(nq, active)
    s = ((u % 7).astype(np.float32) - 3.0) * 0.5          # 7 values: heavy ties
    s[(u >> 8) % 5 == 0] = 0.0
    s[(u >> 12) % 5 == 0] = -0.0
    fine = w.normal32(seed, 12, nq * active).reshape(nq, active)
    mix = ((u >> 16) % 3 == 0)
    s[mix] = fine[mix]
    return np.ascontiguousarray(s)


@pytest.mark.parametrize("nq,active,k", [
    (1, 1, 1), (2, 2, 1), (3, 3, 2), (4, 31, 30), (5, 1000, 1), (6, 1000, 999), (3, 4097, 64),
    (2, 8193, 4096), (7, 16385, 512), (1, 65536, 128), (4, 65536, 512), (200, 5003, 77),
    (2, 100003, 1000), (2, 393216, 1000), (1, 393213, 2)])
def test_topk_exact_on_given_scores(dev, o, nq, active, k):
    S = _tie_heavy(nq, active, seed=active * 31 + k)
    ids = qsa.block_topk(to_dev(S, dev), k).cpu().numpy()
    assert np.array_equal(ids, o.topk_f32(S, k))
    parity.check_ids_valid(ids, active, k)


@pytest.mark.parametrize("active", [2, 511, 512, 513, 2048, 2049, 4096, 4097, 8191, 8192, 8193, 16384])
@pytest.mark.parametrize("kind", ["ties", "signed", "smooth"])
def test_topk_register_path_rows(dev, o, active, kind):
    """Rows of at most 8,192 scores take the register-resident path: every
    register width (4, 8, 16 scores per thread) and its boundaries (and the
    first rows past it), with
    tie-heavy rows, rows mixing +-0, +-inf and NaN, and smooth rows; k from 1
    to active - 1, and the decode k = 128."""
    nq = 3
    if kind == "ties":
        S = _tie_heavy(nq, active, seed=active + 5)
    elif kind == "signed":
        u = w.u32(active + 7, 3, nq * active).reshape(nq, active)
        vals = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1.0, -1.0, 2.5], dtype=np.float32)
        S = vals[u % 8]
    else:
        S = w.normal32(active + 9, 2, nq * active).reshape(nq, active)
    S = np.ascontiguousarray(S)
    for k in sorted({1, min(128, active - 1), active // 2, active - 1} - {0}):
        ids = qsa.block_topk(to_dev(S, dev), k).cpu().numpy()
        assert np.array_equal(ids, o.topk_f32(S, k)), (active, kind, k)
        parity.check_ids_valid(ids, active, k)


@pytest.mark.parametrize("m", [4095, 4096, 4097, 8000])
def test_topk_candidate_list_capacity(dev, o, m):
    """Exact path (rows under 8,192 scores): the leading-digit bin holds m
    keys; at and below the candidate-list capacity (4,096) the refinement
    runs on the list, above it on the row."""
    active = 8191
    S = np.full((2, active), -1.0, dtype=np.float32)
    S[:, :100] = 4.0 + np.arange(100, dtype=np.float32) * 0.01
    vals = (1.0 + np.arange(m, dtype=np.float64) * 2.0 ** -20).astype(np.float32)
    S[0, 100:100 + m] = vals
    S[1, 100:100 + m] = vals[::-1]
    S[1, 100 + m // 3] = S[1, 100 + m // 2]          # an exact tie inside the bin
    for k in (100 + m // 2, 100 + m - 1, 101):
        ids = qsa.block_topk(to_dev(S, dev), k).cpu().numpy()
        assert np.array_equal(ids, o.topk_f32(S, k)), (m, k)


def _sampled_positions(active):
    """Row indices the sampled-threshold path reads (one 16-byte group per
    512 bytes, 16 groups in), for rows whose start is 16-byte aligned."""
    g = np.arange(active // 4 // 32) * 32 + 16
    return (4 * g[:, None] + np.arange(4)[None, :]).ravel()


def test_topk_sample_sees_only_the_largest(dev, o):
    """Every sampled score is large and every other one small: the sample's
    threshold leaves fewer than k scores listed, so the row must take the
    exact passes and still return the exact top-k."""
    active, k = 65536, 512
    S = w.normal32(41, 1, 3 * active).reshape(3, active).astype(np.float32)
    pos = _sampled_positions(active)
    S[:, pos] = 100.0 + np.abs(S[:, pos])
    S[2, pos[::2]] = 50.0                              # ties among the sampled scores
    ids = qsa.block_topk(to_dev(S, dev), k).cpu().numpy()
    assert np.array_equal(ids, o.topk_f32(S, k))


@pytest.mark.parametrize("outlier", [1e30, np.inf, 1e10, 100.0, -1e-30])
def test_topk_sample_maximum_far_above_the_rest(dev, o, outlier):
    """A few sampled scores (fewer than the sample rank the threshold uses)
    far above the rest put the threshold's rank many octaves below the
    sample maximum (1e30, inf, 1e10: past the sampled window, so the exact
    passes run), a few octaves below it (100), or make every sampled score
    but some tiny negatives negative and large (-1e-30 on an all-negative
    row): the top-k stays exact."""
    active, k = 65536, 512
    S = w.normal32(43, 1, 3 * active).reshape(3, active).astype(np.float32)
    if outlier < 0:
        S = -np.abs(S) - 1.0
    pos = _sampled_positions(active)
    S[0, pos[:3]] = outlier
    S[1, pos[5:25:4]] = outlier
    S[2, pos[-2:]] = outlier
    S[2, 7] = outlier                                  # and one unsampled
    ids = qsa.block_topk(to_dev(S, dev), k).cpu().numpy()
    assert np.array_equal(ids, o.topk_f32(S, k))


@pytest.mark.parametrize("nq,active,k", [(5, 70001, 64), (3, 70003, 700), (3, 100002, 5000),
                                         (2, 16384, 1000), (2, 16383, 1000), (3, 8192, 700), (3, 8191, 700),
                                         (3, 50001, 600), (2, 49153, 3000),
                                         (2, 393215, 1200),
                                         (2, 393215, 4000)])
def test_topk_ragged_rows_random(dev, o, nq, active, k):
    """Rows of odd length start at every 4-byte offset, so the listing pass
    meets ragged heads and tails; smooth data keeps the list within capacity
    for small k and overflows it for large k."""
    S = w.normal32(active + k, 2, nq * active).reshape(nq, active)
    ids = qsa.block_topk(to_dev(S, dev), k).cpu().numpy()
    assert np.array_equal(ids, o.topk_f32(S, k))


@pytest.mark.parametrize("n_pos,n_zero,n_inf,k", [(500, 2500, 0, 1000), (1000, 2000, 0, 800),
                                                   (0, 0, 3000, 1000), (200, 0, 3000, 2500)])
def test_topk_threshold_at_signed_zero_and_inf(dev, o, n_pos, n_zero, n_inf, k):
    """Counts chosen so that the sampled threshold tends to fall on the
    zeros (both signs, equal keys) or on +inf (ties to the lower id)."""
    active, nq = 65536, 3
    u = w.u32(n_pos + n_zero + n_inf + k, 3, nq * active).reshape(nq, active)
    S = -1.0 - (u % 1000).astype(np.float32)
    for r in range(nq):
        perm = np.argsort(u[r] >> 10, kind="stable")
        S[r, perm[:n_pos]] = 1.0 + (u[r, perm[:n_pos]] % 4096).astype(np.float32)
        z = perm[n_pos:n_pos + n_zero]
        S[r, z] = np.where(u[r, z] & 1, np.float32(0.0), np.float32(-0.0))
        S[r, perm[n_pos + n_zero:n_pos + n_zero + n_inf]] = np.inf
    ids = qsa.block_topk(to_dev(S, dev), k).cpu().numpy()
    assert np.array_equal(ids, o.topk_f32(S, k))


def test_topk_nan_ranks_lowest(dev, o):
    S = _tie_heavy(3, 3001, seed=5)
    S[0, ::3] = np.nan
    S[1, :] = np.nan
    S[1, 17] = -np.inf
    S[2, 5] = np.inf
    ids = qsa.block_topk(to_dev(S, dev), 1500).cpu().numpy()
    assert np.array_equal(ids, o.topk_f32(S, 1500))


@pytest.mark.parametrize("active,k", [(10, 10), (10, 13), (1, 4), (0, 3)])
def test_topk_k_at_least_active(dev, o, active, k):
    S = _tie_heavy(3, max(active, 1), seed=3)[:, :active].copy()
    ids = qsa.block_topk(to_dev(S, dev), k).cpu().numpy()
    assert np.array_equal(ids, o.topk_f32(S, k))


@pytest.mark.parametrize("nq", [37, 3, 200])
def test_outputs_stay_in_bounds(dev, o, nq):
    """Canary words after the scores and ids must survive; capacity rows
    (NaN) must not be read."""
    W = w.normal_case(nq=nq, active=2051, k=100, max_blocks=2300)
    q, kb = to_dev(W.q, dev), to_dev(W.kblk, dev)
    n_s, n_i = W.nq * W.active, W.nq * W.k
    buf_s = torch.full((n_s + 64,), 12345.0, dtype=torch.float32, device=dev)
    buf_i = torch.full((n_i + 64,), 777, dtype=torch.int32, device=dev)
    s = buf_s[:n_s].view(W.nq, W.active)
    ids = buf_i[:n_i].view(W.nq, W.k)
    qsa.block_scores(q, kb, W.active, out=s)
    qsa.block_topk(s, W.k, out=ids)
    assert torch.all(buf_s[n_s:] == 12345.0) and torch.all(buf_i[n_i:] == 777)
    check_select(o, W, s)


@pytest.mark.parametrize("nq,active,k", [(160, 70001, 200), (256, 33, 8), (140, 38912, 1000)])
def test_two_query_groups_ragged(dev, o, nq, active, k):
    """Two query groups (the scorer's clusters then share each key tile's
    conversion): a partial second group, ragged tile tails, few tiles."""
    W = w.normal_case(nq=nq, active=active, k=k, max_blocks=active + 3)
    check_select(o, W, gpu_scores(W, dev))


def test_side_stream(dev, o):
    W = w.normal_case(nq=9, active=3000, k=50)
    st = torch.cuda.Stream(dev)
    q, kb = to_dev(W.q, dev), to_dev(W.kblk, dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        s, ids = qsa.block_select_gmax(q, kb, W.active, W.k)
    st.synchronize()
    check_select(o, W, s)


def test_no_kernel_reported_a_timeout(dev):
    assert qsa.device_error(dev) == 0
