"""GPU parity of the group-maximum side output (32-block group maxima of the
scores) and of the top-k that reads only the groups reaching its threshold.

Expected values come from the oracle: group maxima from its key definition
applied to the GPU's own scores, ids from its full-sort top-k of those
scores. The group-maximum top-k must equal the plain top-k bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
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


def keys(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("kind,nq,active", [
    ("f32", 37, 1000), ("f32", 130, 4099), ("f32", 256, 65536), ("f32", 5, 31), ("f32", 9, 32),
    ("q8", 9, 4100), ("q8", 200, 65536),
    ("f32", 3, 1001), ("f32", 1, 65536), ("q8", 4, 65536), ("q8", 2, 33)])
def test_scores_gmax(dev, o, kind, nq, active):
    """Scores equal the plain scorer's bits; each group maximum is the key of
    the largest of its (up to) 32 scores. nq >= 5 runs the tensor-core
    epilogue, nq <= 4 the decode scorer and its group kernel."""
    q = None
    if kind == "f32":
        W = w.normal_case(nq, active, 1)
        q, kb = to_dev(W.q, dev), to_dev(W.kblk, dev)
        s0 = qsa.block_scores(q, kb, active)
        s, gm = qsa.block_scores_gmax(q, kb, active)
    else:
        W = w.int8_case(nq, active, 1)
        q, kq, ks = to_dev(W.q, dev), to_dev(W.kq8, dev), to_dev(W.kscale.view(np.int16), dev)
        s0 = qsa.block_scores_q8(q, kq, ks, active)
        s, gm = qsa.block_scores_q8_gmax(q, kq, ks, active)
    torch.cuda.synchronize()
    assert torch.equal(s, s0)
    assert np.array_equal(keys(gm), o.group_max_keys(s.cpu().numpy()))


@pytest.mark.parametrize("active", [1, 31, 32, 33, 4099, 65536])
def test_group_max_of_given_scores(dev, o, active):
    """Special values: NaN counts as -inf, -0 as +0, infinities included."""
    S = w.normal32(71, 1, 3 * active).reshape(3, active).astype(np.float32)
    S[0, ::7] = np.nan
    S[1, ::5] = -0.0
    S[1, 3::11] = 0.0
    S[2, ::13] = np.inf
    S[2, 1::17] = -np.inf
    gm = qsa.block_group_max(to_dev(S, dev))
    assert np.array_equal(keys(gm), o.group_max_keys(S))


def topk_both(S, k, dev):
    s = to_dev(S, dev)
    gm = qsa.block_group_max(s)
    return qsa.block_topk_gmax(s, gm, k).cpu().numpy(), qsa.block_topk(s, k).cpu().numpy()


@pytest.mark.parametrize("nq,active,k", [
    (3, 65536, 512), (3, 65536, 1), (3, 65536, 1024), (2, 65536, 1025), (4, 65536, 64),
    (3, 50001, 600), (5, 70001, 64), (4, 4099, 60), (3, 1000, 15), (2, 64, 1), (3, 16383, 255),
    (2, 65535, 700)])
def test_topk_gmax_random(dev, o, nq, active, k):
    """Normal and Student-t rows of aligned and ragged lengths; k above half
    the group count, or rows past 2,048 groups, take the plain path."""
    S = w.normal32(active + k, 3, nq * active).reshape(nq, active)
    S[-1] = w.student_t3_32(active + k, 4, active)
    ids_g, ids_p = topk_both(S, k, dev)
    ref = o.topk_f32(S, k)
    assert np.array_equal(ids_g, ref)
    assert np.array_equal(ids_p, ref)


@pytest.mark.parametrize("levels,k", [(3, 512), (40, 512), (1, 512), (200, 100), (9, 1000)])
def test_topk_gmax_ties(dev, o, levels, k):
    """Scores on a few levels: many groups share their maximum, so the
    threshold sits on a tie of group maxima (and of scores); one level makes
    every score equal and the group list overflows (plain exact path)."""
    active, nq = 65536, 3
    u = w.u32(levels + k, 5, nq * active).reshape(nq, active)
    S = ((u % levels).astype(np.float32) - levels / 2) * np.float32(0.25)
    S[1] = -np.abs(S[1]) - 1.0                 # all negative
    ids_g, _ = topk_both(S, k, dev)
    assert np.array_equal(ids_g, o.topk_f32(S, k))


@pytest.mark.parametrize("outlier", [1e30, np.inf, 1e10, 3.0])
def test_topk_gmax_outlier_group(dev, o, outlier):
    """A few groups far above the rest put the k-th group maximum past the
    threshold window (1e30, inf, 1e10: plain exact path) or inside it (3)."""
    active, k = 65536, 512
    S = w.normal32(81, 1, 3 * active).reshape(3, active).astype(np.float32)
    S[0, [5, 1000, 40000]] = outlier
    S[1, :32] = outlier
    S[2, 7] = outlier
    S[2, 64 * 32 + 3] = -outlier
    ids_g, _ = topk_both(S, k, dev)
    assert np.array_equal(ids_g, o.topk_f32(S, k))


def test_select_full_headline_equals_plain_path(dev, o):
    """At the headline size (256 x 65,536 Student-t, k = 512): block_select
    (group maxima) gives the same scores and ids as block_scores then
    block_topk, and the ids of 8 sampled rows equal the oracle's."""
    W = w.full(512)
    q, kb = to_dev(W.q, dev), to_dev(W.kblk, dev)
    s, ids = qsa.block_select_gmax(q, kb, W.active, 512)
    s0 = qsa.block_scores(q, kb, W.active)
    ids0 = qsa.block_topk(s0, 512)
    torch.cuda.synchronize()
    assert torch.equal(s, s0)
    assert torch.equal(ids, ids0)
    rows = np.arange(0, 256, 32)
    S = s[rows].cpu().numpy()
    assert np.array_equal(ids[rows].cpu().numpy(), o.topk_f32(S, 512))
