"""qsa_block_select: the ids of qsa_block_topk(qsa_block_scores(...)),
bit for bit, without storing the scores (lists of the scores at or above a
sampled per-row threshold), on the parity workloads and on inputs that force
its fallback (lists that overflow, lists shorter than k, NaN scores)."""
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


def to_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _check(W, dev, k=None, kblk=None):
    """ids of the fused call == ids of the two plain calls == the oracle's
    exact top-k of those scores."""
    k = W.k if k is None else k
    kb_np = W.kblk if kblk is None else kblk
    q, kb = to_dev(W.q, dev), to_dev(kb_np, dev)
    ids = qsa.block_select(q, kb, W.active, k)
    s = qsa.block_scores(q, kb, W.active)
    ids2 = qsa.block_topk(s, k)
    torch.cuda.synchronize()
    got, want = ids.cpu().numpy(), ids2.cpu().numpy()
    assert np.array_equal(got, want)
    assert np.array_equal(want, oracle.get().topk_f32(s.cpu().numpy(), k))
    assert qsa.device_error(dev) == 0
    return got


@pytest.mark.parametrize("k", [64, 256, 512, 1024])
def test_full_capacity(dev, k):
    _check(w.full(k=k), dev)


def test_long_needles(dev):
    W = qsa_cases.long_with_needles(oracle.get())
    ids = _check(W, dev)
    for i, nd in enumerate(W.meta["needles"]):
        assert set(nd) <= set(ids[i])


@pytest.mark.parametrize("nq,active,k", [(200, 70001, 300), (37, 9001, 100), (129, 8193, 1), (256, 393216, 1024),
                                         (5, 20000, 7)])
def test_ragged_shapes(dev, nq, active, k):
    _check(w.normal_case(nq=nq, active=active, k=k, max_blocks=active + 5), dev)


def test_plain_branches(dev):
    # nq <= 4, rows within the register-resident top-k's reach, k past the list limit, k >= active
    for nq, active, k in [(4, 65536, 128), (64, 8192, 256), (64, 20000, 2000), (16, 300, 300), (16, 300, 700)]:
        _check(w.normal_case(nq=nq, active=active, k=k), dev)


def test_overflowing_lists_fall_back(dev):
    """Every key the same: every score of a row ties, every score reaches the
    threshold, each list overflows, and the lower ids must win."""
    W = w.normal_case(nq=150, active=30000, k=500)
    kb = np.tile(W.kblk[:1], (W.max_blocks, 1))
    ids = _check(W, dev, kblk=kb)
    assert np.array_equal(ids, np.tile(np.arange(500, dtype=np.int32), (150, 1)))


def test_short_lists_fall_back(dev):
    """The sampled blocks score far above the rest: the threshold comes from
    them alone and lists only a few blocks per row (fewer than k)."""
    W = w.normal_case(nq=140, active=65536, k=512)
    kb = W.kblk.copy()
    sample = (np.arange(1024, dtype=np.int64) * W.active) // 1024
    kb[sample] *= 1000.0
    _check(W, dev, kblk=kb)


def test_nan_scores(dev):
    """NaN keys give NaN scores, which rank below every other score (and
    fail every threshold), in the lists and in the fallback alike."""
    W = w.normal_case(nq=130, active=20000, k=200)
    kb = W.kblk.copy()
    kb[::7, 3] = np.nan
    _check(W, dev, kblk=kb)
    kb2 = W.kblk.copy()
    kb2[:W.active - 150, 0] = np.nan   # fewer than k finite scores per row
    _check(W, dev, kblk=kb2)


def test_scratch_checks(dev):
    W = w.normal_case(nq=130, active=9000, k=10)
    q, kb = to_dev(W.q, dev), to_dev(W.kblk, dev)
    small = torch.empty((qsa.select_scratch_bytes(130) - 16,), dtype=torch.uint8, device=dev)
    with pytest.raises(qsa.QSAError):
        qsa.block_select(q, kb, W.active, W.k, scratch=small)
