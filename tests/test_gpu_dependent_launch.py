"""Kernels launched as programmatic dependents read their inputs correctly.

Every kernel of the library may start while the previous grid on its stream
is still running and reads that grid's outputs only after waiting for it. A
read of those outputs through the read-only path, or from an L1 line an
earlier kernel left on the SM, would return stale data (this was measured:
a top-k launched right behind its scorer read old scores at reused
addresses). These tests launch the dependent sequences back to back -- the
two launches of qsa_block_select_static from C, and a CUDA graph of scores,
top-k and attention -- while other kernels keep reading and rewriting the
same memory between calls, and check every call against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import sparse_attention_kv_qsa_gb300 as qsa
from sparse_attention_kv_qsa_gb300 import workloads as w

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def to_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _churn(nq, active, k, dev, keep):
    # new data at recycled addresses, read through the library's top-k
    x = torch.randn((nq, active), device=dev)
    keep.append(qsa.block_topk(x, k))
    del x
    if len(keep) > 4:
        keep.pop(0)


# register-resident top-k, the group-maximum mode, the sampled listing path
@pytest.mark.parametrize("nq,active,k", [(37, 4099, 60), (16, 65536, 512), (9, 70001, 300)])
def test_static_select_back_to_back(dev, nq, active, k):
    o = oracle.get()
    W = w.normal_case(nq, active, k)
    q, kb = to_dev(W.q, dev), to_dev(W.kblk, dev)
    keep, ref = [], None
    for _ in range(60):
        s, ids = qsa.block_select_static(q, kb, active, k)
        torch.cuda.synchronize()
        S = s.cpu().numpy()
        if ref is None:
            ref = S.copy()
            parity.check_scores(ref, o.scores(W.q, W.kblk, W.active))
            want = o.topk_f32(ref, k)
        assert np.array_equal(S, ref)
        assert np.array_equal(ids.cpu().numpy(), want)
        _churn(nq, active, k, dev, keep)
    assert qsa.device_error(dev) == 0


@pytest.mark.parametrize("nq", [4, 160])   # decode scorer + CUDA-core attention / tensor cores for both
def test_graph_scores_topk_attention(dev, nq):
    """One graph: scores (with group maxima), top-k, attention over the
    selected blocks. The attention reads the ids of the grid before it."""
    o = oracle.get()
    k, cells = 96, 32768
    A = w.attn_case(nq, cells, k)
    W = w.normal_case(nq, cells // 4, k)
    q, kb = to_dev(A.q, dev), to_dev(W.kblk, dev)
    kc, vc = to_dev(A.kc, dev), to_dev(A.vc, dev)
    ks, vs = to_dev(A.ks.view(np.int16), dev), to_dev(A.vs.view(np.int16), dev)
    s = torch.empty((nq, W.active), dtype=torch.float32, device=dev)
    gm = torch.empty((nq, qsa.groups(W.active)), dtype=torch.int32, device=dev)
    ids = torch.empty((nq, k), dtype=torch.int32, device=dev)
    out = torch.empty((nq, 4, 128), dtype=torch.float32, device=dev)

    def step():
        qsa.block_scores_gmax(q, kb, W.active, out=s, gmax_out=gm)
        qsa.block_topk_gmax(s, gm, k, out=ids)
        qsa.sparse_attn(q, kc, ks, vc, vs, ids, out=out)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.synchronize()
    S = s.cpu().numpy()
    want_ids = o.topk_f32(S, k)
    want_out = o.sparse_attn(A.q, A.kc, A.ks, A.vc, A.vs, want_ids)
    keep, out0 = [], None
    for _ in range(40):
        s.fill_(float("nan"))
        ids.fill_(-7)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(s.cpu().numpy(), S)
        assert np.array_equal(ids.cpu().numpy(), want_ids)
        if out0 is None:   # the attention itself: near the FP64 oracle, then bit-identical on every replay
            out0 = out.cpu().numpy()
            err = np.abs(out0.astype(np.float64) - want_out).max()
            assert err <= 1e-4 * max(1.0, np.abs(want_out).max()), err
        assert np.array_equal(out.cpu().numpy(), out0)
        _churn(nq, W.active, k, dev, keep)
    assert qsa.device_error(dev) == 0
