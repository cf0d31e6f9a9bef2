"""The bounded waits' failure path, made to run on the GPU without a fault.

A diagnostic call (qsa_debug_inject) plants a wait that can never complete
and shortens every wait's limit to 1 ms: the scorer's CTA 0 never loads one
key piece, or the fused decode select's grid barrier waits for one arrival
more than its grid has. The call must end within a fraction of a second (the
scorer's CTA abandons its other waits at once instead of running each out),
report the time-out in the device error word, and leave the device usable:
the next normal call returns the oracle's results and no error.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import parity
import sparse_attention_kv_qsa_gb300 as qsa
from sparse_attention_kv_qsa_gb300 import qsa as Q
from sparse_attention_kv_qsa_gb300 import workloads as w

pytestmark = pytest.mark.gpu
LIMIT_NS = 1_000_000   # 1 ms


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    assert qsa.device_error(d) == 0
    yield d
    Q.debug_inject(0)


def to_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _normal_call_is_exact(dev):
    W = w.normal_case(nq=256, active=4099, k=100, max_blocks=4101)
    s = qsa.block_scores(to_dev(W.q, dev), to_dev(W.kblk, dev), W.active)
    ids = qsa.block_topk(s, W.k)
    torch.cuda.synchronize()
    o = oracle.get()
    S = s.cpu().numpy()
    parity.check_scores(S, o.scores(W.q, W.kblk, W.active))
    assert np.array_equal(ids.cpu().numpy(), o.topk_f32(S, W.k))
    assert qsa.device_error(dev) == 0


@pytest.mark.parametrize("pair_mode", [True, False])
def test_scorer_wait_runs_out_and_the_cta_aborts(dev, pair_mode):
    # 256 queries: 2 query groups (CTA pairs at full size); 200 queries with a
    # 1-tile key range: one CTA per group and tile sequence, no pair.
    nq, active = (256, 65536) if pair_mode else (200, 100)
    W = w.normal_case(nq=nq, active=active, k=8)
    q, kb = to_dev(W.q, dev), to_dev(W.kblk, dev)
    torch.cuda.synchronize()
    Q.debug_inject(Q.INJECT_SCORER_STALL, LIMIT_NS)
    try:
        t0 = time.perf_counter()
        qsa.block_scores(q, kb, W.active)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        Q.debug_inject(0)
    code = qsa.device_error(dev)
    assert code & 0x100, hex(code)
    assert dt < 0.5, f"the aborted call took {dt:.3f} s"
    _normal_call_is_exact(dev)


def test_decode_grid_barrier_runs_out(dev):
    W = w.decode(1, 262144)
    q, kq = to_dev(W.q, dev), to_dev(W.kq8, dev)
    ks = to_dev(W.kscale.view(np.int16), dev)
    torch.cuda.synchronize()
    Q.debug_inject(Q.INJECT_DECODE_BARRIER, LIMIT_NS)
    try:
        t0 = time.perf_counter()
        qsa.block_select_small(q, W.active, W.k, kblk_q8=kq, kscale_f16=ks)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        Q.debug_inject(0)
    code = qsa.device_error(dev)
    assert code & 0x2, hex(code)
    assert dt < 0.5, f"the call took {dt:.3f} s"
    # the next calls (its barrier's counters included) are normal again
    for _ in range(3):
        s, ids = qsa.block_select_small(q, W.active, W.k, kblk_q8=kq, kscale_f16=ks)
    torch.cuda.synchronize()
    assert qsa.device_error(dev) == 0
    o = oracle.get()
    assert np.array_equal(ids.cpu().numpy(), o.topk_f32(s.cpu().numpy(), W.k))
    _normal_call_is_exact(dev)
