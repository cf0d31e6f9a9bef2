"""qsa_block_select_static: scores and exact top-k in one call that allocates
nothing (its group-maximum scratch is a fixed 1 MiB device array in the
library image).

CPU tests check its argument and size errors (nothing is launched for
them); GPU tests check its results against the two-call path and the oracle,
and that repeated calls leave the device's free memory unchanged.
"""
import ctypes

import numpy as np
import pytest

from sparse_attention_kv_qsa_gb300 import build as qsa_build
from sparse_attention_kv_qsa_gb300 import qsa

A = 0x10000      # fake, 16-byte aligned "device" addresses: never dereferenced
B = 0x20000
MIS = 0x20004


@pytest.fixture(scope="module")
def lib():
    qsa_build.build()
    return qsa.lib()


def test_static_select_argument_and_size_errors(lib):
    f = lib.qsa_block_select_static
    OK, INVALID, UNSUPPORTED = qsa.QSA_OK, qsa.QSA_ERR_INVALID, qsa.QSA_ERR_UNSUPPORTED
    assert f(A, B, 8, 100, 50, 0, A, B, None) == INVALID        # k < 1
    assert f(A, B, 8, 100, 50, 5, A, None, None) == INVALID     # null ids
    assert f(A, B, 8, 100, 50, 5, A, MIS, None) == INVALID      # misaligned ids
    assert f(A, None, 8, 100, 50, 5, A, B, None) == INVALID     # null keys
    assert f(A, B, 8, 100, 101, 5, A, B, None) == INVALID       # active > max_blocks
    assert f(None, None, 0, 100, 50, 5, None, None, None) == OK  # no rows
    # the scratch bound: nq * ceil(active / 32) groups
    gmax = qsa.SELECT_STATIC_GROUPS_MAX
    assert f(A, B, 257, 40000, 32768, 5, A, B, None) == UNSUPPORTED
    assert f(A, B, 1, 10 ** 7, 32 * gmax + 1, 5, A, B, None) == UNSUPPORTED
    # within the scratch bound but past the top-k's row limit: refused before
    # the scorer launches (these fake pointers would fault a launched kernel)
    assert f(A, B, 1, 10 ** 7, qsa.TOPK_MAX_ACTIVE + 1, 5, A, B, None) == UNSUPPORTED
    assert f(A, B, 1, 10 ** 7, 400000, 5, A, B, None) == UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("nq,active,k", [(37, 4099, 60), (8, 65536, 512), (3, 65536, 128), (256, 32768, 256),
                                         (5, 1000, 1000), (4, 31, 40)])
def test_static_select_matches_two_calls_and_oracle(nq, active, k):
    import torch
    import oracle
    from sparse_attention_kv_qsa_gb300 import workloads as w
    dev = torch.device("cuda:0")
    W = w.normal_case(nq, active, k)
    q = torch.from_numpy(W.q).to(dev)
    kb = torch.from_numpy(np.ascontiguousarray(W.kblk)).to(dev)
    s, ids = qsa.block_select_static(q, kb, active, k)
    s2, ids2 = qsa.block_select_gmax(q, kb, active, k)
    torch.cuda.synchronize()
    assert torch.equal(s, s2)
    assert torch.equal(ids, ids2)
    assert np.array_equal(ids.cpu().numpy(), oracle.get().topk_f32(s.cpu().numpy(), k))


@pytest.mark.gpu
def test_static_select_allocates_nothing():
    import torch
    from sparse_attention_kv_qsa_gb300 import workloads as w
    dev = torch.device("cuda:0")
    W = w.normal_case(128, 65536, 512)
    q = torch.from_numpy(W.q).to(dev)
    kb = torch.from_numpy(np.ascontiguousarray(W.kblk)).to(dev)
    s = torch.empty((128, 65536), dtype=torch.float32, device=dev)
    ids = torch.empty((128, 512), dtype=torch.int32, device=dev)
    qsa.block_select_static(q, kb, 65536, 512, scores_out=s, ids_out=ids)   # first call: warm everything up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    for _ in range(20):
        qsa.block_select_static(q, kb, 65536, 512, scores_out=s, ids_out=ids)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0
    assert torch.cuda.memory_allocated(dev) == alloc0
    assert qsa.device_error(dev) == 0


@pytest.mark.gpu
def test_static_select_past_the_scratch_raises():
    import torch
    dev = torch.device("cuda:0")
    q = torch.zeros((257, 4, 128), dtype=torch.float32, device=dev)
    kb = torch.zeros((32768, 128), dtype=torch.float32, device=dev)
    with pytest.raises(qsa.QSAError):
        qsa.block_select_static(q, kb, 32768, 8)
