"""qsa_block_select_small: scores and top-k for 1..4 queries in one
cooperative launch, against the plain calls (bit-identical scores and ids)
and the oracle's top-k of those scores. CPU tests check the argument and
size errors (nothing is launched for them)."""
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


def test_select_small_argument_and_size_errors(lib):
    f = lib.qsa_block_select_small
    OK, INVALID, UNSUPPORTED = qsa.QSA_OK, qsa.QSA_ERR_INVALID, qsa.QSA_ERR_UNSUPPORTED
    assert f(A, B, None, None, 5, 100, 50, 5, A, B, None) == UNSUPPORTED      # nq > 4
    assert f(A, B, B, B, 2, 100, 50, 5, A, B, None) == INVALID               # both key forms
    assert f(A, None, None, None, 2, 100, 50, 5, A, B, None) == INVALID      # no keys
    assert f(A, None, B, None, 2, 100, 50, 5, A, B, None) == INVALID         # int8 keys without scales
    assert f(A, None, B, B + 1, 2, 100, 50, 5, A, B, None) == INVALID        # odd scale address
    assert f(A, B, None, None, 2, 100, 50, 0, A, B, None) == INVALID         # k < 1
    assert f(A, B, None, None, 2, 100, 50, 5, A, MIS, None) == INVALID       # misaligned ids
    assert f(A, B, None, None, 2, 10 ** 6, qsa.TOPK_MAX_ACTIVE + 1, 5, A, B, None) == UNSUPPORTED
    assert f(None, None, None, None, 0, 100, 50, 5, None, None, None) == OK  # no rows


def _case(kind, nq, active, k, dev):
    import torch
    from sparse_attention_kv_qsa_gb300 import workloads as w
    if kind == "f32":
        W = w.normal_case(nq, active, k)
        q, kb = torch.from_numpy(W.q).to(dev), torch.from_numpy(np.ascontiguousarray(W.kblk)).to(dev)
        ref = qsa.block_scores(q, kb, active)
        return ref, (lambda: qsa.block_select_small(q, active, k, kblk=kb))
    W = w.int8_case(nq, active, k)
    q, kq = torch.from_numpy(W.q).to(dev), torch.from_numpy(W.kq8).to(dev)
    ks = torch.from_numpy(W.kscale.view(np.int16)).to(dev)
    ref = qsa.block_scores_q8(q, kq, ks, active)
    return ref, (lambda: qsa.block_select_small(q, active, k, kblk_q8=kq, kscale_f16=ks))


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["f32", "q8"])
@pytest.mark.parametrize("nq,active,k", [(1, 65536, 128), (4, 65536, 128), (3, 4099, 60), (2, 1000, 15),
                                         (1, 31, 1), (4, 33, 40), (2, 16384, 1025), (1, 393215, 1200),
                                         (4, 131072, 512), (2, 50, 50)])
def test_select_small_matches_plain_calls_and_oracle(kind, nq, active, k):
    import torch
    import oracle
    dev = torch.device("cuda:0")
    ref, run = _case(kind, nq, active, k, dev)
    s, ids = run()
    ids_plain = qsa.block_topk(ref, k)
    torch.cuda.synchronize()
    assert torch.equal(s, ref)
    assert torch.equal(ids, ids_plain)
    assert np.array_equal(ids.cpu().numpy(), oracle.get().topk_f32(ref.cpu().numpy(), k))
    assert qsa.device_error(dev) == 0


@pytest.mark.gpu
def test_select_small_repeated_calls_and_ties():
    """Back-to-back calls on one stream (each call's grid barrier uses the
    counter its predecessor cleared, by generation parity), on integer keys
    whose scores tie heavily."""
    import torch
    import oracle
    from sparse_attention_kv_qsa_gb300 import workloads as w
    dev = torch.device("cuda:0")
    W = w.integer_valued(4, 65536, lo=-1, hi=1)
    q, kb = torch.from_numpy(W.q).to(dev), torch.from_numpy(np.ascontiguousarray(W.kblk)).to(dev)
    ref = qsa.block_scores(q, kb, W.active)
    want = oracle.get().topk_f32(ref.cpu().numpy(), 256)
    s = torch.empty_like(ref)
    ids = torch.empty((4, 256), dtype=torch.int32, device=dev)
    free0 = None
    for i in range(30):
        ids.fill_(-7)
        qsa.block_select_small(q, W.active, 256, kblk=kb, scores_out=s, ids_out=ids)
        if i == 0:
            torch.cuda.synchronize()
            free0, _ = torch.cuda.mem_get_info(dev)
        assert np.array_equal(ids.cpu().numpy(), want), i
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free0      # nothing allocated per call
    assert qsa.device_error(dev) == 0
