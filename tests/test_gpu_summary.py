"""qsa_block_summary: block summary keys from int8 KV cells, against the
oracle's fp32 restatement, bit for bit (keys, int8 codes and binary16
scales), over whole pools, sub-ranges, ragged tails, empty blocks, and a
cell-by-cell append. CPU tests check the argument errors (nothing is
launched for them)."""
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


def test_block_summary_argument_errors(lib):
    f = lib.qsa_block_summary
    OK, INVALID = qsa.QSA_OK, qsa.QSA_ERR_INVALID
    assert f(A, B, -1, 0, 4, A, None, None, None) == INVALID        # ncells < 0
    assert f(A, B, 16, -1, 4, A, None, None, None) == INVALID       # begin < 0
    assert f(A, B, 16, 5, 4, A, None, None, None) == INVALID        # end < begin
    assert f(A, B, 16, 0, 4, None, None, None, None) == INVALID     # no output
    assert f(A, B, 16, 0, 4, None, A, None, None) == INVALID        # codes without scales
    assert f(A, B, 16, 0, 4, MIS, None, None, None) == INVALID      # misaligned keys
    assert f(MIS, B, 16, 0, 4, A, None, None, None) == INVALID      # misaligned cells
    assert f(A, B + 1, 16, 0, 4, A, None, None, None) == INVALID    # odd cell-scale address
    assert f(A, B, 16, 0, 4, None, A, B + 1, None) == INVALID       # odd block-scale address
    assert f(None, None, 16, 0, 4, A, None, None, None) == INVALID  # cells missing
    assert f(A, B, 16, 3, 3, A, None, None, None) == OK             # empty range
    assert f(A, B, 16, 0, 2 ** 29, A, None, None, None) == qsa.QSA_ERR_UNSUPPORTED   # cell indices past int


def _pool(ncells, seed_index=11):
    from sparse_attention_kv_qsa_gb300 import workloads as w
    W = w.attn_case(1, ncells, 1, config_index=seed_index)
    return W.kc, W.ks


def _dev_buffers(nrows, dev):
    import torch
    key = torch.full((nrows, 128), float("nan"), dtype=torch.float32, device=dev)
    q8 = torch.full((nrows, 128), 99, dtype=torch.int8, device=dev)
    sc = torch.full((nrows,), 0x7E00, dtype=torch.int16, device=dev)   # binary16 NaN sentinel
    return key, q8, sc


@pytest.mark.gpu
@pytest.mark.parametrize("ncells,b0,b1", [(4099 * 4 + 3, 0, 4101), (262144, 0, 65536), (65536, 100, 357),
                                          (4099 * 4 + 3, 4099, 4100), (17, 0, 8), (0, 0, 3)])
def test_block_summary_matches_oracle(ncells, b0, b1):
    import torch
    import oracle
    dev = torch.device("cuda:0")
    kc, ks = _pool(max(ncells, 1))
    kc, ks = kc[:ncells], ks[:ncells]
    key, q8, sc = _dev_buffers(b1 + 2, dev)
    qsa.block_summary(torch.from_numpy(np.ascontiguousarray(kc)).to(dev), torch.from_numpy(ks.view(np.int16)).to(dev),
                      b0, b1, kblk=key, kblk_q8=q8, kblk_scale_f16=sc)
    torch.cuda.synchronize()
    wk, wq, ws = oracle.get().block_summary(kc.reshape(ncells, 128), ks, b0, b1)
    assert np.array_equal(key[b0:b1].cpu().numpy().view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(q8[b0:b1].cpu().numpy(), wq)
    assert np.array_equal(sc[b0:b1].cpu().numpy().view(np.uint16), ws)
    # rows outside the range are untouched
    assert torch.isnan(key[:b0]).all() and torch.isnan(key[b1:]).all()
    assert (q8[b1:] == 99).all() and (sc[b1:] == 0x7E00).all()
    assert qsa.device_error(dev) == 0


@pytest.mark.gpu
def test_block_summary_append_cell_by_cell():
    """Appending cells one at a time and refreshing the touched block each
    time gives the same summaries as one pass over the final pool; the fp32
    form alone and the int8 form alone give the same rows as both."""
    import torch
    import oracle
    dev = torch.device("cuda:0")
    kc, ks = _pool(4096 + 9)
    kc_d = torch.from_numpy(np.ascontiguousarray(kc)).to(dev)
    ks_d = torch.from_numpy(ks.view(np.int16)).to(dev)
    key, q8, sc = _dev_buffers(1030, dev)
    qsa.block_summary(kc_d[:4096], ks_d[:4096], 0, 1024, kblk=key, kblk_q8=q8, kblk_scale_f16=sc)
    for n in range(4097, 4096 + 10):
        qsa.block_summary(kc_d[:n], ks_d[:n], (n - 1) // 4, (n + 3) // 4, kblk=key, kblk_q8=q8, kblk_scale_f16=sc)
    key_only, q8_only, sc_only = _dev_buffers(1030, dev)
    qsa.block_summary(kc_d, ks_d, 0, 1027, kblk=key_only)
    qsa.block_summary(kc_d, ks_d, 0, 1027, kblk_q8=q8_only, kblk_scale_f16=sc_only)
    torch.cuda.synchronize()
    wk, wq, ws = oracle.get().block_summary(kc, ks, 0, 1027)
    for k_, q_, s_ in ((key, q8, sc), (key_only, q8_only, sc_only)):
        assert np.array_equal(k_[:1027].cpu().numpy().view(np.uint32), wk.view(np.uint32))
        assert np.array_equal(q_[:1027].cpu().numpy(), wq)
        assert np.array_equal(s_[:1027].cpu().numpy().view(np.uint16), ws)


@pytest.mark.gpu
def test_block_summary_feeds_the_int8_scorer():
    """The int8 summaries and scales are the qsa_block_scores_q8 key layout:
    scoring them equals scoring the same summaries through the oracle."""
    import torch
    import oracle
    from sparse_attention_kv_qsa_gb300 import workloads as w
    dev = torch.device("cuda:0")
    kc, ks = _pool(8192)
    key, q8, sc = _dev_buffers(2048, dev)
    qsa.block_summary(torch.from_numpy(np.ascontiguousarray(kc)).to(dev), torch.from_numpy(ks.view(np.int16)).to(dev),
                      0, 2048, kblk_q8=q8, kblk_scale_f16=sc)
    q = w.normal_case(3, 16, 4).q
    s = qsa.block_scores_q8(torch.from_numpy(q).to(dev), q8, sc, 2048)
    torch.cuda.synchronize()
    S = oracle.get().scores_q8(q, q8.cpu().numpy(), sc.cpu().numpy().view(np.uint16), 2048)
    tol = 1e-6 * np.abs(S).max(axis=1, keepdims=True)
    assert np.all(np.abs(s.cpu().numpy().astype(np.float64) - S) <= tol)
