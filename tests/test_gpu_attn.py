"""qsa_sparse_attn: attention of each query's 4 heads over the int8 KV cells
of its selected blocks, against the FP64 oracle.

Tolerance, derived from the kernel's fp32 arithmetic (u = 2^-24): a logit is
a 128-term dot product (4-term FMA chains, then a 5-level shuffle tree) times
the key scale and the temperature, so its error is at most ~16 u S_c with
S_c = T ks[c] sum_d |q_hd kq_cd|; a logit error d changes every softmax
weight by a relative factor of at most 2 d; the fp32 accumulation of the
weighted values (online rescaling per step, the warp and cluster merges,
expf within 2 ulp) adds at most ~256 u of the largest value. So

    |out - out64| <= max_c |v[c]| * (32 u max_c S_c + 256 u)

per (query, head), with the maxima over the query's attended cells.

Queries at least as many as the SMs take the tensor-core kernel: q (scaled
per head by a power of two) and the weights p * vs (likewise) enter the
MMAs as binary16 high parts plus remainders times 2^11, about 2^-22
relative each, and the MMAs accumulate in fp32; the logits and the weighted
sums then stay within the same bound. Its cases use nq >= 152 (the GB300's
SM count; the test asserts the device has no more). CPU tests check the
argument errors (nothing is launched for them)."""
import numpy as np
import pytest

from sparse_attention_kv_qsa_gb300 import build as qsa_build
from sparse_attention_kv_qsa_gb300 import qsa

A = 0x10000      # fake, 16-byte aligned "device" addresses: never dereferenced
B = 0x20000
MIS = 0x20004
U = 2.0 ** -24
T = 1.0 / np.sqrt(128.0)


@pytest.fixture(scope="module")
def lib():
    qsa_build.build()
    return qsa.lib()


def test_sparse_attn_argument_errors(lib):
    f = lib.qsa_sparse_attn
    OK, INVALID = qsa.QSA_OK, qsa.QSA_ERR_INVALID
    assert f(A, B, B, B, B, 100, A, -1, 4, A, None) == INVALID       # nq < 0
    assert f(A, B, B, B, B, 100, A, 2, 0, A, None) == INVALID        # k < 1
    assert f(A, B, B, B, B, -4, A, 2, 4, A, None) == INVALID         # ncells < 0
    assert f(None, B, B, B, B, 100, A, 2, 4, A, None) == INVALID     # no q
    assert f(A, B, B, B, B, 100, None, 2, 4, A, None) == INVALID     # no ids
    assert f(A, B, B, B, B, 100, A, 2, 4, None, None) == INVALID     # no out
    assert f(A, B, B, B, B, 100, A, 2, 4, MIS, None) == INVALID      # misaligned out
    assert f(A, MIS, B, B, B, 100, A, 2, 4, A, None) == INVALID      # misaligned key cells
    assert f(A, B, B + 1, B, B, 100, A, 2, 4, A, None) == INVALID    # odd key-scale address
    assert f(A, B, B, B, None, 100, A, 2, 4, A, None) == INVALID     # no value scales
    assert f(None, None, None, None, None, 0, None, 0, 4, None, None) == OK   # no queries
    assert f(A, B, B, B, B, 2 ** 31 - 2, A, 2, 4, A, None) == qsa.QSA_ERR_UNSUPPORTED   # cell indices past int


def tolerance(q, kc, ks, vc, vs, ids) -> np.ndarray:
    """The derived bound per (query, head), ``[nq, 4]``."""
    nq, k = ids.shape
    ncells = kc.shape[0]
    nblocks = (ncells + 3) // 4
    ksf = ks.view(np.float16).astype(np.float64)
    vsf = vs.view(np.float16).astype(np.float64)
    tol = np.zeros((nq, 4))
    for i in range(nq):
        b = ids[i][(ids[i] >= 0) & (ids[i] < nblocks)].astype(np.int64)
        cells = (4 * b[:, None] + np.arange(4)[None, :]).ravel()
        cells = cells[cells < ncells]
        if cells.size == 0:
            continue
        vmax = np.max(np.abs(vc[cells].astype(np.float64)) * vsf[cells, None])
        S = T * ksf[cells, None] * (np.abs(kc[cells].astype(np.float64)) @ np.abs(q[i].astype(np.float64)).T)
        tol[i] = vmax * (32 * U * S.max(axis=0) + 256 * U)
    return tol


def _run(W, dev):
    import torch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    ks = torch.from_numpy(W.ks.view(np.int16)).to(dev)
    vs = torch.from_numpy(W.vs.view(np.int16)).to(dev)
    return qsa.sparse_attn(t(W.q), t(W.kc), ks, t(W.vc), vs, t(W.ids))


def _check(W, out):
    import oracle
    want = oracle.get().sparse_attn(W.q, W.kc, W.ks, W.vc, W.vs, W.ids)
    got = out.cpu().numpy().astype(np.float64)
    err = np.abs(got - want).max(axis=2)
    tol = tolerance(W.q, W.kc, W.ks, W.vc, W.vs, W.ids)
    assert np.all(err <= tol), (err.max(), tol.min())
    return err


@pytest.mark.gpu
@pytest.mark.parametrize("nq,ncells,k,pad", [(1, 262144, 128, 0),      # decode: clusters of 4
                                             (4, 262144, 128, 0),
                                             (30, 65536, 256, 3),       # clusters of 4
                                             (60, 16384, 64, 0),        # pairs
                                             (100, 16384, 512, 17),     # tensor cores: more than half the SMs
                                             (3, 4099 * 4 + 3, 60, 7),  # partial last block
                                             (2, 17, 5, 0),             # every block, ragged
                                             (5, 4096, 1, 0),           # one block
                                             (2, 262144, 4096, 0),      # long lists: 16,384 cells per query
                                             (7, 65536, 300, 290),      # mostly padding
                                             # tensor-core kernel (nq >= SMs):
                                             (200, 16384, 512, 17),
                                             (256, 262144, 512, 0),     # the bench's many-query shape
                                             (152, 4099 * 4 + 3, 60, 7),
                                             (160, 17, 5, 0),
                                             (152, 4096, 1, 0),
                                             (153, 65536, 300, 290),
                                             (152, 262144, 4096, 0),    # 16,384 cells per query
                                             # 8-warp CTAs, two per SM (SMs < nq <= 2 SMs) and
                                             # 4-warp CTAs, four per SM (beyond; 640: more than one wave):
                                             (305, 16384, 512, 17),
                                             (400, 65536, 300, 290),
                                             (640, 4099 * 4 + 3, 64, 0)])
def test_sparse_attn_matches_oracle(nq, ncells, k, pad):
    import torch
    from sparse_attention_kv_qsa_gb300 import workloads as w
    dev = torch.device("cuda:0")
    assert torch.cuda.get_device_properties(dev).multi_processor_count <= 152
    W = w.attn_case(nq, ncells, k, pad=pad)
    out = _run(W, dev)
    torch.cuda.synchronize()
    _check(W, out)
    again = _run(W, dev)
    torch.cuda.synchronize()
    assert torch.equal(out, again)          # fixed merge order: bit-identical reruns
    assert qsa.device_error(dev) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("nq", [4, 160, 320])   # CUDA-core / tensor-core kernel (8- and 4-warp CTAs)
def test_sparse_attn_padding_duplicates_and_empty(nq):
    """All-padding rows give zeros; ids past the last block are skipped; a
    block listed twice counts twice; no cells at all gives zeros."""
    import torch
    from sparse_attention_kv_qsa_gb300 import workloads as w
    dev = torch.device("cuda:0")
    W = w.attn_case(nq, 1000, 6)
    W.ids[0] = -1
    W.ids[1] = [5, 5, 5, 7, 9999, -3]
    W.ids[2] = [249, 249, 0, 1, 2, 3]        # block 249 = cells 996..999
    out = _run(W, dev)
    torch.cuda.synchronize()
    _check(W, out)
    assert torch.count_nonzero(out[0]) == 0
    empty = w.attn_case(nq, 8, 2)
    empty.kc, empty.vc = empty.kc[:0], empty.vc[:0]
    empty.ks, empty.vs = empty.ks[:0], empty.vs[:0]
    z = _run(empty, dev)
    torch.cuda.synchronize()
    assert torch.count_nonzero(z) == 0


def _rescale_half(bits, mul):
    return (bits.view(np.float16).astype(np.float64) * mul).astype(np.float16).view(np.uint16)


@pytest.mark.gpu
@pytest.mark.parametrize("nq", [8, 160, 320])   # CUDA-core / tensor-core kernel (8- and 4-warp CTAs)
@pytest.mark.parametrize("qmul,vsmul,ksmul", [(1e5, 1.0, 1.0),     # near one-hot softmax
                                              (1e-20, 1.0, 1.0),   # uniform softmax, tiny q
                                              (1.0, 6.0e5, 1.0),   # value scales up to 6e4
                                              (1.0, 1e-4, 1.0),    # binary16-subnormal value scales
                                              (1.0, 1.0, 1e-4)])   # binary16-subnormal key scales
def test_sparse_attn_input_ranges(nq, qmul, vsmul, ksmul):
    """Inputs far from the recipe's ranges: the tensor-core kernel's power-of-two
    scalings keep its binary16 operands finite and normal, so both kernels
    stay within the derived bound."""
    import torch
    from sparse_attention_kv_qsa_gb300 import workloads as w
    dev = torch.device("cuda:0")
    W = w.attn_case(nq, 4099 * 4 + 1, 40, pad=3)
    W.q = (W.q.astype(np.float64) * qmul).astype(np.float32)
    W.vs = _rescale_half(W.vs, vsmul)
    W.ks = _rescale_half(W.ks, ksmul)
    assert np.all(np.isfinite(W.vs.view(np.float16))) and np.all(W.vs.view(np.float16) != 0)
    out = _run(W, dev)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    _check(W, out)


@pytest.mark.gpu
def test_sparse_attn_after_topk():
    """The decode pipeline: one-launch scores + top-k on the decode keys, then
    attention over the selected blocks' cells (KV cells from the attention
    recipe, 4 per block), against the oracle on those ids."""
    import torch
    from sparse_attention_kv_qsa_gb300 import workloads as w
    dev = torch.device("cuda:0")
    D = w.decode(4, 262144)
    q = torch.from_numpy(D.q).to(dev)
    kq = torch.from_numpy(D.kq8).to(dev)
    ks = torch.from_numpy(D.kscale.view(np.int16)).to(dev)
    _, ids = qsa.block_select_small(q, D.active, D.k, kblk_q8=kq, kscale_f16=ks)
    W = w.attn_case(4, 4 * D.active, D.k)
    W.q = D.q
    W.ids = ids.cpu().numpy()
    out = _run(W, dev)
    torch.cuda.synchronize()
    _check(W, out)
