"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with something the pages or the mathematics fix:

- brute force over every k-subset of tiny rows (the unique subset that
  dominates its complement under "higher score, then lower id");
- hand-derived scores with closed forms (one-hot queries, all-tie rows);
- exact integer arithmetic (numpy int64) and library float64 matmul;
- numpy's binary16 conversion over all 65,536 bit patterns;
- invariants of an exact selection, padding and capacity independence;
- a hand-computed golden fixture (``golden/hand_scores.json``).

The definition being pinned: score = sum over the 4 query heads of the
head's dot product with the block's summary key, over active blocks only
("#3108 optimize exact QSA block scoring and top-k selection on gfx12",
Summary items 1 and 4; "#337 gfx12 QSA select", What items 1-2); the top-k
is exact with ties broken by lower block id and ids returned ascending.

``test_oracle_mutants.py`` runs every pin against deliberately broken
builds of the oracle to show that the pins catch plausible mistakes.
"""

from __future__ import annotations

import itertools
import json
import os

import numpy as np

H, D = 4, 128
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed: int) -> np.random.Generator:
    # test-local randomness for pin construction only (never a parity input)
    return np.random.default_rng(seed)


def _dominates(vals: np.ndarray, subset: tuple[int, ...]) -> bool:
    """True iff every member beats every non-member (value desc, id asc)."""
    inside = set(subset)
    def rank(i):
        v = -np.inf if np.isnan(vals[i]) else float(vals[i])   # NaN counts as -inf
        return (v, -i)
    for i in inside:
        for j in range(len(vals)):
            if j not in inside and not rank(i) > rank(j):
                return False
    return True


def brute_force_topk(vals: np.ndarray, k: int) -> np.ndarray:
    n = len(vals)
    m = min(k, n)
    winners = [s for s in itertools.combinations(range(n), m) if _dominates(vals, s)]
    assert len(winners) == 1, f"expected exactly one dominating subset, got {len(winners)}"
    out = np.full(k, -1, dtype=np.int32)
    out[:m] = sorted(winners[0])
    return out


def pin_brute_force_topk(o) -> None:
    r = _rng(11)
    rows = []
    for n in range(1, 10):
        rows.append(r.normal(size=n))                                   # distinct
        rows.append(r.integers(-2, 3, size=n).astype(np.float64))       # many ties
        rows.append(np.where(r.random(n) < 0.5, 0.0, -0.0))             # +-0 ties
    rows.append(np.array([1.0, np.nan, 1.0, -np.inf, np.inf, np.nan, -1.0]))
    rows.append(np.array([np.nan, -np.inf, 2.0, np.nan, -np.inf]))
    for vals in rows:
        n = len(vals)
        for k in range(1, n + 3):
            want = brute_force_topk(vals, k)
            got32 = o.topk_f32(vals.astype(np.float32)[None, :], k)[0]
            got64 = o.topk_f64(vals[None, :], k)[0]
            assert np.array_equal(got32, want), (vals, k, got32, want)
            assert np.array_equal(got64, want), (vals, k, got64, want)


def _onehot_workload(nq: int, active: int):
    """q[i][h] = e_{4i+h}; kblk[b][d] = b - d.  Then
    S[i][b] = sum_h kblk[b][4i+h] = sum_h (b - 4i - h) = 4b - 16i - 6."""
    q = np.zeros((nq, H, D), dtype=np.float32)
    for i in range(nq):
        for h in range(H):
            q[i, h, 4 * i + h] = 1.0
    b = np.arange(active, dtype=np.float32)[:, None]
    d = np.arange(D, dtype=np.float32)[None, :]
    return q, (b - d).astype(np.float32)


def pin_closed_form_onehot(o) -> None:
    nq, active = 5, 300
    q, kblk = _onehot_workload(nq, active)
    S = o.scores(q, kblk, active)
    i = np.arange(nq)[:, None]
    b = np.arange(active)[None, :]
    assert np.array_equal(S, (4 * b - 16 * i - 6).astype(np.float64))
    for k in (1, 7, 64, 299, 300, 301):
        ids = o.topk_f64(S, k)
        m = min(k, active)
        want = np.concatenate([np.arange(active - m, active), -np.ones(k - m)]).astype(np.int32)
        assert all(np.array_equal(row, want) for row in ids), (k, ids[0][:8])


def pin_all_ties_lower_id(o) -> None:
    """Every block holds the same key, so every score ties; the lower-id
    rule then selects ids 0..k-1. The same key with a sign flip on odd
    blocks splits the row into two tie groups."""
    nq, active = 3, 50
    q = np.tile(np.arange(1, H + 1, dtype=np.float32)[None, :, None], (nq, 1, D))
    key = (np.arange(D) % 7 - 3).astype(np.float32)
    kblk = np.tile(key, (active, 1))
    S = o.scores(q, kblk, active)
    assert np.all(S == S[0, 0]) and S[0, 0] == 10.0 * float(np.sum(key))
    for k in (1, 10, 49, 50):
        assert all(np.array_equal(r, np.arange(k)) for r in o.topk_f64(S, k))
    sgn = np.where(np.arange(active) % 2 == 0, 1.0, -1.0).astype(np.float32)
    key2 = np.ones(D, dtype=np.float32)
    kblk2 = (sgn[:, None] * key2[None, :]).astype(np.float32)
    S2 = o.scores(q, kblk2, active)
    ids = o.topk_f64(S2, 30)
    want = np.concatenate([np.arange(0, active, 2), np.arange(1, 11, 2)])
    assert all(np.array_equal(r, np.sort(want)) for r in ids), ids[0]


def pin_integer_exact(o) -> None:
    """Integer-valued inputs: compare with exact int64 arithmetic (numpy
    einsum on int64) and a library sort (numpy lexsort)."""
    r = _rng(7)
    for nq, active, k in ((3, 97, 10), (4, 256, 255), (2, 33, 40)):
        q = r.integers(-8, 9, size=(nq, H, D))
        kb = r.integers(-8, 9, size=(active, D))
        S = o.scores(q.astype(np.float32), kb.astype(np.float32), active)
        exact = np.einsum("ihd,bd->ib", q.astype(np.int64), kb.astype(np.int64))
        assert np.array_equal(S, exact.astype(np.float64))
        ids = o.topk_f64(S, k)
        for i in range(nq):
            order = np.lexsort((np.arange(active), -exact[i]))
            m = min(k, active)
            want = np.concatenate([np.sort(order[:m]), -np.ones(k - m)]).astype(np.int32)
            assert np.array_equal(ids[i], want)


def pin_float_vs_numpy(o) -> None:
    """Random fp32 inputs: FP64 scores agree with numpy's float64 matmul to
    rounding (1e-12 of the row scale); ids agree with a lexsort of the
    oracle's own scores."""
    r = _rng(5)
    nq, active, k = 6, 777, 31
    q = r.normal(size=(nq, H, D)).astype(np.float32)
    kb = r.standard_t(3, size=(active, D)).astype(np.float32)
    S = o.scores(q, kb, active)
    ref = np.einsum("ihd,bd->ib", q.astype(np.float64), kb.astype(np.float64))
    scale = np.abs(ref).max(axis=1, keepdims=True)
    assert np.all(np.abs(S - ref) <= 1e-12 * scale)
    ids = o.topk_f64(S, k)
    for i in range(nq):
        order = np.lexsort((np.arange(active), -S[i]))
        assert np.array_equal(ids[i], np.sort(order[:k]))


def pin_half_to_double(o) -> None:
    """All 65,536 binary16 patterns against numpy's float16 conversion."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([o.half_to_double(int(h)) for h in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_q8_scores(o) -> None:
    """int8 keys times binary16 scales: exact against int64 arithmetic when
    q is integer-valued and the scales are powers of two; within rounding
    of numpy float64 otherwise."""
    r = _rng(3)
    nq, active = 3, 200
    kq = r.integers(-127, 128, size=(active, D)).astype(np.int8)
    e = r.integers(-10, -2, size=active)
    sc = (2.0 ** e).astype(np.float16).view(np.uint16)
    qi = r.integers(-8, 9, size=(nq, H, D))
    S = o.scores_q8(qi.astype(np.float32), kq, sc, active)
    exact = np.einsum("ihd,bd->ib", qi.astype(np.int64), kq.astype(np.int64)).astype(np.float64)
    assert np.array_equal(S, exact * (2.0 ** e)[None, :])
    sc2 = r.uniform(1e-3, 1e-1, size=active).astype(np.float16)
    qf = r.normal(size=(nq, H, D)).astype(np.float32)
    S2 = o.scores_q8(qf, kq, sc2.view(np.uint16), active)
    ref = np.einsum("ihd,bd->ib", qf.astype(np.float64),
                    kq.astype(np.float64) * sc2.astype(np.float64)[:, None])
    assert np.all(np.abs(S2 - ref) <= 1e-12 * np.abs(ref).max(axis=1, keepdims=True))


def pin_padding_and_empty(o) -> None:
    S = np.array([[3.0, 1.0, 2.0], [0.0, 0.0, -1.0]])
    assert np.array_equal(o.topk_f64(S, 5), [[0, 1, 2, -1, -1], [0, 1, 2, -1, -1]])
    assert np.array_equal(o.topk_f64(S, 2), [[0, 2], [0, 1]])
    assert np.array_equal(o.topk_f64(np.zeros((2, 0)), 3), -np.ones((2, 3), dtype=np.int32))


def pin_capacity_independence(o) -> None:
    """Only the first ``active`` key rows are read: NaN-filled capacity rows
    change nothing."""
    r = _rng(9)
    nq, active, cap = 2, 40, 47
    q = r.normal(size=(nq, H, D)).astype(np.float32)
    kb = r.normal(size=(cap, D)).astype(np.float32)
    kb_nan = kb.copy()
    kb_nan[active:] = np.nan
    S1 = o.scores(q, kb[:active].copy(), active)
    S2 = o.scores(q, kb_nan, active)
    assert S2.shape == (nq, active) and np.array_equal(S1, S2)
    kq = r.integers(-127, 128, size=(cap, D)).astype(np.int8)
    sc = np.full(cap, 0x7E00, dtype=np.uint16)
    sc[:active] = np.float16(0.01).view(np.uint16)
    assert not np.isnan(o.scores_q8(q, kq, sc, active)).any()


def pin_selection_invariants(o) -> None:
    """Exactness: unique, in-range ids; min(k, active) of them; every
    selected score >= every unselected one; boundary ties to lower ids."""
    r = _rng(13)
    for active, k in ((500, 50), (64, 64), (1000, 1)):
        S = np.round(r.normal(size=(4, active)) * 4) / 4      # coarse grid: many ties
        ids = o.topk_f64(S, k)
        for i in range(S.shape[0]):
            sel = ids[i][ids[i] >= 0]
            assert len(sel) == min(k, active) and len(np.unique(sel)) == len(sel)
            assert np.all(np.diff(sel) > 0) and sel.min() >= 0 and sel.max() < active
            mask = np.zeros(active, bool)
            mask[sel] = True
            if (~mask).any():
                lo_in, hi_out = S[i][mask].min(), S[i][~mask].max()
                assert lo_in >= hi_out
                if lo_in == hi_out:
                    tied_in = np.nonzero(mask & (S[i] == lo_in))[0]
                    tied_out = np.nonzero(~mask & (S[i] == lo_in))[0]
                    assert tied_in.max() < tied_out.min()


def pin_golden_hand(o) -> None:
    """Hand-derived scores and selections (see the fixture's derivation)."""
    with open(os.path.join(GOLDEN, "hand_scores.json")) as f:
        g = json.load(f)
    nq, active = g["nq"], g["active"]
    q = np.zeros((nq, H, D), dtype=np.float32)
    for i, h, d, v in g["q_nonzero"]:
        q[i, h, d] = v
    kb = np.zeros((active, D), dtype=np.float32)
    for b, d, v in g["kblk_nonzero"]:
        kb[b, d] = v
    S = o.scores(q, kb, active)
    assert np.array_equal(S, np.array(g["scores"], dtype=np.float64)), S
    for k, want in g["topk"].items():
        assert np.array_equal(o.topk_f64(S, int(k)), np.array(want, dtype=np.int32)), (k, want)


def pin_score_keys_order(o) -> None:
    """The radix key of the boundary header is order-preserving: on values
    listed in ascending order the keys ascend strictly, -0 and +0 share a
    key, NaN has the key of -inf; and on random pairs (with NaN read as -inf)
    key order equals value order."""
    f32 = np.float32
    asc = np.array([-np.inf, -3e38, -1.5, -1.0, -1e-30, -1e-45, 0.0, 1e-45, 1e-30, 1.0, 1.5, 3e38, np.inf],
                   dtype=f32)
    k = o.score_keys(asc)
    assert np.all(np.diff(k.astype(np.int64)) > 0)
    assert o.score_keys(np.array([-0.0], dtype=f32))[0] == o.score_keys(np.array([0.0], dtype=f32))[0]
    assert o.score_keys(np.array([np.nan], dtype=f32))[0] == o.score_keys(np.array([-np.inf], dtype=f32))[0]
    rng = _rng(61)
    v = rng.standard_normal(600).astype(f32) * f32(10.0) ** rng.integers(-30, 30, 600).astype(f32)
    v[::37] = np.nan
    v[5::41] = -0.0
    v[7::43] = 0.0
    kv = o.score_keys(v).astype(np.int64)
    w = np.where(np.isnan(v), -np.inf, v).astype(np.float64)
    assert np.array_equal(kv[:, None] < kv[None, :], w[:, None] < w[None, :])
    assert np.array_equal(kv[:, None] == kv[None, :], w[:, None] == w[None, :])


def pin_group_max_keys(o) -> None:
    """Group maxima: on an ascending row each group's maximum is its last
    element (the short last group too); on random rows with NaN and signed
    zeros it is the key of the element the oracle's own sort ranks first in
    that group."""
    f32 = np.float32
    row = np.linspace(-5, 5, 100, dtype=f32)[None, :]
    gm = o.group_max_keys(row)
    assert gm.shape == (1, 4)
    assert np.array_equal(gm[0], o.score_keys(row[0, [31, 63, 95, 99]]))
    rng = _rng(62)
    S = rng.standard_normal((3, 230)).astype(f32)
    S[0, ::11] = np.nan
    S[1, 40:72] = -0.0
    S[1, 50] = 0.0
    S[2, 200:230] = np.nan
    gm = o.group_max_keys(S)
    assert gm.shape == (3, 8)
    for g in range(8):
        part = np.ascontiguousarray(S[:, 32 * g:32 * g + 32])
        top = o.topk_f32(part, 1)[:, 0]
        assert np.array_equal(gm[:, g], o.score_keys(part[np.arange(3), top]))


# ---- attention over the selected blocks ------------------------------------
# The definition pinned: query i's 4 heads attend the cells of its listed
# blocks (block b = cells 4b .. 4b+3 below ncells; negative or past-the-end
# ids are padding), key/value = int8 x one binary16 scale per cell, logits
# scaled by 1/sqrt(128), softmax per head, output the weighted sum of values
# ("#3224 [Engine] perf(hip): tune RDNA4 QSA prompt WMMA path", Summary and
# Evidence section 2; "#3102 perf(hip): enable wave32 QSA decode attention and
# MMVQ row reuse on gfx12", item D5).

def _half_bits(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def _attn_case(ncells: int, seed: int):
    r = _rng(seed)
    kq = r.integers(-127, 128, (ncells, D)).astype(np.int8)
    vq = r.integers(-127, 128, (ncells, D)).astype(np.int8)
    ks = _half_bits(r.uniform(0.002, 0.02, ncells))
    vs = _half_bits(r.uniform(0.01, 0.1, ncells))
    return kq, vq, ks, vs


def pin_attn_single_cell(o) -> None:
    """One attended cell: every head's output is that cell's value exactly
    (weight 1), whatever the query."""
    kq, vq, ks, vs = _attn_case(9, 101)          # block 2 holds only cell 8
    q = _rng(102).standard_normal((3, H, D)).astype(np.float32)
    ids = np.array([[2, -1], [-1, 2], [2, 7]], dtype=np.int32)   # 7 is past the last block
    out = o.sparse_attn(q, kq, ks, vq, vs, ids)
    value = vq[8].astype(np.float64) * float(np.uint16(vs[8]).view(np.float16))
    for i in range(3):
        for h in range(H):
            assert np.array_equal(out[i, h], value), (i, h)


def pin_attn_uniform_weights(o) -> None:
    """Zero keys give equal logits, so each head's output is the plain mean
    of the attended values (numpy, cell by cell)."""
    _, vq, ks, vs = _attn_case(16, 103)
    kq = np.zeros((16, D), dtype=np.int8)
    q = _rng(104).standard_normal((1, H, D)).astype(np.float32)
    ids = np.array([[3, 0, 1]], dtype=np.int32)
    out = o.sparse_attn(q, kq, ks, vq, vs, ids)
    cells = [12, 13, 14, 15, 0, 1, 2, 3, 4, 5, 6, 7]
    vals = np.stack([vq[c].astype(np.float64) * float(np.uint16(vs[c]).view(np.float16)) for c in cells])
    want = vals.mean(axis=0)
    for h in range(H):
        assert np.allclose(out[0, h], want, rtol=0, atol=1e-14 * np.abs(vals).max()), h


def pin_attn_two_cells_logistic(o) -> None:
    """Two cells whose logits differ by a known amount: the weights are the
    logistic function of that difference, which fixes the 1/sqrt(128)
    temperature and both scales. Head h has its own query scale."""
    kq = np.zeros((4, D), dtype=np.int8)
    vq = np.zeros((4, D), dtype=np.int8)
    kq[0, 5], kq[1, 5] = 3, -2                   # key elements on d = 5
    vq[0, :], vq[1, :] = 7, -5
    ks = _half_bits([0.5, 0.5, 0.5, 0.5])
    vs = _half_bits([0.25, 0.125, 1.0, 1.0])
    ncells = 2                                   # block 0 holds cells 0 and 1 only
    q = np.zeros((1, H, D), dtype=np.float32)
    for h in range(H):
        q[0, h, 5] = 1.5 * (h + 1)
    out = o.sparse_attn(q, kq[:ncells], ks[:ncells], vq[:ncells], vs[:ncells], np.array([[0]], dtype=np.int32))
    import math
    for h in range(H):
        a = 1.5 * (h + 1)
        l0, l1 = a * 3 * 0.5 / math.sqrt(128.0), a * (-2) * 0.5 / math.sqrt(128.0)
        w0 = 1.0 / (1.0 + math.exp(l1 - l0))
        want = w0 * 7 * 0.25 + (1.0 - w0) * (-5) * 0.125
        assert abs(out[0, h, 0] - want) <= 1e-15 * 2, (h, out[0, h, 0], want)
        assert np.all(out[0, h] == out[0, h, 0])


def pin_attn_python_loops(o) -> None:
    """A small ragged case against a pure-Python FP64 restatement that sums
    in the reverse order and does not subtract the maximum (duplicated and
    padded ids, a partial last block)."""
    import math
    ncells = 23                                   # blocks 0..5, block 5 holds cells 20..22
    kq, vq, ks, vs = _attn_case(ncells, 105)
    q = _rng(106).standard_normal((3, H, D)).astype(np.float32)
    ids = np.array([[5, 1, -1, 3], [0, 0, 2, -1], [-1, -1, -1, 4]], dtype=np.int32)
    out = o.sparse_attn(q, kq, ks, vq, vs, ids)
    half = lambda u: float(np.uint16(u).view(np.float16))
    for i in range(ids.shape[0]):
        cells = [4 * int(b) + t for b in ids[i] if b >= 0 for t in range(4) if 4 * int(b) + t < ncells]
        for h in range(H):
            qh = [float(x) for x in q[i, h]]
            lg = []
            for c in reversed(cells):
                kc = [int(x) * half(ks[c]) for x in kq[c]]
                lg.append((c, sum(qh[d] * kc[d] for d in reversed(range(D))) / math.sqrt(D)))
            e = [(c, math.exp(x)) for c, x in lg]
            tot = sum(x for _, x in e)
            want = [sum(x / tot * int(vq[c, d]) * half(vs[c]) for c, x in e) for d in range(D)]
            scale = max(abs(w) for w in want) + 1e-300
            assert np.allclose(out[i, h], want, rtol=0, atol=1e-12 * scale), (i, h)


def pin_attn_padding_and_order(o) -> None:
    """No attended cell gives zeros; the order of the listed ids and extra
    padding do not change the result beyond rounding."""
    kq, vq, ks, vs = _attn_case(40, 107)
    q = _rng(108).standard_normal((2, H, D)).astype(np.float32)
    empty = o.sparse_attn(q, kq, ks, vq, vs, np.array([[-1, -1], [10, 99]], dtype=np.int32))
    assert np.array_equal(empty, np.zeros_like(empty))
    a = o.sparse_attn(q, kq, ks, vq, vs, np.array([[1, 4, 7, -1], [9, 0, 2, 3]], dtype=np.int32))
    b = o.sparse_attn(q, kq, ks, vq, vs, np.array([[7, -1, 1, 4], [3, 2, 0, 9]], dtype=np.int32))
    assert np.allclose(a, b, rtol=0, atol=1e-13 * np.abs(a).max())


# ---- block summary keys -----------------------------------------------------
# The reading pinned (the pages time an "append" step but define no summary
# function, so the definition itself stays a reading): a block's key is the
# element-wise mean of its present cells (int8 x binary16 scale per cell);
# the int8 form has scale binary16(max|key| / 127) and codes rint(key / s).

def pin_float_to_half(o) -> None:
    """The oracle's binary32 -> binary16 rounding against numpy's, on
    normals, subnormals, exact ties and the largest finite values."""
    r = _rng(201)
    x = (r.standard_normal(30000) * 10.0 ** r.integers(-9, 5, 30000)).astype(np.float32)
    ties = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 2 ** -24 * 0.5, 2 ** -24 * 1.5, 2 ** -24 * 2.5,
                     65504.0, 65519.0, 2 ** -14, 2 ** -14 * (1 - 2 ** -11), 0.0, -0.0, -(1 + 2 ** -11)],
                    dtype=np.float32)
    for v in np.concatenate([x, ties, -ties]):
        assert o.float_to_half(v) == int(np.float16(v).view(np.uint16)), float(v)


def _summary_cells(rows, scales):
    return np.asarray(rows, dtype=np.int8), _half_bits(scales)


def pin_summary_exact_means(o) -> None:
    """Cells whose sums are exact in fp32 (small integers, power-of-two
    scales): the key is the exact mean over the present cells (4, 2 or 1 of
    them), and a block with no present cell is zero."""
    from fractions import Fraction
    r = _rng(202)
    rows = r.integers(-100, 101, (11, D))
    scales = 2.0 ** r.integers(-6, 2, 11)
    kq, ks = _summary_cells(rows, scales)
    key, _, _ = o.block_summary(kq, ks, 0, 4)           # blocks of 4, 4, 3 cells and none
    for b, n in ((0, 4), (1, 4)):
        for d in range(D):
            want = sum(Fraction(int(rows[4 * b + t, d])) * Fraction(float(scales[4 * b + t])) for t in range(n)) / n
            assert Fraction(float(key[b, d])) == want, (b, d)
    k2, _, _ = o.block_summary(kq[:10], ks[:10], 2, 3)  # block 2 holds cells 8, 9
    for d in range(D):
        want = (Fraction(int(rows[8, d])) * Fraction(float(scales[8])) +
                Fraction(int(rows[9, d])) * Fraction(float(scales[9]))) / 2
        assert Fraction(float(k2[0, d])) == want, d
    k1, _, _ = o.block_summary(kq[:9], ks[:9], 2, 3)    # block 2 holds cell 8 only
    assert np.array_equal(k1[0], rows[8].astype(np.float32) * np.float32(scales[8]))
    assert np.all(key[3] == 0.0)


def pin_summary_codes(o) -> None:
    """int8 form: the scale is numpy's binary16 of max|key| / 127, every code
    is within half a step of the key, the largest |key| gets |code| 127, and
    a zero block gets scale 0 and zero codes."""
    r = _rng(203)
    kq = r.integers(-127, 128, (64, D)).astype(np.int8)
    ks = _half_bits(np.exp(r.uniform(np.log(1e-3), np.log(1e-1), 64)))
    kq[40:44] = 0
    key, q8, sc = o.block_summary(kq, ks, 0, 16)
    for b in range(16):
        top = np.float32(np.abs(key[b]).max())
        assert sc[b] == int(np.float16(top / np.float32(127.0)).view(np.uint16)), b
        s = float(np.uint16(sc[b]).view(np.float16))
        if top == 0:
            assert s == 0 and np.all(q8[b] == 0)
            continue
        assert np.all(np.abs(q8[b].astype(np.float64) * s - key[b]) <= 0.5 * s * (1 + 2 ** -20)), b
        assert abs(int(q8[b][np.argmax(np.abs(key[b]))])) == 127
    assert np.all(q8[10] == 0) and sc[10] == 0          # cells 40..43 are zero


def pin_summary_padding(o) -> None:
    """A block's key depends only on its own present cells: the same block
    from a longer or a cut pool, and blocks past the cells are zero."""
    kq, _, ks, _ = _attn_case(23, 204)
    a = o.block_summary(kq, ks, 0, 8)
    b = o.block_summary(kq[:20], ks[:20], 0, 8)
    for x, y in zip(a, b):
        assert np.array_equal(x[:5], y[:5])               # blocks 0..4 whole in both
    assert not np.array_equal(a[0][5], b[0][5])           # block 5: cells 20..22 against none
    assert np.all(b[0][5:] == 0) and np.all(b[1][5:] == 0) and np.all(b[2][5:] == 0)
    c = o.block_summary(kq, ks, 3, 6)
    for x, y in zip(a, c):
        assert np.array_equal(x[3:6], y)                  # a sub-range gives the same rows


ALL_PINS = [
    pin_brute_force_topk,
    pin_float_to_half,
    pin_summary_exact_means,
    pin_summary_codes,
    pin_summary_padding,
    pin_attn_single_cell,
    pin_attn_uniform_weights,
    pin_attn_two_cells_logistic,
    pin_attn_python_loops,
    pin_attn_padding_and_order,
    pin_closed_form_onehot,
    pin_all_ties_lower_id,
    pin_integer_exact,
    pin_float_vs_numpy,
    pin_half_to_double,
    pin_q8_scores,
    pin_padding_and_empty,
    pin_capacity_independence,
    pin_selection_invariants,
    pin_golden_hand,
    pin_score_keys_order,
    pin_group_max_keys,
]
