"""CPU oracle for exact QSA block selection -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path never does: it runs
the CUDA library or fails.

The arithmetic lives in ``qsa_oracle.c`` (FP64 scores, full-sort top-k, FP64
attention over the selected blocks, fp32 block summary keys; see its header
comment for the definitions and the passages they follow). The block summary
keys are "parity unpinned" as to their definition (the pages define no
summary function; the mean of the cells is a reading). This module compiles
the C source with the host C compiler and marshals numpy arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

H, D = 4, 128

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "qsa_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libqsa_oracle.so")


def build(force: bool = False, source: str = SOURCE, out: str = _LIB) -> str:
    """Compile the oracle (``gcc -O2``, no hand SIMD) into a shared library."""
    stale = not os.path.exists(out) or os.path.getmtime(out) < max(
        os.path.getmtime(source), os.path.getmtime(os.path.join(_HERE, "qsa_oracle.h")))
    if force or stale:
        os.makedirs(os.path.dirname(out), exist_ok=True)
        tmp = out + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared",
                               "-pthread", "-I", _HERE, "-o", tmp, source, "-lm"])
        os.replace(tmp, out)
    return out


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, lib_path: str | None = None):
        self.lib = ctypes.CDLL(lib_path or build())
        L, vp, lg, i = self.lib, ctypes.c_void_p, ctypes.c_long, ctypes.c_int
        L.qsa_oracle_default_threads.restype = i
        L.qsa_oracle_half_to_double.argtypes = [ctypes.c_uint16]
        L.qsa_oracle_half_to_double.restype = ctypes.c_double
        L.qsa_oracle_scores.argtypes = [vp, vp, lg, lg, vp, i]
        L.qsa_oracle_scores_q8.argtypes = [vp, vp, vp, lg, lg, vp, i]
        L.qsa_oracle_topk_f64.argtypes = [vp, lg, lg, lg, vp, i]
        L.qsa_oracle_topk_f32.argtypes = [vp, lg, lg, lg, vp, i]
        L.qsa_oracle_sparse_attn.argtypes = [vp, vp, vp, vp, vp, lg, vp, lg, lg, vp, i]
        L.qsa_oracle_block_summary.argtypes = [vp, vp, lg, lg, lg, vp, vp, vp]
        L.qsa_oracle_block_summary.restype = None
        L.qsa_oracle_float_to_half.argtypes = [ctypes.c_float]
        L.qsa_oracle_float_to_half.restype = ctypes.c_uint16
        for f in ("qsa_oracle_scores", "qsa_oracle_scores_q8", "qsa_oracle_topk_f64",
                  "qsa_oracle_topk_f32", "qsa_oracle_sparse_attn"):
            getattr(L, f).restype = None

    def default_threads(self) -> int:
        return self.lib.qsa_oracle_default_threads()

    def half_to_double(self, h: int) -> float:
        return self.lib.qsa_oracle_half_to_double(int(h))

    @staticmethod
    def _c(a: np.ndarray, dtype) -> np.ndarray:
        return np.ascontiguousarray(a, dtype=dtype)

    def scores(self, q: np.ndarray, kblk: np.ndarray, active: int, nthreads: int = 0) -> np.ndarray:
        """FP64 block scores ``[nq, active]`` for fp32 keys."""
        q = self._c(q, np.float32)
        kblk = self._c(kblk, np.float32)
        nq = q.shape[0]
        assert q.shape[1:] == (H, D) and kblk.shape[1] == D and kblk.shape[0] >= active
        S = np.empty((nq, active), dtype=np.float64)
        self.lib.qsa_oracle_scores(q.ctypes.data, kblk.ctypes.data, nq, active, S.ctypes.data, nthreads)
        return S

    def scores_q8(self, q: np.ndarray, kq8: np.ndarray, kscale: np.ndarray, active: int,
                  nthreads: int = 0) -> np.ndarray:
        """FP64 block scores ``[nq, active]`` for int8 keys with binary16 scales."""
        q = self._c(q, np.float32)
        kq8 = self._c(kq8, np.int8)
        kscale = self._c(kscale, np.uint16)
        nq = q.shape[0]
        assert q.shape[1:] == (H, D) and kq8.shape[1] == D and kq8.shape[0] >= active
        assert kscale.shape[0] >= active
        S = np.empty((nq, active), dtype=np.float64)
        self.lib.qsa_oracle_scores_q8(q.ctypes.data, kq8.ctypes.data, kscale.ctypes.data, nq, active,
                                      S.ctypes.data, nthreads)
        return S

    def topk_f64(self, S: np.ndarray, k: int, nthreads: int = 0) -> np.ndarray:
        """Exact top-k ids ``[nq, k]`` (ascending, -1 padded) of FP64 scores."""
        S = self._c(S, np.float64)
        nq, active = S.shape
        ids = np.empty((nq, k), dtype=np.int32)
        self.lib.qsa_oracle_topk_f64(S.ctypes.data, nq, active, k, ids.ctypes.data, nthreads)
        return ids

    def topk_f32(self, scores: np.ndarray, k: int, nthreads: int = 0) -> np.ndarray:
        """Exact top-k ids of given fp32 scores (the same order and tie rule)."""
        scores = self._c(scores, np.float32)
        nq, active = scores.shape
        ids = np.empty((nq, k), dtype=np.int32)
        self.lib.qsa_oracle_topk_f32(scores.ctypes.data, nq, active, k, ids.ctypes.data, nthreads)
        return ids

    @staticmethod
    def score_keys(scores: np.ndarray) -> np.ndarray:
        """The order-preserving uint32 key of each fp32 score, as the
        boundary's header defines it: -0 counts as +0 and NaN as -inf, then a
        negative value's bits are inverted and a positive value gets the sign
        bit set."""
        x = np.ascontiguousarray(scores, dtype=np.float32)
        x = np.where(np.isnan(x), np.float32(-np.inf), x) + np.float32(0.0)
        bits = x.view(np.uint32)
        return np.where(bits >> np.uint32(31) != 0, ~bits, bits | np.uint32(0x80000000)).astype(np.uint32)

    @classmethod
    def group_max_keys(cls, scores: np.ndarray, group: int = 32) -> np.ndarray:
        """Per row, the key of the largest score of each run of ``group``
        consecutive blocks (the last run may be shorter): ``[nq, ceil(active /
        group)]`` uint32."""
        keys = cls.score_keys(scores)
        starts = np.arange(0, keys.shape[1], group)
        return np.maximum.reduceat(keys, starts, axis=1).astype(np.uint32)

    def sparse_attn(self, q: np.ndarray, kq: np.ndarray, ks: np.ndarray, vq: np.ndarray, vs: np.ndarray,
                    ids: np.ndarray, nthreads: int = 0) -> np.ndarray:
        """FP64 attention of each query's 4 heads over the cells of its
        selected blocks ``[nq, 4, 128]`` (int8 K/V cells ``[ncells, 128]``,
        binary16 scales ``[ncells]`` as uint16, ids ``[nq, k]``)."""
        q = self._c(q, np.float32)
        kq, vq = self._c(kq, np.int8), self._c(vq, np.int8)
        ks, vs = self._c(ks, np.uint16), self._c(vs, np.uint16)
        ids = self._c(ids, np.int32)
        nq, k = ids.shape
        ncells = kq.shape[0]
        assert q.shape == (nq, H, D) and kq.shape == (ncells, D) and vq.shape == (ncells, D)
        assert ks.shape == (ncells,) and vs.shape == (ncells,)
        out = np.empty((nq, H, D), dtype=np.float64)
        self.lib.qsa_oracle_sparse_attn(q.ctypes.data, kq.ctypes.data, ks.ctypes.data, vq.ctypes.data,
                                        vs.ctypes.data, ncells, ids.ctypes.data, nq, k, out.ctypes.data,
                                        nthreads)
        return out

    def float_to_half(self, x: float) -> int:
        return int(self.lib.qsa_oracle_float_to_half(float(x)))

    def block_summary(self, kq: np.ndarray, ks: np.ndarray, b0: int, b1: int):
        """Summary keys of blocks b0..b1-1 from int8 cells ``[ncells, 128]``
        with binary16 scales ``[ncells]``: ``(key fp32 [n, 128], kq8 int8
        [n, 128], kscale uint16 [n])``, n = b1 - b0."""
        kq, ks = self._c(kq, np.int8), self._c(ks, np.uint16)
        ncells = kq.shape[0]
        assert kq.shape == (ncells, D) and ks.shape == (ncells,) and 0 <= b0 <= b1
        n = b1 - b0
        key = np.empty((n, D), dtype=np.float32)
        kq8 = np.empty((n, D), dtype=np.int8)
        ksc = np.empty(n, dtype=np.uint16)
        self.lib.qsa_oracle_block_summary(kq.ctypes.data, ks.ctypes.data, ncells, b0, b1, key.ctypes.data,
                                          kq8.ctypes.data, ksc.ctypes.data)
        return key, kq8, ksc

    def select(self, q, kblk, active: int, k: int, nthreads: int = 0):
        """Scores then ids: ``(S[nq, active] fp64, ids[nq, k])``."""
        S = self.scores(q, kblk, active, nthreads)
        return S, self.topk_f64(S, k, nthreads)


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from this directory's source."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
