"""Seeded synthetic inputs for QSA block selection.

This module only draws random numbers and lays them out; it computes no
block score and no selection. Both sides of every parity check (the CUDA
path and the CPU oracle) receive the buffers it returns. The draws come from
a small C library (``gen/qsa_gen.c``: PCG32 XSH-RR 64/32, Box-Muller normals,
Student-t, integer maps) so that multi-million-element workloads take well
under a second.

Workload shapes follow the QSA selection path of the pages
("#3108 optimize exact QSA block scoring and top-k selection on gfx12",
Microbenchmark & Parity section 1; "#337 gfx12 QSA select", What item 1 and
Results): 4 query heads of D=128 per KV head, one summary key per 4-cell
block, capacity ``max_blocks = max_context/4 + 2``.
"""

from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

D = 128          # head dimension
H = 4            # query heads sharing one KV head
CELLS_PER_BLOCK = 4

# One independent PCG32 stream per tensor of a workload.
STREAM_Q = 1
STREAM_KBLK = 2
STREAM_DIRECTION = 3
STREAM_NEEDLES = 4
STREAM_TIES = 5
STREAM_SCALES = 6
STREAM_V = 7         # attention: value cells
STREAM_V_SCALES = 8
STREAM_IDS = 9

SEED_BASE = 0x9E3779B9

_HERE = os.path.dirname(os.path.abspath(__file__))
_GEN_SRC = os.path.join(_HERE, "gen", "qsa_gen.c")
_GEN_LIB = os.path.join(_HERE, "gen", "_build", "libqsa_gen.so")


def build_gen(force: bool = False) -> str:
    """Compile the generator library with the host C compiler."""
    if force or not os.path.exists(_GEN_LIB) or os.path.getmtime(_GEN_LIB) < os.path.getmtime(_GEN_SRC):
        os.makedirs(os.path.dirname(_GEN_LIB), exist_ok=True)
        tmp = _GEN_LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _GEN_SRC, "-lm"])
        os.replace(tmp, _GEN_LIB)
    return _GEN_LIB


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        L = ctypes.CDLL(build_gen())
        u64, sz, vp = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p
        for name in ("qsa_gen_u32", "qsa_gen_uniform_f64", "qsa_gen_normal_f64",
                     "qsa_gen_normal_f32", "qsa_gen_student_t3_f32", "qsa_gen_int8_127"):
            getattr(L, name).argtypes = [u64, u64, sz, vp]
            getattr(L, name).restype = None
        L.qsa_gen_int_range_f32.argtypes = [u64, u64, sz, ctypes.c_int, ctypes.c_int, vp]
        L.qsa_gen_int_range_f32.restype = None
        _lib_handle = L
    return _lib_handle


def _fill(fn: str, seed: int, stream: int, n: int, dtype) -> np.ndarray:
    out = np.empty(n, dtype=dtype)
    getattr(_lib(), fn)(seed, stream, n, out.ctypes.data)
    return out


def u32(seed: int, stream: int, n: int) -> np.ndarray:
    return _fill("qsa_gen_u32", seed, stream, n, np.uint32)


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    return _fill("qsa_gen_uniform_f64", seed, stream, n, np.float64)


def normal64(seed: int, stream: int, n: int) -> np.ndarray:
    return _fill("qsa_gen_normal_f64", seed, stream, n, np.float64)


def normal32(seed: int, stream: int, n: int) -> np.ndarray:
    return _fill("qsa_gen_normal_f32", seed, stream, n, np.float32)


def student_t3_32(seed: int, stream: int, n: int) -> np.ndarray:
    return _fill("qsa_gen_student_t3_f32", seed, stream, n, np.float32)


def int8_127(seed: int, stream: int, n: int) -> np.ndarray:
    return _fill("qsa_gen_int8_127", seed, stream, n, np.int8)


def int_range32(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _lib().qsa_gen_int_range_f32(seed, stream, n, lo, hi, out.ctypes.data)
    return out


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of range(n) driven by the uniform stream."""
    u = uniform(seed, stream, n)
    j = (u * (np.arange(n) + 1)).astype(np.int64)
    p = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        jj = j[i]
        p[i], p[jj] = p[jj], p[i]
    return p


def capacity_blocks(max_context_cells: int) -> int:
    """Block capacity for a context capacity: ``max_context/4 + 2`` (the
    "#337" page, What item 1)."""
    return max_context_cells // CELLS_PER_BLOCK + 2


def seed_for(config_index: int) -> int:
    return SEED_BASE + config_index


@dataclass
class Workload:
    """One seeded selection problem.

    q:      float32 [nq, H, D], contiguous (2 KiB per query)
    kblk:   float32 [max_blocks, D] (None for the int8 form); rows at and
            beyond ``active`` are capacity and hold NaN, so a kernel that
            reads them shows it.
    kq8:    int8 [max_blocks, D] and kscale: uint16 [max_blocks] (IEEE
            binary16 bit patterns) for the int8-key form.
    """
    name: str
    nq: int
    active: int
    max_blocks: int
    k: int
    q: np.ndarray
    kblk: np.ndarray | None = None
    kq8: np.ndarray | None = None
    kscale: np.ndarray | None = None
    meta: dict = field(default_factory=dict)


def _capacity_fill(rows_active: np.ndarray, max_blocks: int) -> np.ndarray:
    out = np.full((max_blocks, D), np.nan, dtype=np.float32)
    out[:rows_active.shape[0]] = rows_active
    return out


def tiny(config_index: int = 0) -> Workload:
    """nq=8, 4,096 cells (1,024 blocks), capacity = active, k=64, N(0,1).

    Exact-tie blocks are planted on top of this by the test fixtures.
    """
    s = seed_for(config_index)
    nq, active, k = 8, 1024, 64
    q = normal32(s, STREAM_Q, nq * H * D).reshape(nq, H, D)
    kb = normal32(s, STREAM_KBLK, active * D).reshape(active, D)
    return Workload("tiny_4k_nq8_k64", nq, active, active, k, q, kblk=kb)


def mid(config_index: int = 1) -> Workload:
    """32,768 cells (8,192 blocks) under a 262,144-cell capacity, nq=256,
    k=256; keys are N(0,1) noise plus 0.5 times one shared random unit
    direction (skewed scores)."""
    s = seed_for(config_index)
    nq, active, k = 256, 8192, 256
    max_blocks = capacity_blocks(262144)
    q = normal32(s, STREAM_Q, nq * H * D).reshape(nq, H, D)
    noise = normal64(s, STREAM_KBLK, active * D).reshape(active, D)
    u = normal64(s, STREAM_DIRECTION, D)
    u = u / math.sqrt(float(np.sum(u * u)))
    kb = (noise + 0.5 * u[None, :]).astype(np.float32)
    return Workload("mid_32k_nq256_k256", nq, active, max_blocks, k, q,
                    kblk=_capacity_fill(kb, max_blocks), meta={"direction": u})


def long(config_index: int = 2) -> Workload:
    """131,072 cells (32,768 blocks) under a 262,144-cell capacity, nq=256,
    k=256, N(0,1). The 16 needle blocks per query are planted by the test
    fixtures; ``meta['needles']`` holds their seeded, disjoint choice."""
    s = seed_for(config_index)
    nq, active, k = 256, 32768, 256
    max_blocks = capacity_blocks(262144)
    q = normal32(s, STREAM_Q, nq * H * D).reshape(nq, H, D)
    kb = normal32(s, STREAM_KBLK, active * D).reshape(active, D)
    needles = permutation(s, STREAM_NEEDLES, active)[:nq * 16].reshape(nq, 16)
    return Workload("long_131k_nq256_k256", nq, active, max_blocks, k, q,
                    kblk=_capacity_fill(kb, max_blocks), meta={"needles": needles})


def full(k: int = 512, config_index: int = 3, nq: int = 256) -> Workload:
    """262,144 cells (65,536 blocks, capacity 65,538), nq=256, k=512 (the
    sweep adds 64/256/1024); q and keys Student-t(3) at unit variance."""
    s = seed_for(config_index)
    active = 65536
    max_blocks = capacity_blocks(262144)
    q = student_t3_32(s, STREAM_Q, 256 * H * D).reshape(256, H, D)[:nq].copy()
    kb = student_t3_32(s, STREAM_KBLK, active * D).reshape(active, D)
    return Workload(f"full_262k_nq{nq}_k{k}", nq, active, max_blocks, k, q,
                    kblk=_capacity_fill(kb, max_blocks))


def decode(nq: int, cells: int, config_index: int = 4, k: int = 128) -> Workload:
    """Decode-shaped int8 keys: nq in {1,4}, context cells in {2K, 16K, 64K,
    262K} under a 262,144-cell capacity, k=128. Keys uniform on [-127,127];
    one binary16 scale per block, log-uniform in [1e-3, 1e-1]; q is N(0,1).
    Capacity rows hold key bytes 0 and a NaN scale."""
    s = seed_for(config_index)
    active = cells // CELLS_PER_BLOCK
    max_blocks = capacity_blocks(262144)
    q = normal32(s, STREAM_Q, nq * H * D).reshape(nq, H, D)
    kq = np.zeros((max_blocks, D), dtype=np.int8)
    kq[:active] = int8_127(s, STREAM_KBLK, active * D).reshape(active, D)
    sc = np.full(max_blocks, 0x7E00, dtype=np.uint16)          # binary16 NaN
    u = uniform(s, STREAM_SCALES, active)
    lo, hi = math.log(1e-3), math.log(1e-1)
    sc[:active] = np.exp(lo + (hi - lo) * u).astype(np.float16).view(np.uint16)
    return Workload(f"decode_{cells // 1024}k_nq{nq}_k{k}", nq, active, max_blocks, k, q,
                    kq8=kq, kscale=sc)


def integer_valued(nq: int, active: int, max_blocks: int | None = None, lo: int = -8,
                   hi: int = 8, k: int = 0, config_index: int = 7) -> Workload:
    """q and keys integer-valued in [lo, hi]. With |lo|, |hi| <= 8 every
    partial sum of a score is an integer of magnitude below 2^24, so fp32
    scoring is exact in any summation order."""
    s = seed_for(config_index)
    max_blocks = active if max_blocks is None else max_blocks
    q = int_range32(s, STREAM_Q, nq * H * D, lo, hi).reshape(nq, H, D)
    kb = int_range32(s, STREAM_KBLK, active * D, lo, hi).reshape(active, D)
    return Workload(f"int_{active}_nq{nq}", nq, active, max_blocks, k, q,
                    kblk=_capacity_fill(kb, max_blocks))


def normal_case(nq: int, active: int, k: int, max_blocks: int | None = None,
                config_index: int = 8) -> Workload:
    """Generic N(0,1) case of any shape, for ragged-size coverage."""
    s = seed_for(config_index)
    max_blocks = active if max_blocks is None else max_blocks
    q = normal32(s, STREAM_Q, nq * H * D).reshape(nq, H, D)
    kb = normal32(s, STREAM_KBLK, active * D).reshape(active, D)
    return Workload(f"normal_{active}_nq{nq}_k{k}", nq, active, max_blocks, k, q,
                    kblk=_capacity_fill(kb, max_blocks))


def int8_case(nq: int, active: int, k: int, max_blocks: int | None = None,
              config_index: int = 9) -> Workload:
    """Generic int8-key case of any shape (same recipe as ``decode``)."""
    s = seed_for(config_index)
    max_blocks = active if max_blocks is None else max_blocks
    q = normal32(s, STREAM_Q, nq * H * D).reshape(nq, H, D)
    kq = np.zeros((max_blocks, D), dtype=np.int8)
    kq[:active] = int8_127(s, STREAM_KBLK, active * D).reshape(active, D)
    sc = np.full(max_blocks, 0x7E00, dtype=np.uint16)
    u = uniform(s, STREAM_SCALES, active)
    lo, hi = math.log(1e-3), math.log(1e-1)
    sc[:active] = np.exp(lo + (hi - lo) * u).astype(np.float16).view(np.uint16)
    return Workload(f"int8_{active}_nq{nq}_k{k}", nq, active, max_blocks, k, q,
                    kq8=kq, kscale=sc)


@dataclass
class AttnWorkload:
    """One seeded attention-over-selected-blocks problem.

    q:      float32 [nq, H, D]
    kc, vc: int8 [ncells, D] (key and value cells of one KV head)
    ks, vs: uint16 [ncells] (IEEE binary16 bit patterns, one scale per cell)
    ids:    int32 [nq, k] (listed blocks per query; -1 = padding)
    """
    name: str
    nq: int
    ncells: int
    k: int
    q: np.ndarray
    kc: np.ndarray
    ks: np.ndarray
    vc: np.ndarray
    vs: np.ndarray
    ids: np.ndarray


def _log_uniform_half(seed: int, stream: int, n: int, lo: float, hi: float) -> np.ndarray:
    u = uniform(seed, stream, n)
    a, b = math.log(lo), math.log(hi)
    return np.exp(a + (b - a) * u).astype(np.float16).view(np.uint16)


def attn_case(nq: int, ncells: int, k: int, pad: int = 0, config_index: int = 10) -> AttnWorkload:
    """KV cells for attention over the selected blocks, with the decode
    recipe's distributions: K and V int8 uniform on [-127, 127], one binary16
    scale per cell each, log-uniform in [1e-3, 1e-1]; q is N(0,1). Each query
    lists k - pad distinct blocks (drawn from the seeded stream, ascending, as
    the top-k returns them) followed by pad slots of -1."""
    s = seed_for(config_index)
    q = normal32(s, STREAM_Q, nq * H * D).reshape(nq, H, D)
    kc = int8_127(s, STREAM_KBLK, ncells * D).reshape(ncells, D)
    vc = int8_127(s, STREAM_V, ncells * D).reshape(ncells, D)
    ks = _log_uniform_half(s, STREAM_SCALES, ncells, 1e-3, 1e-1)
    vs = _log_uniform_half(s, STREAM_V_SCALES, ncells, 1e-3, 1e-1)
    nblocks = (ncells + CELLS_PER_BLOCK - 1) // CELLS_PER_BLOCK
    take = k - pad
    assert 0 <= take <= nblocks
    ids = np.full((nq, k), -1, dtype=np.int32)
    draws = u32(s, STREAM_IDS, nq * 4 * max(take, 1)).reshape(nq, -1) % np.uint32(max(nblocks, 1))
    for i in range(nq):
        _, first = np.unique(draws[i], return_index=True)
        picked = draws[i][np.sort(first)][:take]
        if picked.shape[0] < take:                 # few blocks: take them all in a seeded order
            picked = permutation(s + i, STREAM_IDS, nblocks)[:take]
        ids[i, :take] = np.sort(picked.astype(np.int32))
    return AttnWorkload(f"attn_{ncells}_nq{nq}_k{k}", nq, ncells, k, q, kc, ks, vc, vs, ids)


def pcg32_reference(seed: int, stream: int, n: int) -> list[int]:
    """Scalar PCG32 in pure Python, one output at a time, for checking the
    C generator."""
    m64 = (1 << 64) - 1
    mult = 6364136223846793005
    inc = ((stream << 1) | 1) & m64
    state = (inc) & m64                      # step from 0
    state = (state + seed) & m64
    state = (state * mult + inc) & m64
    out = []
    for _ in range(n):
        old = state
        state = (old * mult + inc) & m64
        xs = (((old >> 18) ^ old) >> 27) & 0xFFFFFFFF
        rot = old >> 59
        out.append(((xs >> rot) | (xs << ((-rot) & 31))) & 0xFFFFFFFF)
    return out
