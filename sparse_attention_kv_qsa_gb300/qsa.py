"""Python binding of the C ABI in include/qsa.h (argument marshalling only).

Every step of the selection runs in ``libqsa.so``'s CUDA kernels; this module
checks tensor shapes, dtypes and devices, allocates outputs with torch, and
passes raw device pointers and the current CUDA stream. There is no fallback:
if the library is missing, importing the functions raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

D = 128
HEADS = 4
GROUP_BLOCKS = 32   # blocks per group of the group-maximum side output
TOPK_MAX_ACTIVE = 393216
SELECT_STATIC_GROUPS_MAX = 262144   # scratch bound of qsa_block_select_static

QSA_OK, QSA_ERR_INVALID, QSA_ERR_UNSUPPORTED, QSA_ERR_CUDA = 0, 1, 2, 3

EXPORTED = ("qsa_block_scores", "qsa_block_scores_q8", "qsa_block_scores_ffma", "qsa_block_topk",
            "qsa_block_scores_gmax", "qsa_block_scores_q8_gmax", "qsa_block_group_max", "qsa_block_topk_gmax",
            "qsa_block_select_static", "qsa_block_select_small", "qsa_sparse_attn", "qsa_block_summary",
            "qsa_get_device_error", "qsa_debug_inject", "qsa_status_string", "qsa_block_select",
            "qsa_block_select_scratch_bytes")


class QSAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded ``libqsa.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(the QSA kernels have no fallback)")
        L = ctypes.CDLL(path)
        vp, i = ctypes.c_void_p, ctypes.c_int
        L.qsa_block_scores.argtypes = [vp, vp, i, i, i, vp, vp]
        L.qsa_block_scores_q8.argtypes = [vp, vp, vp, i, i, i, vp, vp]
        L.qsa_block_scores_ffma.argtypes = [vp, vp, vp, vp, i, i, i, vp, vp]
        L.qsa_block_topk.argtypes = [vp, i, i, i, vp, vp]
        L.qsa_block_scores_gmax.argtypes = [vp, vp, i, i, i, vp, vp, vp]
        L.qsa_block_scores_q8_gmax.argtypes = [vp, vp, vp, i, i, i, vp, vp, vp]
        L.qsa_block_topk_gmax.argtypes = [vp, vp, i, i, i, vp, vp]
        L.qsa_block_group_max.argtypes = [vp, i, i, vp, vp]
        L.qsa_block_select_static.argtypes = [vp, vp, i, i, i, i, vp, vp, vp]
        L.qsa_block_select_small.argtypes = [vp, vp, vp, vp, i, i, i, i, vp, vp, vp]
        L.qsa_sparse_attn.argtypes = [vp, vp, vp, vp, vp, i, vp, i, i, vp, vp]
        L.qsa_block_summary.argtypes = [vp, vp, i, i, i, vp, vp, vp, vp]
        L.qsa_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
        L.qsa_block_select.argtypes = [vp, vp, i, i, i, i, vp, vp, vp, ctypes.c_size_t, vp]
        L.qsa_block_select.restype = i
        L.qsa_block_select_scratch_bytes.argtypes = [i]
        L.qsa_block_select_scratch_bytes.restype = ctypes.c_size_t
        L.qsa_debug_inject.argtypes = [ctypes.c_uint32, ctypes.c_uint64]
        L.qsa_debug_inject.restype = i
        L.qsa_status_string.argtypes = [i]
        L.qsa_status_string.restype = ctypes.c_char_p
        for f in ("qsa_block_scores", "qsa_block_scores_q8", "qsa_block_scores_ffma", "qsa_block_topk",
                  "qsa_block_scores_gmax", "qsa_block_scores_q8_gmax", "qsa_block_topk_gmax",
                  "qsa_block_group_max", "qsa_block_select_static", "qsa_block_select_small",
                  "qsa_sparse_attn", "qsa_block_summary", "qsa_get_device_error"):
            getattr(L, f).restype = i
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().qsa_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != QSA_OK:
        raise QSAError(status, what)


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None or t.numel() == 0 else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


def _scores_out(q: torch.Tensor, active_blocks: int, out: torch.Tensor | None) -> torch.Tensor:
    nq = q.shape[0]
    if out is None:
        return torch.empty((nq, active_blocks), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, 2)
    if tuple(out.shape) != (nq, active_blocks):
        raise ValueError(f"out must have shape {(nq, active_blocks)}")
    return out


def _check_q(q: torch.Tensor) -> None:
    _need(q, "q", torch.float32, 3)
    if tuple(q.shape[1:]) != (HEADS, D):
        raise ValueError(f"q must be [nq, {HEADS}, {D}]")


def block_scores(q: torch.Tensor, kblk: torch.Tensor, active_blocks: int,
                 out: torch.Tensor | None = None) -> torch.Tensor:
    """``qsa_block_scores``: fp32 scores ``[nq, active_blocks]`` for fp32 keys
    ``kblk[max_blocks, 128]`` (only the first ``active_blocks`` rows are read)."""
    _check_q(q)
    _need(kblk, "kblk", torch.float32, 2)
    if kblk.shape[1] != D:
        raise ValueError("kblk must be [max_blocks, 128]")
    out = _scores_out(q, active_blocks, out)
    _check(lib().qsa_block_scores(_ptr(q), _ptr(kblk), q.shape[0], kblk.shape[0], active_blocks,
                                  _ptr(out), _stream(q)), "qsa_block_scores")
    return out


def block_scores_q8(q: torch.Tensor, kblk_q8: torch.Tensor, kscale_f16: torch.Tensor, active_blocks: int,
                    out: torch.Tensor | None = None) -> torch.Tensor:
    """``qsa_block_scores_q8``: int8 keys ``[max_blocks, 128]`` with one
    binary16 scale per block (float16 or int16/uint16-viewed tensor)."""
    _check_q(q)
    _need(kblk_q8, "kblk_q8", torch.int8, 2)
    if kscale_f16.dtype not in (torch.float16, torch.int16, torch.uint16):
        raise ValueError("kscale_f16 must hold binary16 values")
    if not kscale_f16.is_cuda or kscale_f16.dim() != 1 or not kscale_f16.is_contiguous():
        raise ValueError("kscale_f16 must be a contiguous 1-d CUDA tensor")
    if kblk_q8.shape[1] != D or kscale_f16.shape[0] < kblk_q8.shape[0]:
        raise ValueError("kblk_q8 must be [max_blocks, 128] with max_blocks scales")
    out = _scores_out(q, active_blocks, out)
    _check(lib().qsa_block_scores_q8(_ptr(q), _ptr(kblk_q8), _ptr(kscale_f16), q.shape[0], kblk_q8.shape[0],
                                     active_blocks, _ptr(out), _stream(q)), "qsa_block_scores_q8")
    return out


def groups(active_blocks: int) -> int:
    """Number of 32-block groups of a row (the group-maximum row length)."""
    return (active_blocks + GROUP_BLOCKS - 1) // GROUP_BLOCKS


def _gmax_out(q: torch.Tensor, active_blocks: int, out: torch.Tensor | None) -> torch.Tensor:
    shape = (q.shape[0], groups(active_blocks))
    if out is None:
        return torch.empty(shape, dtype=torch.int32, device=q.device)
    _need(out, "gmax_out", torch.int32, 2)
    if tuple(out.shape) != shape:
        raise ValueError(f"gmax_out must have shape {shape}")
    return out


def block_scores_gmax(q: torch.Tensor, kblk: torch.Tensor, active_blocks: int,
                      out: torch.Tensor | None = None, gmax_out: torch.Tensor | None = None):
    """``qsa_block_scores_gmax``: ``(scores, gmax)``; ``gmax`` is an int32
    tensor ``[nq, ceil(active_blocks / 32)]`` holding the uint32 radix keys
    of each 32-block group's largest score (view it as uint32)."""
    _check_q(q)
    _need(kblk, "kblk", torch.float32, 2)
    if kblk.shape[1] != D:
        raise ValueError("kblk must be [max_blocks, 128]")
    out = _scores_out(q, active_blocks, out)
    gmax_out = _gmax_out(q, active_blocks, gmax_out)
    _check(lib().qsa_block_scores_gmax(_ptr(q), _ptr(kblk), q.shape[0], kblk.shape[0], active_blocks,
                                       _ptr(out), _ptr(gmax_out), _stream(q)), "qsa_block_scores_gmax")
    return out, gmax_out


def block_scores_q8_gmax(q: torch.Tensor, kblk_q8: torch.Tensor, kscale_f16: torch.Tensor, active_blocks: int,
                         out: torch.Tensor | None = None, gmax_out: torch.Tensor | None = None):
    """``qsa_block_scores_q8_gmax``: the int8-key form of block_scores_gmax."""
    _check_q(q)
    _need(kblk_q8, "kblk_q8", torch.int8, 2)
    if kscale_f16.dtype not in (torch.float16, torch.int16, torch.uint16):
        raise ValueError("kscale_f16 must hold binary16 values")
    if not kscale_f16.is_cuda or kscale_f16.dim() != 1 or not kscale_f16.is_contiguous():
        raise ValueError("kscale_f16 must be a contiguous 1-d CUDA tensor")
    if kblk_q8.shape[1] != D or kscale_f16.shape[0] < kblk_q8.shape[0]:
        raise ValueError("kblk_q8 must be [max_blocks, 128] with max_blocks scales")
    out = _scores_out(q, active_blocks, out)
    gmax_out = _gmax_out(q, active_blocks, gmax_out)
    _check(lib().qsa_block_scores_q8_gmax(_ptr(q), _ptr(kblk_q8), _ptr(kscale_f16), q.shape[0], kblk_q8.shape[0],
                                          active_blocks, _ptr(out), _ptr(gmax_out), _stream(q)),
           "qsa_block_scores_q8_gmax")
    return out, gmax_out


def block_scores_ffma(q: torch.Tensor, active_blocks: int, kblk: torch.Tensor | None = None,
                      kblk_q8: torch.Tensor | None = None, kscale_f16: torch.Tensor | None = None,
                      out: torch.Tensor | None = None) -> torch.Tensor:
    """``qsa_block_scores_ffma``: the CUDA-core scorer (fp32 or int8 keys)."""
    _check_q(q)
    if kblk is not None:
        _need(kblk, "kblk", torch.float32, 2)
        max_blocks = kblk.shape[0]
    else:
        _need(kblk_q8, "kblk_q8", torch.int8, 2)
        max_blocks = kblk_q8.shape[0]
    out = _scores_out(q, active_blocks, out)
    _check(lib().qsa_block_scores_ffma(_ptr(q), _ptr(kblk), _ptr(kblk_q8), _ptr(kscale_f16), q.shape[0],
                                       max_blocks, active_blocks, _ptr(out), _stream(q)),
           "qsa_block_scores_ffma")
    return out


def block_topk(scores: torch.Tensor, k: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """``qsa_block_topk``: int32 ids ``[nq, k]``, ascending per row, ties to
    the lower block id, ``-1`` padding when ``k > active_blocks``."""
    _need(scores, "scores", torch.float32, 2)
    nq, active = scores.shape
    if out is None:
        out = torch.empty((nq, k), dtype=torch.int32, device=scores.device)
    else:
        _need(out, "out", torch.int32, 2)
        if tuple(out.shape) != (nq, k):
            raise ValueError(f"out must have shape {(nq, k)}")
    _check(lib().qsa_block_topk(_ptr(scores), nq, active, k, _ptr(out), _stream(scores)), "qsa_block_topk")
    return out


def block_group_max(scores: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """``qsa_block_group_max``: the group maxima (int32 tensor of uint32
    keys, as block_scores_gmax writes them) of given scores."""
    _need(scores, "scores", torch.float32, 2)
    nq, active = scores.shape
    shape = (nq, groups(active))
    if out is None:
        out = torch.empty(shape, dtype=torch.int32, device=scores.device)
    else:
        _need(out, "out", torch.int32, 2)
        if tuple(out.shape) != shape:
            raise ValueError(f"out must have shape {shape}")
    _check(lib().qsa_block_group_max(_ptr(scores), nq, active, _ptr(out), _stream(scores)), "qsa_block_group_max")
    return out


def block_topk_gmax(scores: torch.Tensor, gmax: torch.Tensor, k: int,
                    out: torch.Tensor | None = None) -> torch.Tensor:
    """``qsa_block_topk_gmax``: block_topk's result, using the group maxima
    that block_scores_gmax wrote for these scores."""
    _need(scores, "scores", torch.float32, 2)
    nq, active = scores.shape
    _need(gmax, "gmax", torch.int32, 2)
    if tuple(gmax.shape) != (nq, groups(active)):
        raise ValueError(f"gmax must have shape {(nq, groups(active))}")
    if out is None:
        out = torch.empty((nq, k), dtype=torch.int32, device=scores.device)
    else:
        _need(out, "out", torch.int32, 2)
        if tuple(out.shape) != (nq, k):
            raise ValueError(f"out must have shape {(nq, k)}")
    _check(lib().qsa_block_topk_gmax(_ptr(scores), _ptr(gmax), nq, active, k, _ptr(out), _stream(scores)),
           "qsa_block_topk_gmax")
    return out


def block_select_gmax(q: torch.Tensor, kblk: torch.Tensor, active_blocks: int, k: int,
                      scores_out: torch.Tensor | None = None, ids_out: torch.Tensor | None = None,
                      gmax_out: torch.Tensor | None = None):
    """Scores (with group maxima) then top-k, both on the current stream:
    ``(scores, ids)``; the ids equal ``block_topk(block_scores(...), k)``."""
    s, gm = block_scores_gmax(q, kblk, active_blocks, scores_out, gmax_out)
    return s, block_topk_gmax(s, gm, k, ids_out)


def select_scratch_bytes(nq: int) -> int:
    """``qsa_block_select_scratch_bytes``: scratch bytes qsa_block_select needs."""
    return int(lib().qsa_block_select_scratch_bytes(int(nq)))


def block_select(q: torch.Tensor, kblk: torch.Tensor, active_blocks: int, k: int,
                 ids_out: torch.Tensor | None = None, scores_buf: torch.Tensor | None = None,
                 scratch: torch.Tensor | None = None) -> torch.Tensor:
    """``qsa_block_select``: the ids of ``block_topk(block_scores(...), k)``
    without writing the scores (fp32 keys). ``scores_buf`` ``[nq, active]``
    fp32 is the fallback's buffer (contents unspecified afterwards) and
    ``scratch`` a uint8 tensor of at least ``select_scratch_bytes(nq)``
    bytes; both are allocated when not given."""
    _check_q(q)
    _need(kblk, "kblk", torch.float32, 2)
    if kblk.shape[1] != D:
        raise ValueError("kblk must be [max_blocks, 128]")
    nq = q.shape[0]
    scores_buf = _scores_out(q, active_blocks, scores_buf)
    if ids_out is None:
        ids_out = torch.empty((nq, k), dtype=torch.int32, device=q.device)
    else:
        _need(ids_out, "ids_out", torch.int32, 2)
        if tuple(ids_out.shape) != (nq, k):
            raise ValueError(f"ids_out must have shape {(nq, k)}")
    need = select_scratch_bytes(nq)
    if scratch is None:
        scratch = torch.empty((max(need, 16),), dtype=torch.uint8, device=q.device)
    elif scratch.dtype != torch.uint8 or not scratch.is_cuda or not scratch.is_contiguous():
        raise ValueError("scratch must be a contiguous uint8 CUDA tensor")
    _check(lib().qsa_block_select(_ptr(q), _ptr(kblk), nq, kblk.shape[0], active_blocks, k, _ptr(scores_buf),
                                  _ptr(ids_out), _ptr(scratch), scratch.numel(), _stream(q)), "qsa_block_select")
    return ids_out


def block_select_static(q: torch.Tensor, kblk: torch.Tensor, active_blocks: int, k: int,
                        scores_out: torch.Tensor | None = None, ids_out: torch.Tensor | None = None):
    """``qsa_block_select_static``: ``(scores, ids)`` as block_select_gmax, with
    the group maxima in the library's fixed device scratch (the call
    allocates nothing; calls on one device must be ordered)."""
    _check_q(q)
    _need(kblk, "kblk", torch.float32, 2)
    if kblk.shape[1] != D:
        raise ValueError("kblk must be [max_blocks, 128]")
    nq = q.shape[0]
    scores_out = _scores_out(q, active_blocks, scores_out)
    if ids_out is None:
        ids_out = torch.empty((nq, k), dtype=torch.int32, device=q.device)
    else:
        _need(ids_out, "ids_out", torch.int32, 2)
        if tuple(ids_out.shape) != (nq, k):
            raise ValueError(f"ids_out must have shape {(nq, k)}")
    _check(lib().qsa_block_select_static(_ptr(q), _ptr(kblk), nq, kblk.shape[0], active_blocks, k, _ptr(scores_out),
                                         _ptr(ids_out), _stream(q)), "qsa_block_select_static")
    return scores_out, ids_out


def block_select_small(q: torch.Tensor, active_blocks: int, k: int, kblk: torch.Tensor | None = None,
                       kblk_q8: torch.Tensor | None = None, kscale_f16: torch.Tensor | None = None,
                       scores_out: torch.Tensor | None = None, ids_out: torch.Tensor | None = None):
    """``qsa_block_select_small``: ``(scores, ids)`` for 1..4 queries in one
    cooperative launch (fp32 keys, or int8 keys with binary16 scales)."""
    _check_q(q)
    if kblk is not None:
        _need(kblk, "kblk", torch.float32, 2)
        max_blocks = kblk.shape[0]
    else:
        _need(kblk_q8, "kblk_q8", torch.int8, 2)
        if kscale_f16 is None or not kscale_f16.is_cuda or kscale_f16.dim() != 1:
            raise ValueError("kscale_f16 must be a 1-d CUDA tensor of binary16 values")
        max_blocks = kblk_q8.shape[0]
    nq = q.shape[0]
    scores_out = _scores_out(q, active_blocks, scores_out)
    if ids_out is None:
        ids_out = torch.empty((nq, k), dtype=torch.int32, device=q.device)
    else:
        _need(ids_out, "ids_out", torch.int32, 2)
        if tuple(ids_out.shape) != (nq, k):
            raise ValueError(f"ids_out must have shape {(nq, k)}")
    _check(lib().qsa_block_select_small(_ptr(q), _ptr(kblk), _ptr(kblk_q8), _ptr(kscale_f16), nq, max_blocks,
                                        active_blocks, k, _ptr(scores_out), _ptr(ids_out), _stream(q)),
           "qsa_block_select_small")
    return scores_out, ids_out


def sparse_attn(q: torch.Tensor, k_cells: torch.Tensor, k_scale_f16: torch.Tensor, v_cells: torch.Tensor,
                v_scale_f16: torch.Tensor, ids: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """``qsa_sparse_attn``: each query's 4 heads attend the int8 KV cells of
    the blocks listed in its row of ``ids`` -> ``out [nq, 4, 128]`` fp32.
    ``k_cells``/``v_cells`` int8 ``[ncells, 128]``; the scales are binary16
    bit patterns ``[ncells]`` (int16 or uint16 storage)."""
    _check_q(q)
    _need(k_cells, "k_cells", torch.int8, 2)
    _need(v_cells, "v_cells", torch.int8, 2)
    _need(ids, "ids", torch.int32, 2)
    ncells = k_cells.shape[0]
    if tuple(v_cells.shape) != tuple(k_cells.shape) or k_cells.shape[1] != 128:
        raise ValueError("k_cells and v_cells must both be [ncells, 128]")
    for name, t in (("k_scale_f16", k_scale_f16), ("v_scale_f16", v_scale_f16)):
        if not t.is_cuda or t.dim() != 1 or t.shape[0] != ncells or t.element_size() != 2 or not t.is_contiguous():
            raise ValueError(f"{name} must be a 1-d CUDA tensor of {ncells} binary16 values")
    nq, k = ids.shape
    if nq != q.shape[0]:
        raise ValueError("ids must have one row per query")
    if out is None:
        out = torch.empty((nq, 4, 128), dtype=torch.float32, device=q.device)
    else:
        _need(out, "out", torch.float32, 3)
        if tuple(out.shape) != (nq, 4, 128):
            raise ValueError(f"out must have shape {(nq, 4, 128)}")
    _check(lib().qsa_sparse_attn(_ptr(q), _ptr(k_cells), _ptr(k_scale_f16), _ptr(v_cells), _ptr(v_scale_f16),
                                 ncells, _ptr(ids), nq, k, _ptr(out), _stream(q)), "qsa_sparse_attn")
    return out


def block_summary(k_cells: torch.Tensor, k_scale_f16: torch.Tensor, block_begin: int, block_end: int,
                  kblk: torch.Tensor | None = None, kblk_q8: torch.Tensor | None = None,
                  kblk_scale_f16: torch.Tensor | None = None) -> None:
    """``qsa_block_summary``: rewrites rows ``block_begin .. block_end-1`` of the
    summary keys from the int8 cells (``k_cells [ncells, 128]``, binary16
    scales ``[ncells]``): fp32 ``kblk`` and/or int8 ``kblk_q8`` with binary16
    ``kblk_scale_f16`` (capacity buffers with at least ``block_end`` rows)."""
    _need(k_cells, "k_cells", torch.int8, 2)
    ncells = k_cells.shape[0]
    if k_cells.shape[1] != 128:
        raise ValueError("k_cells must be [ncells, 128]")
    if (not k_scale_f16.is_cuda or k_scale_f16.dim() != 1 or k_scale_f16.shape[0] != ncells
            or k_scale_f16.element_size() != 2 or not k_scale_f16.is_contiguous()):
        raise ValueError(f"k_scale_f16 must be a 1-d CUDA tensor of {ncells} binary16 values")
    if kblk is not None:
        _need(kblk, "kblk", torch.float32, 2)
        if kblk.shape[1] != 128 or kblk.shape[0] < block_end:
            raise ValueError(f"kblk must be [>= {block_end}, 128]")
    if kblk_q8 is not None:
        _need(kblk_q8, "kblk_q8", torch.int8, 2)
        if kblk_q8.shape[1] != 128 or kblk_q8.shape[0] < block_end:
            raise ValueError(f"kblk_q8 must be [>= {block_end}, 128]")
        if (kblk_scale_f16 is None or not kblk_scale_f16.is_cuda or kblk_scale_f16.dim() != 1
                or kblk_scale_f16.shape[0] < block_end or kblk_scale_f16.element_size() != 2):
            raise ValueError(f"kblk_scale_f16 must be a 1-d CUDA tensor of >= {block_end} binary16 values")
    _check(lib().qsa_block_summary(_ptr(k_cells), _ptr(k_scale_f16), ncells, block_begin, block_end, _ptr(kblk),
                                   _ptr(kblk_q8), _ptr(kblk_scale_f16), _stream(k_cells)), "qsa_block_summary")


def device_error(device: torch.device | None = None) -> int:
    """Reads and clears the library's device error word (synchronises)."""
    code = ctypes.c_uint32(0)
    stream = torch.cuda.current_stream(device).cuda_stream
    _check(lib().qsa_get_device_error(ctypes.byref(code), stream), "qsa_get_device_error")
    return int(code.value)


WAIT_LIMIT_DEFAULT_NS = 2_000_000_000
INJECT_SCORER_STALL = 1    # the tensor-core scorer's CTA 0 never loads its first key piece
INJECT_DECODE_BARRIER = 2  # the fused decode select's grid barrier waits for one arrival too many


def debug_inject(faults: int, wait_limit_ns: int = WAIT_LIMIT_DEFAULT_NS) -> None:
    """``qsa_debug_inject``: diagnostics for the bounded waits. Kernels
    launched afterwards give up every spin-wait after ``wait_limit_ns`` and
    carry the planted faults (bits above); ``debug_inject(0)`` restores normal
    operation."""
    _check(lib().qsa_debug_inject(int(faults), int(wait_limit_ns)), "qsa_debug_inject")


def default_scorer_kernel() -> tuple[str, str]:
    """(kernel name, source file) of the scorer behind qsa_block_scores."""
    return "scores_tc_kernel", "scores_tc.cu"
