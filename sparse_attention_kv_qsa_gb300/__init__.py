"""Exact QSA block selection on GB300: block scoring, per-query top-k,
attention over the selected blocks, and block summary keys on append.

The computation lives in ``libqsa.so`` (CUDA kernels for sm_103a behind the C
ABI of ``include/qsa.h``); ``qsa`` is its Python binding and ``workloads``
the seeded synthetic input generator.
"""

from .qsa import (  # noqa: F401
    QSAError,
    block_group_max,
    block_scores,
    block_scores_ffma,
    block_scores_gmax,
    block_scores_q8,
    block_scores_q8_gmax,
    block_select,
    block_select_gmax,
    block_select_small,
    block_select_static,
    block_summary,
    block_topk,
    block_topk_gmax,
    groups,
    select_scratch_bytes,
    debug_inject,
    default_scorer_kernel,
    device_error,
    sparse_attn,
)
