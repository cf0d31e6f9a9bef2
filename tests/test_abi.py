"""The C-ABI library: it builds, loads, exports every declared symbol, and
rejects bad arguments before launching anything (CPU only: no call here
reaches a kernel)."""
import ctypes
import os
import re

import pytest

from sparse_attention_kv_qsa_gb300 import build as qsa_build
from sparse_attention_kv_qsa_gb300 import qsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")

OK, INVALID, UNSUPPORTED = qsa.QSA_OK, qsa.QSA_ERR_INVALID, qsa.QSA_ERR_UNSUPPORTED
A = 0x10000      # fake, 16-byte aligned "device" addresses: never dereferenced
B = 0x20000
MIS = 0x20004    # misaligned


@pytest.fixture(scope="module")
def lib():
    qsa_build.build()
    return qsa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert set(names) == set(qsa.EXPORTED), names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and nothing from the oracle leaks into the product library
    with pytest.raises(AttributeError):
        getattr(lib, "qsa_oracle_scores")


def test_debug_inject_arguments(lib):
    f = lib.qsa_debug_inject
    assert f(4, 10 ** 6) == INVALID                 # unknown fault bit
    assert f(0, 0) == INVALID                       # zero limit
    assert f(0, 61 * 10 ** 9) == INVALID            # above 60 s
    assert f(0, qsa.WAIT_LIMIT_DEFAULT_NS) == OK    # normal operation (nothing launched)


def test_select_scratch_and_argument_errors(lib):
    f = lib.qsa_block_select
    n = qsa.select_scratch_bytes(256)
    assert n >= 256 * 4096 * 8 and qsa.select_scratch_bytes(0) == 0
    assert qsa.select_scratch_bytes(257) > n
    assert f(A, B, 8, 100, 50, 0, A, B, A, n, None) == INVALID            # k < 1
    assert f(A, B, 8, 100, 50, 5, A, None, A, n, None) == INVALID         # null ids
    assert f(A, B, 8, 100, 50, 5, A, B, None, n, None) == INVALID         # null scratch
    assert f(A, B, 8, 100, 50, 5, A, B, MIS, n, None) == INVALID          # misaligned scratch
    assert f(A, B, 8, 100, 50, 5, A, B, A, qsa.select_scratch_bytes(8) - 1, None) == INVALID   # too small
    assert f(A, B, 8, 100, 50, 5, None, B, A, n, None) == INVALID         # null scores
    assert f(A, B, 8, 100, 101, 5, A, B, A, n, None) == INVALID           # active > max_blocks
    assert f(A, B, 1, 10 ** 7, 393217, 5, A, B, A, n, None) == UNSUPPORTED
    assert f(None, None, 0, 100, 50, 5, None, None, None, 0, None) == OK  # no rows


def test_status_strings(lib):
    for s in (OK, INVALID, UNSUPPORTED, qsa.QSA_ERR_CUDA):
        assert qsa.status_string(s).startswith("QSA_")


def test_scores_argument_errors(lib):
    f = lib.qsa_block_scores
    assert f(A, B, 4, 100, 101, A, None) == INVALID        # active > max_blocks
    assert f(A, B, -1, 100, 10, A, None) == INVALID        # nq < 0
    assert f(A, B, 4, 100, -1, A, None) == INVALID         # active < 0
    assert f(None, B, 4, 100, 10, A, None) == INVALID      # null q
    assert f(A, None, 4, 100, 10, A, None) == INVALID      # null kblk
    assert f(A, B, 4, 100, 10, None, None) == INVALID      # null scores
    assert f(MIS, B, 4, 100, 10, A, None) == INVALID       # misaligned q
    assert f(A, MIS, 4, 100, 10, A, None) == INVALID       # misaligned kblk
    assert f(A, B, 4, 100, 10, MIS, None) == INVALID       # misaligned scores
    assert f(None, None, 0, 100, 10, None, None) == OK     # no work
    assert f(None, None, 4, 100, 0, None, None) == OK      # no active blocks


def test_q8_argument_errors(lib):
    f = lib.qsa_block_scores_q8
    assert f(A, B, None, 4, 100, 10, A, None) == INVALID   # null scales
    assert f(A, B, B + 1, 4, 100, 10, A, None) == INVALID  # odd scale address
    assert f(A, MIS, B, 4, 100, 10, A, None) == INVALID    # misaligned keys
    assert f(A, B, B, 4, 10, 11, A, None) == INVALID
    g = lib.qsa_block_scores_ffma
    assert g(A, B, B, B, 4, 100, 10, A, None) == INVALID   # both key forms
    assert g(A, None, None, None, 4, 100, 10, A, None) == INVALID


def test_topk_argument_errors(lib):
    f = lib.qsa_block_topk
    assert f(A, 4, 100, 0, B, None) == INVALID              # k < 1
    assert f(A, -1, 100, 5, B, None) == INVALID
    assert f(A, 4, -3, 5, B, None) == INVALID
    assert f(A, 4, 100, 5, None, None) == INVALID           # null ids
    assert f(None, 4, 100, 5, B, None) == INVALID           # null scores (k < active)
    assert f(MIS, 4, 100, 5, B, None) == INVALID
    assert f(A, 4, 100, 5, MIS, None) == INVALID
    assert f(A, 4, qsa.TOPK_MAX_ACTIVE + 1, 5, B, None) == UNSUPPORTED
    assert f(None, 0, 100, 5, None, None) == OK             # no rows


def test_device_error_argument(lib):
    assert lib.qsa_get_device_error(None, None) == INVALID


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sparse_attention_kv_qsa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".c", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "qsa_oracle" not in text, fn


def test_group_max_argument_errors(lib):
    f = lib.qsa_block_scores_gmax
    assert f(A, B, 8, 100, 10, A, None, None) == INVALID     # null group_max
    assert f(A, B, 8, 100, 10, A, MIS, None) == INVALID      # misaligned group_max
    assert f(A, B, 8, 100, 101, A, B, None) == INVALID       # active > max_blocks
    assert f(None, None, 0, 100, 10, None, None, None) == OK  # no work
    g = lib.qsa_block_scores_q8_gmax
    assert g(A, B, B, 8, 100, 10, A, None, None) == INVALID
    assert g(A, B, B + 1, 8, 100, 10, A, B, None) == INVALID  # odd scale address
    h = lib.qsa_block_group_max
    assert h(A, 4, 100, None, None) == INVALID
    assert h(MIS, 4, 100, B, None) == INVALID
    assert h(A, -1, 100, B, None) == INVALID
    assert h(None, 0, 100, None, None) == OK
    t = lib.qsa_block_topk_gmax
    assert t(A, None, 4, 100, 5, B, None) == INVALID          # null group_max
    assert t(A, MIS, 4, 100, 5, B, None) == INVALID
    assert t(A, B, 4, 100, 0, B, None) == INVALID             # k < 1
    assert t(A, B, 4, qsa.TOPK_MAX_ACTIVE + 1, 5, B, None) == UNSUPPORTED
    assert t(None, None, 0, 100, 5, None, None) == OK
