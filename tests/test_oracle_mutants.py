"""Negative controls for the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of the oracle's C source
(a dropped head, a wrong sign, a wrong stride, a reversed tie rule, ...),
builds it into a temporary library, and requires that at least one pin
fails. A mutation whose target text is missing fails the test, so the list
cannot silently go stale when the oracle changes.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "dropped_head": ("h < QSA_H; ++h", "h < QSA_H - 1; ++h"),
    "wrong_sign": ("dot += (double)qh[d] * (double)kb[d]", "dot -= (double)qh[d] * (double)kb[d]"),
    "head_stride": ("qi + h * QSA_D", "qi + h"),
    "short_d_loop": ("for (int d = 0; d < QSA_D; ++d) dot += (double)qh[d] * (double)kb[d]",
                     "for (int d = 1; d < QSA_D; ++d) dot += (double)qh[d] * (double)kb[d]"),
    "tie_to_higher_id": ("return (a->id < b->id) ? -1 : (a->id > b->id);",
                         "return (a->id > b->id) ? -1 : (a->id < b->id);"),
    "ascending_scores": ("if (va > vb) return -1;", "if (va < vb) return -1;"),
    "nan_ranks_first": ("isnan(s) ? -INFINITY : s", "isnan(s) ? INFINITY : s"),
    "ids_in_rank_order": ("qsort(out, (size_t)m, sizeof(int32_t), by_id_asc);", ""),
    "zero_padding": ("for (long j = m; j < c->k; ++j) out[j] = -1;",
                     "for (long j = m; j < c->k; ++j) out[j] = 0;"),
    "half_bias": ("ldexp((double)(1024 + m), e - 25)", "ldexp((double)(1024 + m), e - 24)"),
    "half_subnormal": ("ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    "scale_dropped": ("((double)kb[d] * scale)", "((double)kb[d])"),
    "float_key_trunc": ("(double)c->S32[(size_t)i * n + b]", "(double)(int)c->S32[(size_t)i * n + b]"),
    "attn_no_temperature": ("w[t] = dot * temperature;", "w[t] = dot;"),
    "attn_cell_index": ("if (4 * b + t < c->ncells) cells[n++] = 4 * b + t;",
                        "if (4 * b + t < c->ncells) cells[n++] = 4 * b;"),
    "attn_k_scale_dropped": ("((double)kc[d] * scale)", "((double)kc[d])"),
    "attn_v_scale_dropped": ("((double)vc[d] * scale)", "((double)vc[d])"),
    "attn_head_stride": ("((size_t)i * QSA_H + (size_t)h) * QSA_D", "((size_t)i * QSA_H) * QSA_D"),
    "attn_unnormalised": ("const double p = w[t] / total;", "const double p = w[t];"),
    "attn_exponent_sign": ("w[t] = exp(w[t] - top);", "w[t] = exp(top - w[t]);"),
    "summary_divide_by_4": ("mean[d] = n > 0 ? sum / (float)n : 0.0f;", "mean[d] = n > 0 ? sum / 4.0f : 0.0f;"),
    "summary_scale_255": ("float_to_half_rne(top / 127.0f)", "float_to_half_rne(top / 255.0f)"),
    "summary_truncated_codes": ("rintf(mean[d] / s)", "truncf(mean[d] / s)"),
    "summary_cell_stride": ("const long c = 4 * b + t;", "const long c = 2 * b + t;"),
    "summary_scale_dropped": ("(float)kq[(size_t)c * QSA_D + d] * (float)qsa_oracle_half_to_double(ks[c])",
                              "(float)kq[(size_t)c * QSA_D + d]"),
    "half_no_rounding": ("if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;", ""),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert old in src, f"mutation target for {name} not found in the oracle source"
    mut = tmp_path / "qsa_oracle_mutant.c"
    mut.write_text(src.replace(old, new))
    # the mutant includes the oracle's own header from the oracle directory
    lib = oracle.build(force=True, source=str(mut), out=str(tmp_path / "libmutant.so"))
    o = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path):
    with open(oracle.SOURCE) as f:
        src = f.read()
    cp = tmp_path / "qsa_oracle_copy.c"
    cp.write_text(src)
    o = oracle.Oracle(oracle.build(force=True, source=str(cp), out=str(tmp_path / "libcopy.so")))
    for pin in oracle_pins.ALL_PINS:
        pin(o)
    assert os.path.exists(tmp_path / "libcopy.so")
