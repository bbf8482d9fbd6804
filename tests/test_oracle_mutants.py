"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a private copy of the oracle's C source (a
dropped term, a wrong sign, a wrong index or head mapping, an off-by-one mask
edge, a swapped operand), compiles it on the CPU, and checks that at least one
pin from test_oracle_pins fails against it. The real oracle is untouched.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_bwd_pins as bpins
from tests import test_oracle_mla_pins as mpins
from tests import test_oracle_paged_pins as ppins
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_ref.c")

MUTANTS = {
    "scale_dropped": ("sj = P->scale * dot + (brow ? brow[j] : 0.0);", "sj = dot + (brow ? brow[j] : 0.0);"),
    "bias_dropped": ("sj = P->scale * dot + (brow ? brow[j] : 0.0);", "sj = P->scale * dot;"),
    "bias_scaled": ("sj = P->scale * dot + (brow ? brow[j] : 0.0);",
                    "sj = P->scale * (dot + (brow ? brow[j] : 0.0));"),
    "exp_sign": ("double p = exp(sc[j] - m);", "double p = exp(m - sc[j]);"),
    "no_normalise": ("double wj = sc[j] / l;", "double wj = sc[j];"),
    "k_for_v": ("o[d] += wj * vh[j * D + d];", "o[d] += wj * kh[j * D + d];"),
    "gqa_modulo": ("const int64_t hk = hq / group;", "const int64_t hk = hq % s->Hkv;"),
    "causal_strict": ("!(j <= i + (Sk - Sq))", "!(j < i + (Sk - Sq))"),
    "causal_top_left": ("!(j <= i + (Sk - Sq))", "!(j <= i)"),
    "padding_inclusive": ("int visible = j < key_limit;", "int visible = j <= key_limit;"),
    "bias_row_index": ("brow = P->bias + ((bb * s->bias_h + bh) * Sq + i) * Sk;",
                       "brow = P->bias + ((bb * s->bias_h + bh) * Sq + (Sq - 1 - i)) * Sk;"),
    "bias_head_ignored": ("int64_t bh = (s->bias_h == 1) ? 0 : hq;", "int64_t bh = 0;"),
    "lse_no_max": ("if (lse) *lse = m + log(l);", "if (lse) *lse = log(l);"),
    "lse_log2": ("if (lse) *lse = m + log(l);", "if (lse) *lse = m + log2(l);"),
    "q_head_index": ("const double* qi = P->q + ((b * s->Hq + hq) * Sq + i) * D;",
                     "const double* qi = P->q + ((b * s->Hq + hk) * Sq + i) * D;"),
}


# Mistakes in the backward, caught by the backward pins.
MUTANTS_BWD = {
    "bwd_no_row_term": ("const double ds = w[j] * (dw[j] - wdw);", "const double ds = w[j] * dw[j];"),
    "bwd_dq_unscaled": ("dqi[d] += P->scale * ds * kh[j * D + d];", "dqi[d] += ds * kh[j * D + d];"),
    "bwd_dk_uses_k": ("dkh[j * D + d] += P->scale * ds * qi[d];", "dkh[j * D + d] += P->scale * ds * kh[j * D + d];"),
    "bwd_dv_uses_ds": ("dvh[j * D + d] += w[j] * gi[d];", "dvh[j * D + d] += ds * gi[d];"),
    "bwd_dw_uses_k": ("for (int64_t d = 0; d < D; ++d) g += gi[d] * vh[j * D + d];",
                      "for (int64_t d = 0; d < D; ++d) g += gi[d] * kh[j * D + d];"),
    "bwd_gqa_first_head_only": ("for (int64_t hq = hk * group; hq < (hk + 1) * group; ++hq) {",
                                "for (int64_t hq = hk * group; hq < hk * group + 1; ++hq) {"),
    "bwd_dv_sign": ("dvh[j * D + d] += w[j] * gi[d];", "dvh[j * D + d] -= w[j] * gi[d];"),
}


# Mistakes in the paged-cache attention, caught by the paged pins.
MUTANTS_PAGED = {
    "paged_row_reversed": ("const double* kj = kc + ((page * page_size + j % page_size) * Hkv + hk) * D;",
                           "const double* kj = kc + ((page * page_size + (page_size - 1 - j % page_size)) * Hkv + hk) * D;"),
    "paged_table_stride": ("if (!causal || j <= pos) {\n            const int64_t page = table[s * max_pages + j / page_size];",
                           "if (!causal || j <= pos) {\n            const int64_t page = table[s + j / page_size];"),
    "paged_causal_strict": ("if (!causal || j <= pos) {\n            const int64_t page",
                            "if (!causal || j < pos) {\n            const int64_t page"),
    "paged_default_positions": ("const int64_t pos = positions ? positions[t] : L - n + (t - q_off[s]);\n"
                                "      for (int64_t h = 0; h < Hq; ++h) {",
                                "const int64_t pos = positions ? positions[t] : L - n + (t - q_off[s]) - 1;\n"
                                "      for (int64_t h = 0; h < Hq; ++h) {"),
    "paged_v_head": ("const double* vj = vc + ((page * page_size + j % page_size) * Hkv + hk) * D;",
                     "const double* vj = vc + ((page * page_size + j % page_size) * Hkv + 0) * D;"),
}


# Mistakes in MLA, caught by the MLA pins.
MUTANTS_MLA = {
    "mla_no_positional_term": ("for (int64_t d = 0; d < Pd; ++d) dot += qpi[d] * kp[row * Pd + d];",
                               "for (int64_t d = 0; d < Pd; ++d) dot += 0.0 * qpi[d] * kp[row * Pd + d];"),
    "mla_value_from_query": ("for (int64_t d = 0; d < R; ++d) o[d] += w * lat[row * R + d];",
                             "for (int64_t d = 0; d < R; ++d) o[d] += w * qi[d];"),
    "mla_head_stride": ("const double* qpi = qp + (t * H + h) * Pd;", "const double* qpi = qp + (t * H) * Pd;"),
}


# Mistakes in the paged and MLA backward, caught by the paged backward pins.
MUTANTS_PBWD = {
    "pbwd_no_row_term": ("const double dsj = w[j] * (dw[j] - wdw);\n          for (int64_t d = 0; d < D; ++d) {",
                         "const double dsj = w[j] * dw[j];\n          for (int64_t d = 0; d < D; ++d) {"),
    "pbwd_dv_uses_ds": ("dv[row * D + d] += w[j] * gi[d];", "dv[row * D + d] += dsj * gi[d];"),
    "pbwd_dk_unscaled": ("dk[row * D + d] += scale * dsj * qi[d];", "dk[row * D + d] += dsj * qi[d];"),
    "pbwd_dk_overwrites": ("dk[row * D + d] += scale * dsj * qi[d];", "dk[row * D + d] = scale * dsj * qi[d];"),
    "mla_bwd_no_value_part": ("dlat[row * R + d] += scale * dsj * qi[d] + w[j] * gi[d];",
                              "dlat[row * R + d] += scale * dsj * qi[d];"),
    "mla_bwd_dkp_uses_q": ("dkp[row * Pd + d] += scale * dsj * qpt[d];", "dkp[row * Pd + d] += scale * dsj * qi[d];"),
    "mla_bwd_dqp_from_latent": ("dqpi[d] += scale * dsj * kp[row * Pd + d];",
                                "dqpi[d] += scale * dsj * lat[row * R + d];"),
}


def _pbwd_pins():
    from tests import test_oracle_paged_bwd_pins as pb
    yield lambda: pb.test_paged_bwd_matches_finite_differences(True, None)
    yield pb.test_shared_page_gradient_is_the_sum_over_private_copies
    yield lambda: pb.test_mla_bwd_is_paged_bwd_over_concatenated_keys(True, 2)
    yield pb.test_mla_bwd_matches_finite_differences


def _mla_pins():
    yield mpins.test_mla_single_key_returns_its_latent_row
    for causal in (True, False):
        for positions in (False, True):
            yield lambda c=causal, p=positions: mpins.test_mla_is_single_head_attention_over_concatenated_keys(c, p, 16)


def _paged_pins():
    for ps in (1, 4, 16):
        for sq_sk in ((5, 5), (3, 11), (1, 9)):
            yield lambda p=ps, s=sq_sk: ppins.test_equal_lengths_equal_dense_bottom_right_causal(p, s)
    yield ppins.test_variable_lengths_non_causal_equal_dense_key_padding
    yield ppins.test_decode_step_sees_every_key


def _bwd_pins():
    yield bpins.test_single_key
    yield bpins.test_identical_keys_give_zero_query_gradient
    yield lambda: bpins.test_key_gradients_sum_to_zero(0)
    yield lambda: bpins.test_matches_finite_differences_of_the_forward(0, None, (4, 4))
    yield lambda: bpins.test_matches_finite_differences_of_the_forward(pins.CAUSAL, (1, 4), (3, 6))


def _pins():
    yield pins.test_golden_single_row_service_example
    yield pins.test_golden_tensai_causal_mask_pattern
    yield pins.test_hand_solved_two_by_two
    yield pins.test_single_head_textbook_softmax
    yield pins.test_gqa_equals_mha_with_repeated_kv_heads
    yield pins.test_lse_hand_solved_and_single_key
    yield pins.test_lse_merges_two_key_halves
    for mask in (0, pins.CAUSAL, pins.PAD, pins.CAUSAL | pins.PAD):
        yield lambda m=mask: pins.test_identical_keys_give_mean_of_visible_values(m)
        yield lambda m=mask: pins.test_weights_are_row_stochastic_and_zero_where_masked(m)
        for bshape in (None, (1, 4), (2, 1)):
            for sq_sk in ((3, 3), (2, 5), (5, 3)):
                yield lambda m=mask, b=bshape, s=sq_sk: pins.test_brute_force_tiny(m, b, s)


@pytest.mark.parametrize("name", sorted(MUTANTS) + sorted(MUTANTS_BWD) + sorted(MUTANTS_PAGED) + sorted(MUTANTS_MLA)
                         + sorted(MUTANTS_PBWD))
def test_pins_catch_mutant(name, tmp_path, monkeypatch):
    old, new = {**MUTANTS, **MUTANTS_BWD, **MUTANTS_PAGED, **MUTANTS_MLA, **MUTANTS_PBWD}[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mut = tmp_path / "attn_mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", str(so), str(mut), "-lm"],
                   check=True)
    oracle._load()  # make sure the real one is configured, then swap the handle's functions
    import ctypes
    lib = ctypes.CDLL(str(so))
    real = oracle._lib
    lib.oracle_attention.argtypes = real.oracle_attention.argtypes
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = real.oracle_attention_rows.argtypes
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_attention_bwd.argtypes = real.oracle_attention_bwd.argtypes
    lib.oracle_attention_bwd.restype = ctypes.c_int
    lib.oracle_paged_attention.argtypes = real.oracle_paged_attention.argtypes
    lib.oracle_paged_attention.restype = ctypes.c_int
    lib.oracle_paged_mla.argtypes = real.oracle_paged_mla.argtypes
    lib.oracle_paged_mla.restype = ctypes.c_int
    for fn in ("oracle_paged_attention_bwd", "oracle_paged_mla_bwd"):
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
        getattr(lib, fn).restype = ctypes.c_int
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    pins_for = (_pins if name in MUTANTS else _bwd_pins if name in MUTANTS_BWD
                else _paged_pins if name in MUTANTS_PAGED else _mla_pins if name in MUTANTS_MLA else _pbwd_pins)
    for pin in pins_for():
        try:
            pin()
        except AssertionError:
            caught.append(pin)
            break
    assert caught, f"no pin detects the planted mistake {name!r}"
