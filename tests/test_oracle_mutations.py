"""The pins catch plausible mistakes in the oracle.

Each case copies the oracle's C source, plants one mistake by a textual edit,
compiles the copy into a temporary directory and runs every pin against it:
at least one pin must fail.  The real oracle is never modified.  CPU only.
"""
import os

import pytest

import oracle
from oracle import build as obuild

from pins import ALL_PINS

MUTATIONS = {
    # wrong divisor in the mean of squares
    "mean_over_H_minus_1": ("ss / (double)H", "ss / (double)(H - 1)"),
    # eps dropped from under the root
    "drop_eps": ("ss / (double)H + (double)j->eps", "ss / (double)H"),
    # eps outside the root
    "eps_outside_root": ("1.0 / sqrt(ss / (double)H + (double)j->eps)",
                         "1.0 / (sqrt(ss / (double)H) + (double)j->eps)"),
    # weight read at the wrong index
    "gamma_reversed": ("load_elem(j->dt, j->gamma, i)", "load_elem(j->dt, j->gamma, H - 1 - i)"),
    # reciprocal used the wrong way round
    "divide_by_inv": ("(h[i] * inv)", "(h[i] / inv)"),
    # residual not added
    "drop_residual": ("acc = acc + (float)load_elem(j->rdt, j->residual_in, rrow + i);", ""),
    # partial sum kept in binary64 instead of binary32
    "wide_accumulator": ("float acc = (float)load_elem", "double acc = (float)load_elem"),
    # wrong stride between partial buffers
    "partial_stride": ("(int64_t)r * j->slice + xrow + i", "(int64_t)r * j->H + xrow + i"),
    # first partial skipped
    "skip_p0": ("float acc = (float)load_elem(j->dt, j->x, xrow + i);", "float acc = 0.0f;"),
    # sum of squares from the unrounded sum
    "unrounded_h": ("h[i] = round_dt(j->rdt, (double)acc);", "h[i] = (double)acc;"),
    # residual decoded / rounded with the type of x instead of its own
    "residual_decoded_as_x": ("load_elem(j->rdt, j->residual_in", "load_elem(j->dt, j->residual_in"),
    "residual_rounded_as_x": ("h[i] = round_dt(j->rdt, (double)acc);",
                              "h[i] = round_dt(j->dt, (double)acc);"),
    # row strides ignored
    "x_stride": ("const int64_t xrow = t * j->ldx;", "const int64_t xrow = t * j->H;"),
    "residual_stride": ("const int64_t rrow = t * j->ldr;", "const int64_t rrow = t * j->H;"),
    "y_stride": ("const int64_t yrow = t * j->ldy;", "const int64_t yrow = t * j->H;"),
    # ties away from zero instead of to even
    "ties_away": ("nearbyint(ldexp(v, -q))", "round(ldexp(v, -q))"),
    # truncation instead of rounding
    "truncate": ("nearbyint(ldexp(v, -q))", "trunc(ldexp(v, -q))"),
    # f16 subnormal scale off by one
    "f16_subnormal": ("ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    # f16 exponent bias off by one
    "f16_bias": ("ldexp((double)(m + 1024), e - 25)", "ldexp((double)(m + 1024), e - 24)"),
    # bf16 precision wrong
    "bf16_precision": ("return round_to_format(v, 8, -126, 127);",
                       "return round_to_format(v, 9, -126, 127);"),
    # sign of the squares
    "square_sign": ("ss += h[i] * h[i];", "ss += h[i] * fabs(h[i]);"),
    # no overflow to infinity
    "no_overflow": ("if (fabs(out) > max_finite) return copysign(INFINITY, v);", ""),
    # 8-bit output: no saturation (the largest code pattern instead)
    "fp8_no_saturation": ("r = copysign(f->maxf, v);", "r = NAN;"),
    # e4m3 with one significant bit too many / an exponent range off by one
    "e4m3_precision": ("{4, -6, 8, 3, 7, 448.0}", "{5, -6, 8, 3, 7, 448.0}"),
    "e4m3_emin": ("{4, -6, 8, 3, 7, 448.0}", "{4, -7, 8, 3, 7, 448.0}"),
    "e5m2_max": ("{3, -14, 15, 2, 15, 57344.0}", "{3, -14, 15, 2, 15, 61440.0}"),
    # exponent bias off by one in the encoder / decoder
    "fp8_encode_bias": ("((lead + f->bias) << f->mbits)", "((lead + f->bias + 1) << f->mbits)"),
    "fp8_decode_subnormal": ("ldexp((double)m, f->emin - f->mbits)",
                             "ldexp((double)m, f->emin - f->mbits - 1)"),
    # scale applied the wrong way round / per-row divisor wrong
    "fp8_scale_multiplied": ("const double u = v[i] / s;", "const double u = v[i] * s;"),
    "fp8_row_divisor": ("s = amax > 0.0 ? amax / f->maxf : 1.0;",
                        "s = amax > 0.0 ? amax / 256.0 : 1.0;"),
    "fp8_zero_row_scale": ("s = amax > 0.0 ? amax / f->maxf : 1.0;",
                           "s = amax > 0.0 ? amax / f->maxf : 0.0;"),
    # signed maximum instead of the maximum magnitude
    "fp8_signed_amax": ("if (fabs(v[i]) > amax) amax = fabs(v[i]);", "if (v[i] > amax) amax = v[i];"),
    # residual not written back / code rows not strided
    "fp8_residual_not_stored": (
        "for (int64_t i = 0; i < H; ++i) store_exact(dt, residual, rrow + i, h[i]);", ""),
    "fp8_code_stride": ("codes[t * ldq + i]", "codes[t * H + i]"),
    # gamma dropped from the 8-bit path
    "fp8_no_gamma": ("v[i] = (h[i] * inv) * load_elem(dt, gamma, i);", "v[i] = h[i] * inv;"),
    # GEMM producer: strides ignored, a product dropped, |.| dropped
    "gemm_w_stride": ("W64[i * K + k] = load_elem(dt, W, i * ldw + k);",
                      "W64[i * K + k] = load_elem(dt, W, i * K + k);"),
    "gemm_a_stride": ("arow[k] = load_elem(g->dt, g->A, t * g->lda + k);",
                      "arow[k] = load_elem(g->dt, g->A, t * g->K + k);"),
    "gemm_drop_last_k": ("for (int64_t k = 0; k < K; ++k) {\n            const double prod",
                         "for (int64_t k = 0; k < K - 1; ++k) {\n            const double prod"),
    "gemm_abs_signed": ("a += fabs(prod);", "a += prod;"),
    # the partial rounded on its own first / residual not added or not stored
    "gemm_round_partial_first": (
        "h[i] = round_dt(g->dt, P + load_elem(g->dt, g->residual, t * g->ldr + i));",
        "h[i] = round_dt(g->dt, round_dt(g->dt, P) + load_elem(g->dt, g->residual, "
        "t * g->ldr + i));"),
    "gemm_no_residual": (
        "h[i] = round_dt(g->dt, P + load_elem(g->dt, g->residual, t * g->ldr + i));",
        "h[i] = round_dt(g->dt, P);"),
    "gemm_residual_not_stored": (
        "for (int64_t i = 0; i < H; ++i) store_exact(g->dt, g->residual, t * g->ldr + i, h[i]);",
        ""),
    # 8-bit partials: scale dropped / one scale for all / scale after the sum,
    # wrong partial stride, binary64 accumulator, the other format, residual
    # dropped or not stored
    "fp8in_no_scale": ("float acc = (float)decode_fp8(f, j->codes[row + i]) * j->scales[0];",
                       "float acc = (float)decode_fp8(f, j->codes[row + i]);"),
    "fp8in_scale0_for_all": ("j->scales[r];", "j->scales[0];"),
    "fp8in_partial_stride": ("j->codes[(int64_t)r * j->T * H + row + i]",
                             "j->codes[(int64_t)r * H + row + i]"),
    "fp8in_wide_accumulator": ("float acc = (float)decode_fp8", "double acc = (float)decode_fp8"),
    "fp8in_other_format": ("const fp8_format *f = &FP8[j->fmt];",
                           "const fp8_format *f = &FP8[1 - j->fmt];"),
    "fp8in_no_residual": ("acc = acc + (float)load_elem(j->dt, j->residual_in, row + i);", ""),
    "fp8in_residual_not_stored": (
        "if (j->residual_out)\n        for (int64_t i = 0; i < H; ++i) store_exact(j->dt, "
        "j->residual_out, row + i, h[i]);", ""),
    # tensor-parallel form: ranks summed in reverse order, rank 0 skipped, the
    # residual dropped or read from rank 0's block, y gathered into rank 0's
    # buffer only, blocks of rows that overlap or leave gaps
    "tp_reverse_rank_order": (
        "float rank_sum = (float)load_elem(j->dt, j->bufs[0], row + i);\n"
        "        for (int32_t q = 1; q < j->N; ++q)\n"
        "            rank_sum = rank_sum + (float)load_elem(j->dt, j->bufs[q], row + i);",
        "float rank_sum = (float)load_elem(j->dt, j->bufs[j->N - 1], row + i);\n"
        "        for (int32_t q = j->N - 2; q >= 0; --q)\n"
        "            rank_sum = rank_sum + (float)load_elem(j->dt, j->bufs[q], row + i);"),
    "tp_skip_rank0": ("float rank_sum = (float)load_elem(j->dt, j->bufs[0], row + i);",
                      "float rank_sum = 0.0f;"),
    "tp_no_residual": ("rank_sum = rank_sum + (float)load_elem(j->dt, j->residual_in, row + i);",
                       ""),
    "tp_residual_block": ("jr.residual_in = (const char *)residual_in + off;",
                          "jr.residual_in = residual_in;"),
    "tp_gather_rank0_only": (
        "for (int32_t q = 0; q < j->N; ++q) store_exact(j->dt, j->y_out[q], row + i, yv);",
        "store_exact(j->dt, j->y_out[0], row + i, yv);"),
    "tp_blocks_ceil": ("*r0 = T * (int64_t)r / N;", "*r0 = (T * (int64_t)r + N - 1) / N;"),
    "tp_blocks_short": ("*r1 = T * (int64_t)(r + 1) / N;", "*r1 = T * (int64_t)(r + 1) / N - 1;"),
    "tp_wide_accumulator": ("float rank_sum = (float)load_elem", "double rank_sum = (float)load_elem"),
    "gemm_gamma_index": ("round_dt(g->dt, (h[i] * inv) * load_elem(g->dt, g->gamma, i))",
                         "round_dt(g->dt, (h[i] * inv) * load_elem(g->dt, g->gamma, 0))"),
}


@pytest.fixture(scope="module")
def src_text():
    with open(obuild.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, src_text, tmp_path):
    old, new = MUTATIONS[name]
    assert src_text.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src_text.replace(old, new)
    src = os.path.join(tmp_path, "mut.c")
    with open(src, "w") as f:
        f.write(mutated)
    lib = obuild.compile_source(src, os.path.join(tmp_path, "libmut.so"))
    O = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(O)
        except (AssertionError, RuntimeError, ValueError, OverflowError, ZeroDivisionError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {name}"
