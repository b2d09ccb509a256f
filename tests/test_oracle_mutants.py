"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
the pins catch every one of them."""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gemm_tn_oracle.c")

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("drop_beta_term", "v = v + beta * g_decode[*c_elem];", "v = v;"),
    ("drop_alpha", "double v = alpha * acc;", "double v = acc;"),
    ("wrong_operand", "g_decode[a_row[k]] * g_decode[b_row[k]]", "g_decode[a_row[k]] * g_decode[a_row[k]]"),
    ("skip_last_k", "for (int64_t k = 0; k < K; ++k) {\n        acc +=", "for (int64_t k = 0; k + 1 < K; ++k) {\n        acc +="),
    ("b_uses_lda", "B + b * strideB + n * ldb;", "B + b * strideB + n * lda;"),
    ("c_transposed", "(C + b * strideC + m * ldc + n) : NULL;\n            D[", "(C + b * strideC + n * ldc + m) : NULL;\n            D["),
    ("batch_stride_mixup", "const uint16_t* a_row = A + b * strideA + m * lda;\n        for", "const uint16_t* a_row = A + b * strideB + m * lda;\n        for"),
    ("truncate_not_rne", "rint(ldexp(a, -q))", "trunc(ldexp(a, -q))"),
    ("ties_away", "rint(ldexp(a, -q))", "round(ldexp(a, -q))"),
    ("saturate_not_inf", "if (bits >= 0x7c00) bits = 0x7c00;", "if (bits >= 0x7c00) bits = 0x7bff;"),
    ("subnormal_scale", "v = ldexp((double)frac, -24);", "v = ldexp((double)frac, -25);"),
    ("exponent_bias", "expo - 25);", "expo - 24);"),
    ("lost_sign", "return sign ? -v : v;", "return v;"),
    # (mutants stay inside the operand buffers: an out-of-range read would be undefined)
    ("strided_a_unit_k_stride", "A[b * strideA + m * a_rs + k * a_cs]", "A[b * strideA + m * a_rs + k]"),
    ("strided_b_unit_row_stride", "B[b * strideB + n * b_rs + k * b_cs]", "B[b * strideB + n + k * b_cs]"),
    ("transpose_drops_last_row", "for (int64_t r = 0; r < rows; ++r)\n        for (int64_t c = 0; c < cols; ++c) Y[c * ldy + r] = X[r * ldx + c];\n}\n\nvoid gto_transpose_u16",
     "for (int64_t r = 0; r + 1 < rows; ++r)\n        for (int64_t c = 0; c < cols; ++c) Y[c * ldy + r] = X[r * ldx + c];\n}\n\nvoid gto_transpose_u16"),
    ("softmax_sum_drops_last_key", "for (int64_t j = 0; j < N; ++j) {\n            l += exp(",
     "for (int64_t j = 0; j + 1 < N; ++j) {\n            l += exp("),
    ("softmax_max_skips_last_key", "for (int64_t j = 0; j < N; ++j) {\n            const double s =",
     "for (int64_t j = 0; j + 1 < N; ++j) {\n            const double s ="),
    ("softmax_exp_sign", "l += exp(score(q_row, k_base + j * ldk, d, al) - m);", "l += exp(m - score(q_row, k_base + j * ldk, d, al));"),
    ("softmax_max_starts_at_zero", "double m = -INFINITY;", "double m = 0.0;"),
    ("softmax_drops_alpha", "return alpha * acc;", "return acc;"),
    ("softmax_key_uses_ldq", "const double s = score(q_row, k_base + j * ldk, d, al);", "const double s = score(q_row, k_base + j * ldq, d, al);"),
    ("softmax_dot_skips_last", "for (int64_t k = 0; k < d; ++k) acc +=", "for (int64_t k = 0; k + 1 < d; ++k) acc +="),
    ("softmax_key_batch_stride", "const uint16_t* k_base = K + b * strideK;", "const uint16_t* k_base = K + b * strideQ;"),
    ("flush_subnormals", "const int q = (E < -14) ? -24 : E - 10;", "const int q = (E < -14) ? 99 : E - 10;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    path = tmp_path / f"{name}.c"
    path.write_text(mutated)
    lib = oracle.compile_source(str(path), str(tmp_path / f"lib_{name}.so"))
    o = oracle.Oracle.from_path(lib)
    failures = []
    for check in pins.CONVERSION_CHECKS[:3] + pins.GEMM_CHECKS + pins.SOFTMAX_CHECKS:
        try:
            check(o)
        except AssertionError:
            failures.append(check.__name__)
        except Exception as e:  # noqa: BLE001 - a crash in a check also counts as caught
            failures.append(f"{check.__name__}:{type(e).__name__}")
    assert failures, f"mutant {name} passed every pin"
