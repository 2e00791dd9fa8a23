"""Plants plausible slips in a copy of the oracle's C source and checks that the pins catch
every one of them (a pin that no slip can trip would pin nothing).  Runs on the CPU only;
the real oracle is never modified."""
import os

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sgmv_oracle.c")

# (name, text to find, replacement, count) -- each keeps every memory access in bounds.
MUTATIONS = [
    ("overwrite_instead_of_accumulate", "yt[n] += scale * s;", "yt[n] = scale * s;", None),
    ("dropped_scale", "yt[n] += scale * s;", "yt[n] += s;", None),
    ("wrong_sign", "yt[n] += scale * s;", "yt[n] -= scale * s;", None),
    ("transposed_B", "Bk[(size_t)c * (size_t)h_out + (size_t)n]",
     "Bk[(size_t)n * (size_t)r + (size_t)c]", None),
    ("transposed_A", "Ak[(size_t)j * (size_t)r + (size_t)c]",
     "Ak[(size_t)c * (size_t)h_in + (size_t)j]", None),
    ("last_row_dropped", "t < seg_starts[i + 1]; ++t", "t < seg_starts[i + 1] - 1; ++t", None),
    ("adapter_of_first_segment", "const int32_t k = seg_adapter[i];",
     "const int32_t k = seg_adapter[0] < 0 ? seg_adapter[i] : seg_adapter[0];", None),
    ("layer_offset_dropped", "(size_t)layer_idx * (size_t)h_in * (size_t)r",
     "(size_t)0 * (size_t)h_in * (size_t)r", None),
    ("layer_offset_of_B_dropped", "(size_t)layer_idx * (size_t)r * (size_t)h_out",
     "(size_t)0 * (size_t)r * (size_t)h_out", None),
    ("shrink_sum_not_reset", "double s = 0.0;\n                for (int32_t j = 0; j < h_in",
     "double s = (c > 0) ? 1e-3 : 0.0;\n                for (int32_t j = 0; j < h_in", None),
    ("validate_order_off_by_one", "if (seg_starts[i + 1] < seg_starts[i])",
     "if (seg_starts[i + 1] <= seg_starts[i])", None),
    ("negative_id_not_skipped", "if (k < 0) continue;", "if (k < 0) k = 0;", None),
    ("pointer_alignment_8", "A_addr[k] % 16 != 0", "A_addr[k] % 8 != 0", None),
    ("pointer_check_of_empty_segments", "|| seg_starts[i + 1] <= seg_starts[i]) continue;",
     ") continue;", None),
    ("pointer_check_b_alignment_dropped", "B_addr[k] == 0 || B_addr[k] % 16 != 0",
     "B_addr[k] == 0", None),
    ("plan_groups_empty_segments",
     "if (k < 0 || seg_starts[i + 1] <= seg_starts[i]) continue;\n        int32_t seen",
     "if (k < 0) continue;\n        int32_t seen", None),
    ("ranked_scale_of_first_adapter", "yt[n] += scale[k] * s;", "yt[n] += scale[0] * s;",
     None),
    ("ranked_transposed_B", "(size_t)layer_idx * (size_t)h_in * (size_t)r;\n        const double *Bk = B[k] + (size_t)layer_idx * (size_t)r * (size_t)h_out;\n        for (int32_t t = seg_starts[i]; t < seg_starts[i + 1]; ++t) {\n            const double *xt = x + (size_t)t * (size_t)h_in;\n            double *yt = y + (size_t)t * (size_t)h_out;\n            for (int32_t c = 0; c < r; ++c) {\n                double s = 0.0;\n                for (int32_t j = 0; j < h_in; ++j)\n                    s += xt[j] * Ak[(size_t)j * (size_t)r + (size_t)c];\n                v[c] = s;\n            }\n            for (int32_t n = 0; n < h_out; ++n) {\n                double s = 0.0;\n                for (int32_t c = 0; c < r; ++c)\n                    s += v[c] * Bk[(size_t)c * (size_t)h_out + (size_t)n];\n                yt[n] += scale[k] * s;",
     "(size_t)layer_idx * (size_t)h_in * (size_t)r;\n        const double *Bk = B[k] + (size_t)layer_idx * (size_t)r * (size_t)h_out;\n        for (int32_t t = seg_starts[i]; t < seg_starts[i + 1]; ++t) {\n            const double *xt = x + (size_t)t * (size_t)h_in;\n            double *yt = y + (size_t)t * (size_t)h_out;\n            for (int32_t c = 0; c < r; ++c) {\n                double s = 0.0;\n                for (int32_t j = 0; j < h_in; ++j)\n                    s += xt[j] * Ak[(size_t)j * (size_t)r + (size_t)c];\n                v[c] = s;\n            }\n            for (int32_t n = 0; n < h_out; ++n) {\n                double s = 0.0;\n                for (int32_t c = 0; c < r; ++c)\n                    s += v[c] * Bk[(size_t)n * (size_t)r + (size_t)c];\n                yt[n] += scale[k] * s;", None),
    ("base_W0_transposed", "s += xt[j] * wn[j];",
     "s += xt[j] * W0[(size_t)j * (size_t)h_out + (size_t)n];", None),
    ("base_accumulated", "            yt[n] = s;\n", "            yt[n] += s;\n", None),
    ("base_last_row_dropped", "for (int32_t t = 0; t < M; ++t) {",
     "for (int32_t t = 0; t < M - 1; ++t) {", None),
    ("base_lora_term_dropped",
     "return oracle_lora_apply(y, x, A, B, seg_starts, seg_adapter, num_segments, layer_idx, h_in,",
     "return 0 * oracle_lora_apply(y, x, A, B, seg_starts, seg_adapter, 0, layer_idx, h_in,",
     None),
    ("plan_rows_reversed", "rows[n++] = t;",
     "rows[n++] = seg_starts[j + 1] - 1 - (t - seg_starts[j]);", None),
]


@pytest.mark.parametrize("name,find,repl,count", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(tmp_path, name, find, repl, count):
    src = open(SRC).read()
    assert find in src, f"mutation anchor not found: {find!r}"
    if name == "negative_id_not_skipped":
        src = src.replace("const int32_t k = seg_adapter[i];", "int32_t k = seg_adapter[i];")
    mutated = src.replace(find, repl) if count is None else src.replace(find, repl, count)
    path = tmp_path / f"{name}.c"
    path.write_text(mutated)
    lib = oracle.OracleLib(oracle.build(force=True, src=str(path),
                                        out=str(tmp_path / f"{name}.so")))
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted slip {name}"
