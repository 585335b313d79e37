"""Planted mistakes: a copy of the oracle's C source with one plausible error
(a dropped term, a flipped sign, an off-by-one, a transposed operand) is
compiled on the CPU, and at least one pin must then fail.  This shows the pins
constrain the oracle rather than merely re-running it."""
import os
import subprocess

import pytest

import oracle
import test_oracle as pins
import test_oracle_gated_bwd as gated_pins
import test_oracle_tiles as tile_pins

MUTATIONS = [
    ("bias dropped", "float z = acc + bf16_to_f32(b[j]);", "float z = acc;",
     pins.test_hidden_and_down_exact_on_integers),
    ("relu sign flipped", "(z > 0.0f) ? f32_to_bf16(z) : (uint16_t)0", "(z < 0.0f) ? f32_to_bf16(z) : (uint16_t)0",
     pins.test_hidden_row_selection_and_relu_sign),
    ("capacity off by one", "if (cnt <= C) {", "if (cnt < C) {",
     lambda: pins.test_pack_brute_force_all_patterns(4)),
    ("overflow rule >= C", "if (cnt > C) overflow = 1;", "if (cnt >= C) overflow = 1;",
     lambda: pins.test_pack_brute_force_all_patterns(3)),
    ("index stored global", "idx[cell * C + cnt - 1] = (uint8_t)i;", "idx[cell * C + cnt - 1] = (uint8_t)(t * T + i);",
     pins.test_pack_hand_example),
    ("fallback order reversed", "row_fb[n] = n_fb;", "row_fb[n] = (n_fb == 0) ? 1 : (n_fb == 1 ? 0 : n_fb);",
     pins.test_pack_hand_example),
    ("down operand transposed",
     "for (int32_t j = 0; j < f; ++j) acc += bf16_to_f32(h[j]) * bf16_to_f32(W_down[(int64_t)j * d + c]);",
     "for (int32_t j = 0; j < f; ++j) acc += bf16_to_f32(h[j]) * bf16_to_f32(W_down[(int64_t)c * d + j % d]);",
     pins.test_hidden_and_down_exact_on_integers),
    ("l1 gradient dropped", "dZ[(int64_t)r * f + j] = (h > 0.0f) ? acc + lambda : 0.0f;",
     "dZ[(int64_t)r * f + j] = (h > 0.0f) ? acc : 0.0f;", pins.test_backward_closed_form_zero_upstream),
    ("relu mask >= 0 in weight grads", "float dz = (h > 0.0f) ? acc + lambda : 0.0f;",
     "float dz = (h >= 0.0f) ? acc + lambda : 0.0f;", pins.test_backward_closed_form_zero_upstream),
    ("grad input transposed",
     "acc += dZ[(int64_t)r * f + j] * bf16_to_f32(W_inT[(int64_t)j * d + k]);",
     "acc += dZ[(int64_t)r * f + j] * bf16_to_f32(W_inT[((int64_t)k * f + j) % ((int64_t)f * d)]);",
     pins.test_backward_matches_autograd),
    ("dW_down uses dz", "for (int32_t c = 0; c < d; ++c) gdown[c] += h * bf16_to_f32(g[c]);",
     "for (int32_t c = 0; c < d; ++c) gdown[c] += dz * bf16_to_f32(g[c]);",
     pins.test_backward_single_active_unit_rank_one),
    ("gated dG built from the gate", "*dg = dh * u;", "*dg = dh * g;", gated_pins.test_gated_backward_matches_autograd),
    ("gated L1 sign dropped", "float dh = acc + (h > 0.0f ? lambda : -lambda);", "float dh = acc + lambda;",
     gated_pins.test_gated_backward_zero_upstream_closed_form),
    ("gated pattern h > 0", "  if (h == 0.0f) {\n    *dg = 0.0f;", "  if (h <= 0.0f) {\n    *dg = 0.0f;",
     gated_pins.test_gated_backward_matches_autograd),
    ("gated dX without the up term",
     "        acc += dU[(int64_t)r * f + j] * bf16_to_f32(W_uT[(int64_t)j * d + k]);\n", "",
     gated_pins.test_gated_backward_matches_autograd),
    ("gated db from dU", "      gb += dg;", "      gb += du;", gated_pins.test_gated_backward_matches_autograd),
    ("rounding ties away", "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;",
     "if (rest >= 0x8000u) keep += 1u;", pins.test_bf16_rounding_hand_cases),
    ("tile slots out of order", "values[cell * C] = (uint16_t)(n_dense & 0xFFFF);",
     "values[cell * C] = (uint16_t)((n_dense ^ 1) & 0xFFFF);", tile_pins.test_tiles_hand_example),
    ("dense-tile rule >= C", "if (cnt > C) {\n        /* dense tile", "if (cnt >= C) {\n        /* dense tile",
     lambda: tile_pins.test_tiles_brute_force_all_patterns(3)),
    ("dense tiles left out of Y", "acc += bf16_to_f32(tile[i]) * bf16_to_f32(W_down[((int64_t)t * T + i) * d + c]);",
     "acc += 0.0f;", tile_pins.test_tiles_packed_product_equals_dense_bitwise),
    ("checker ignores slot numbers", "if (row_fb[n] != seen_fb) misnumbered = 1;", "",
     pins.test_format_checker_catches_each_violation),
    ("checker rejects unstored overflow rows", "if (row_fb[n] < fb_cap && fb_rows[row_fb[n]] != n) return 7;",
     "if (row_fb[n] >= fb_cap || fb_rows[row_fb[n]] != n) return 7;",
     pins.test_format_checker_catches_each_violation),
    ("checker index bound off by one", "if (i >= T) return 3;\n          if (s > 0 && i <= idx[cell * C + s - 1]) return 4;\n          if (bf16_to_f32(v) == 0.0f) return 5;\n        } else if (v != 0 || i != 0) {\n          return 6;\n        }\n      }\n    }\n  }\n  if (misnumbered)",
     "if (i > T) return 3;\n          if (s > 0 && i <= idx[cell * C + s - 1]) return 4;\n          if (bf16_to_f32(v) == 0.0f) return 5;\n        } else if (v != 0 || i != 0) {\n          return 6;\n        }\n      }\n    }\n  }\n  if (misnumbered)",
     pins.test_format_checker_catches_each_violation),
]


@pytest.mark.parametrize("name,old,new,pin", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_catches_planted_mistake(name, old, new, pin, tmp_path):
    with open(oracle._SRC) as fh:
        src = fh.read()
    assert src.count(old) == 1, name
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(lib), str(path)])
    with oracle.use_library(str(lib)):
        with pytest.raises(AssertionError):
            pin()
    pin()   # and the real oracle passes the same pin
