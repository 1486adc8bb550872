"""Each plausible mistake planted in a copy of the oracle trips at least one pin.

The mistakes are planted on the CPU, in a temporary copy of the C source;
the committed oracle is never modified.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "decode_oracle.c")

# (name, text in the oracle, replacement): each is a mistake a reader could make.
MUTANTS = [
    ("dropped_scale", "s[l] = scale * acc;", "s[l] = acc;"),
    ("gqa_modulo_mapping", "const int kvh = h / group;", "const int kvh = h % h_kv;"),
    ("transposed_K", "(double)K[l * d_k + j]", "(double)K[j * n + l]"),
    ("sign_of_max_shift", "w[l] = exp(s[l] - m);", "w[l] = exp(m - s[l]);"),
    ("unnormalised_weights", "w[l] = w[l] / Z;", "w[l] = w[l];"),
    ("transposed_V", "acc += w[l] * (double)V[l * d_v + d];", "acc += w[l] * (double)V[d * n + l];"),
    ("dropped_last_row", "for (int64_t l = 0; l < n; ++l)\n            acc += w[l]",
     "for (int64_t l = 0; l < n - 1; ++l)\n            acc += w[l]"),
    ("lse_without_max", "if (lse) *lse = m + log(Z);", "if (lse) *lse = log(Z);"),
    ("combine_unnormalised", "acc += (exp(lse_parts[s] - L) / Z) *", "acc += exp(lse_parts[s] - L) *"),
    ("append_head_batch_swapped", "const int64_t row = ((int64_t)b * h_kv + h) * n_max + p;",
     "const int64_t row = ((int64_t)h * B + b) * n_max + p;"),
    ("causal_mask_leaks_next", "S[i * T + j] = (j > i) ?", "S[i * T + j] = (j > i + 1) ?"),
    ("kv_row_stride_uses_dk_for_v", "V + row0 * d_v,", "V + row0 * d_k,"),
    ("q_offset_per_kv_head", "oracle_decode_head(q + u * d_k,", "oracle_decode_head(q + (u / group) * d_k,"),
    ("e4m3_bias_8", "else mag = ldexp(1.0 + (double)M / 8.0, E - 7);",
     "else mag = ldexp(1.0 + (double)M / 8.0, E - 8);"),
    ("e4m3_subnormal_scale", "if (E == 0) mag = ldexp((double)M / 8.0, -6);",
     "if (E == 0) mag = ldexp((double)M / 8.0, -7);"),
    ("int8_unsigned", "return (double)(c >= 128 ? (int)c - 256 : (int)c);", "return (double)c;"),
    ("e4m3_ties_up", "if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
     "if (frac >= 0.5) r += 1.0;"),
    ("int8_limit_128", "const float Q = kind == 1 ? 127.0f : 448.0f;",
     "const float Q = kind == 1 ? 128.0f : 448.0f;"),
    ("absmax_signed", "const float m = fabsf(xr[j]);", "const float m = xr[j];"),
    ("int8_truncates", "const double n = nearbyint((double)v);", "const double n = trunc((double)v);"),
    ("dequant_drops_scale", "out[r * d + j] = (double)scales[r] * oracle_code_value(",
     "out[r * d + j] = oracle_code_value("),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libmutant.so"))
    o = oracle.Oracle(oracle.load_library(lib))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
        except (RuntimeError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
