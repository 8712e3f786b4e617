"""Planted mistakes in copies of the oracle must each fail at least one pin.

This shows the pins are strong enough: a dropped term, a wrong sign, a wrong
index or head map, or a transposed operand anywhere in ne_oracle.c is caught.
Each mutation is a textual edit of a temporary copy of the C source; the real
oracle is untouched.  CPU only.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ne_oracle.c")

# (name, original text, planted text)
MUTATIONS = [
    ("rope_sign", "y[i] = x0 * c - x1 * s;", "y[i] = x0 * c + x1 * s;"),
    ("rope_pairing_interleaved", "double x0 = x[i], x1 = x[i + half];",
     "double x0 = x[2 * i], x1 = x[2 * i + 1];"),
    ("rope_frequency_exponent", "pow(theta, -2.0 * (double)i / (double)d)",
     "pow(theta, -1.0 * (double)i / (double)d)"),
    ("rope_position_one_based", "(long)t + pos_offset, 0);", "(long)t + 1 + pos_offset, 0);"),
    ("gqa_map_interleaved_fwd", "j = h / G;", "j = h % Hkv;"),
    ("gqa_map_interleaved_bwd", "for (int h = j * G; h < (j + 1) * G; ++h)",
     "for (int h = j; h < Hq; h += Hkv)"),
    ("causal_excludes_diagonal", "if (s > t) {", "if (s >= t && t > 0) {"),
    ("score_scale", "double scale = 1.0 / sqrt((double)d);\n    for (int t = 0; t < T; ++t) {",
     "double scale = 1.0 / (double)d;\n    for (int t = 0; t < T; ++t) {"),
    ("lse_log2", "double l = mx + log(sum);", "double l = mx + log2(sum);"),
    ("ds_drops_D", "double ds = p * (dp - Dt);", "double ds = p * dp;"),
    ("dk_drops_scale", "dkr[(size_t)s * d + c] += scale * ds * qr[(size_t)t * d + c];",
     "dkr[(size_t)s * d + c] += ds * qr[(size_t)t * d + c];"),
    ("dq_uses_q_not_k", "dqr[(size_t)t * d + c] += scale * ds * kr[(size_t)s * d + c];",
     "dqr[(size_t)t * d + c] += scale * ds * qr[(size_t)t * d + c];"),
    ("dv_transposed_operand", "dvrow[c] += p * dorow[c];", "dvrow[c] += p * vrow[c];"),
    ("dq_forward_rotation", "rope_row(dqr + (size_t)t * d, dq + IDX(b, t, h, 0, T, Hq, d), d, theta,\n                         (long)t + pos_offset, 1);",
     "rope_row(dqr + (size_t)t * d, dq + IDX(b, t, h, 0, T, Hq, d), d, theta,\n                         (long)t + pos_offset, 0);"),
    ("dk_skips_inverse_rotation", "(long)s + pos_offset, 1);", "(long)s + pos_offset + 3, 1);"),
    ("window_off_by_one", "if (window > 0 && t - s >= window) {",
     "if (window > 0 && t - s > window) {"),
    ("decode_query_position", "(long)(Tk - 1) + pos_offset, 0);", "(long)Tk + pos_offset, 0);"),
    ("decode_kv_head_interleaved", "const int kvh = h / G;", "const int kvh = h % Hkv;"),
    ("decode_drops_normaliser", "double pr = exp(S[s] - lse_bh);", "double pr = exp(S[s] - mx);"),
    ("varlen_lse_padding_zero", "lse[((size_t)b * Hq + h) * T + t] = -INFINITY;",
     "lse[((size_t)b * Hq + h) * T + t] = 0.0;"),
    ("varlen_fwd_full_length", "1, L, Hq, Hkv, d, theta, pos_offset, nthreads, 0);",
     "1, T, Hq, Hkv, d, theta, pos_offset, nthreads, 0);"),
    ("varlen_bwd_reads_padding_dO", "dv + IDX(b, 0, 0, 0, T, Hkv, d), NULL, NULL, NULL, 1, L,",
     "dv + IDX(b, 0, 0, 0, T, Hkv, d), NULL, NULL, NULL, 1, T,"),
    ("varlen_batch_stride", "err = ne_oracle_fwd(q + IDX(b, 0, 0, 0, T, Hq, d),",
     "err = ne_oracle_fwd(q + IDX(b, 0, 0, 0, L, Hq, d),"),
    ("varlen_lse_row_stride", "* T, lse1 + (size_t)h * L, sizeof(double) * L);",
     "* T, lse1 + (size_t)h * T, sizeof(double) * L);"),
    ("packed_output_stride", "o + (size_t)cu[b] * Hq * d, lse1",
     "o + (size_t)cu[b] * Hkv * d, lse1"),
    ("packed_lse_drops_offset", "memcpy(lse + (size_t)h * total + cu[b],",
     "memcpy(lse + (size_t)h * total,"),
    ("packed_bwd_dO_stride", "dO + (size_t)cu[b] * Hq * d,", "dO + (size_t)cu[b] * Hkv * d,"),
]


@pytest.mark.parametrize("name,orig,planted", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, orig, planted):
    text = open(SRC).read()
    assert text.count(orig) == 1, f"mutation {name}: anchor text not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(orig, planted))
    lib = oracle.compile_source(str(src), str(tmp_path / "libmutant.so"))
    mutant = oracle.load_from(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"
