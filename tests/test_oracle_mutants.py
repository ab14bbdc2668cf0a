"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one.  The mutants are compiled from text substitutions of
``oracle/attn_oracle.c`` into a temporary directory; the real oracle is not
touched.  CPU only."""
import os

import pytest

import oracle
from tests import oracle_pins as pins

# (name, original text, mutated text)
MUTANTS = [
    ("causal_off_by_one", "mask == 1 ? (long)q : (long)q + Kb - Qb;",
     "mask == 1 ? (long)q : (long)q + Kb - Qb - 1;"),
    ("top_left_causal", "mask == 1 ? (long)q : (long)q + Kb - Qb;",
     "mask == 1 ? (long)q : (long)q;"),
    ("top_left_off_by_one", "mask == 1 ? (long)q :", "mask == 1 ? (long)q + 1 :"),
    ("top_left_is_bottom_right", "mask == 1 ? (long)q :", "mask == 1 ? (long)q + Kb - Qb :"),
    ("no_mask_drops_last_key", "        *hi = (long)Kb - 1;\n        return;",
     "        *hi = (long)Kb - 2;\n        return;"),
    ("no_mask_is_causal", "    if (mask == 2) {                                   /* no mask: every key */",
     "    if (mask == 3) {                                   /* no mask: every key */"),
    ("head_map_modulo", "const int kh = h / G;", "const int kh = h % Hkv;"),
    ("window_one_wider", "diag - window + 1 > *lo) *lo = diag - window + 1;",
     "diag - window > *lo) *lo = diag - window;"),
    ("scale_dropped", "const double s = scale * acc;", "const double s = acc;"),
    ("lse_without_max", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("lse_base2", "*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    ("no_normalisation", "orow[j] /= l;", "orow[j] /= 1.0;"),
    ("empty_row_lse_zero", "if (hi < lo) { *lse_out = -INFINITY; return; }",
     "if (hi < lo) { *lse_out = 0.0; return; }"),
    ("v_uses_k_stride", "const float *vrow = vbase + k * vstride;",
     "const float *vrow = vbase + k * kstride;"),
    ("padded_row_kept", "            if (qi >= Qb) {", "            if (qi > Qb) {"),
    ("kv_ignores_batch", "oracle_row(q + r * D, k + ((long)b * K * Hkv + kh) * D,",
     "oracle_row(q + r * D, k + ((long)kh) * D,"),
    ("exp_not_shifted", "const double p = exp(s_scratch[k - lo] - m);",
     "const double p = exp(s_scratch[k - lo]) * 1.0000001;"),
    ("q_transposed_index", "oracle_row(q + r * D, k + ((long)b * K * Hkv + kh) * D,",
     "oracle_row(q + ((r % Hq) * Q + (r / Hq) % Q + (r / ((long)Hq * Q)) * Q * Hq) * D, k + ((long)b * K * Hkv + kh) * D,"),
    # backward
    ("bwd_drops_row_term", "const double ds = p * (dp - Dq);", "const double ds = p * dp;"),
    ("bwd_ds_sign", "const double ds = p * (dp - Dq);", "const double ds = p * (Dq - dp);"),
    ("bwd_dk_without_scale", "dkb[kk * (long)Hkv * D + d] += scale * ds * (double)qrow[d];",
     "dkb[kk * (long)Hkv * D + d] += ds * (double)qrow[d];"),
    ("bwd_dq_uses_query", "dqrow[d] += scale * ds * (double)krow[d];",
     "dqrow[d] += scale * ds * (double)qrow[d];"),
    ("bwd_dv_uses_ds", "+= p * (double)dorow[j];", "+= ds * (double)dorow[j];"),
    ("bwd_p_unshifted", "const double p = exp(scale * acc - lse);",
     "const double p = exp(scale * acc);"),
    ("bwd_one_head_per_group", "for (int h = kh * G; h < (kh + 1) * G; ++h)",
     "for (int h = kh * G; h < kh * G + 1; ++h)"),
    ("bwd_last_key_dropped", "for (long kk = lo; kk <= hi; ++kk) {",
     "for (long kk = lo; kk < hi; ++kk) {"),
    ("bwd_rowterm_uses_v", "for (int j = 0; j < Dv; ++j) Dq += (double)dorow[j] * orow[j];",
     "for (int j = 0; j < Dv; ++j) Dq += (double)dorow[j] * vb[j];"),
    # sampled backward (rows of dQ, key blocks of dK / dV)
    ("bwd_sampled_key_head", "const int h = kkh * G + (int)(t / Qb), qi = (int)(t % Qb);",
     "const int h = kkh + (int)(t / Qb), qi = (int)(t % Qb);"),
    ("bwd_sampled_row_term", "const double ds = exp(scale * acc - lse) * (dp - Dq);",
     "const double ds = exp(scale * acc - lse) * dp;"),
    # the arbitrary (boolean) mask
    ("allow_ignored", "if (allow_row[k] != 0) keys[n++] = k;", "keys[n++] = k;"),
    ("allow_inverted", "if (allow_row[k] != 0) keys[n++] = k;", "if (allow_row[k] == 0) keys[n++] = k;"),
    ("allow_kv_head", "const int hm = Hm == 1 ? 0 : h;", "const int hm = Hm == 1 ? 0 : kh;"),
    ("allow_batch_dropped", "allow + (((long)b * Hm + hm) * Q + qi) * (long)K;",
     "allow + (((long)0 * Hm + hm) * Q + qi) * (long)K;"),
    ("allow_row_shifted", "allow + (((long)b * Hm + hm) * Q + qi) * (long)K;",
     "allow + (((long)b * Hm + hm) * Q + (qi + 1 < Qb ? qi + 1 : qi)) * (long)K;"),
    ("allow_ignores_range", "    legal_keys(q, Qb, Kb, window, mask, &lo, &hi);\n    long n = 0;",
     "    legal_keys(q, Qb, Kb, window, mask, &lo, &hi);\n    lo = 0;\n    hi = (long)Kb - 1;\n    long n = 0;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert old in src, f"mutation site for {name} not found"
    path = os.path.join(tmp_path, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    lib = oracle.OracleLib(oracle.build(force=True, src=path,
                                        out=os.path.join(tmp_path, f"mut_{name}.so")))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
