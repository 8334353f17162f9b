"""Plant plausible mistakes in copies of the C++ oracle (CPU only) and require that
every one of them fails at least one pin.  This is evidence that the pins in pins.py
constrain each part of the oracle, not only that the oracle passes them.  Each mutant is
the oracle's source with one edit, compiled on its own."""
import concurrent.futures as cf
import os
import tempfile

import pytest

import pins
from oracle import dsa_oracle

MUTANTS = {
    "relu_dropped": ("const double relu = s > 0.0 ? s : 0.0;", "const double relu = s;"),
    "relu_after_weighting": ("*dst = logit + 0.0;     // -0.0 + 0.0 == +0.0",
                             "*dst = 0.0;\n      { double z = 0.0; for (int h = 0; h < H; ++h) { double s = 0.0;"
                             " for (int d = 0; d < D; ++d) s += qv[static_cast<size_t>(h) * D + d] * kv[d];"
                             " z += weights[t * H + h] * s; } *dst = (z > 0.0 ? z : 0.0) + 0.0; }"),
    "head_dropped": ("for (int h = 0; h < H; ++h) {\n        double s = 0.0;",
                     "for (int h = 0; h < H - 1; ++h) {\n        double s = 0.0;"),
    "causal_off_by_one": ("(L - next_n + i + 1)", "(L - next_n + i)"),
    "page_offset": ("row = blk * block_size + j % block_size;", "row = blk * block_size + j / block_size;"),
    "seq_index": ("const int64_t b = t / next_n, i = t % next_n;", "const int64_t b = t % next_n, i = t / next_n;"),
    "k_scale_rows": ("static_cast<const double*>(k_scale)[row];", "static_cast<const double*>(k_scale)[j];"),
    "q_scale_dropped": ("* q_scale[t * H + h];", ";"),
    "e4m3_bias": ("std::ldexp(1.0, e - 7)", "std::ldexp(1.0, e - 8)"),
    "e4m3_subnormal": ("(m / 8.0) * std::ldexp(1.0, -6)", "(m / 8.0) * std::ldexp(1.0, -7)"),
    "bf16_shift": ("static_cast<uint32_t>(bits) << 16;", "static_cast<uint32_t>(bits) << 15;"),
    "tie_order": ("return a.second < b.second;", "return a.second > b.second;"),
    "neg_inf_selected": ("if (v == kNegInf || std::isnan(v)) continue;", "if (std::isnan(v)) continue;"),
    "no_zero_canon": ("cand.emplace_back(v + 0.0, j);",
                      "cand.emplace_back(std::signbit(v) && v == 0.0 ? -1e-300 : v, j);"),
    "short_row_not_padded": ("        idx[r * k + s] = -1;\n", "        idx[r * k + s] = 0;\n"),
    "nibble_order": ("(e % 2 == 0) ? (byte & 0xF) : (byte >> 4)", "(e % 2 == 0) ? (byte >> 4) : (byte & 0xF)"),
    "e2m1_table": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0, 3.5}"),
    "e2m1_sign": ("return (nibble & 8) ? -mag : mag;", "return (nibble & 4) ? -mag : mag;"),
    "e8m0_ff": ("b == 0xFF ? 0.0 :", "b == 0x100 ? 0.0 :"),
    "e8m0_bias": ("static_cast<int>(b) - 127", "static_cast<int>(b) - 128"),
    "scale_group": ("scale_row[e / 32]", "scale_row[e % 4]"),
    "bf16_truncate": ("(static_cast<uint64_t>(u) + 0x7FFFu + lsb) >> 16", "static_cast<uint64_t>(u) >> 16"),
    "padded_not_zero": ("if (pos < 0) {", "if (pos < -1) {"),
    "gather_seq_row": ("const int64_t blk = col < bt_stride ? block_table[b * bt_stride + col] : -1;",
                       "const int64_t blk = col < bt_stride ? block_table[0 * b * bt_stride + col] : -1;"),
    "gather_offset": ("const int64_t row = blk * block_size + pos % block_size;",
                      "const int64_t row = blk * block_size + pos / block_size % block_size;"),
    "key_kind_ignored": ("} else if (k_kind == kE4M3) {", "} else if (k_kind != kBF16) {"),
    "e4m3_ties_up": ("if (frac > 0.5 || (frac == 0.5 && std::fmod(r, 2.0) != 0.0)) r += 1.0;",
                     "if (frac >= 0.5) r += 1.0;"),
    "e4m3_no_saturation": ("  if (a > 448.0) a = 448.0;\n  double step;", "  double step;"),
    "e4m3_subnormal_step": ("step = std::ldexp(1.0, -9);", "step = std::ldexp(1.0, -10);"),
    "rope_pairs_split": ("const float x0 = y[2 * i], x1 = y[2 * i + 1];", "const float x0 = y[i], x1 = y[i + half];"),
    "rope_sin_sign": ("y[2 * i] = p0 - p1;", "y[2 * i] = p0 + p1;"),
    "q_fp8_max_fnuz": ("amax > 0.0f ? amax / 448.0f : 1.0f", "amax > 0.0f ? amax / 240.0f : 1.0f"),
    "hadamard_sign": ("__builtin_popcount(static_cast<unsigned>(i & j)) & 1", "__builtin_popcount(static_cast<unsigned>(i | j)) & 1"),
    "hadamard_unnormalised": ("y[i] = static_cast<float>(acc * norm);", "y[i] = static_cast<float>(acc);"),
    "mx_shared_exp": ("sexp = (e2 - 1) - 2;", "sexp = (e2 - 1) - 1;"),
    "e2m1_ties_odd": ("if (dc < db || (dc == db && (c & 1) == 0)) best = c;", "if (dc <= db) best = c;"),
    "writer_nibble_order": ("static_cast<uint8_t>(lo | (hi << 4));", "static_cast<uint8_t>(hi | (lo << 4));"),
    "attn_sink_dropped": ("double denom = std::exp(sink[h] - m);", "double denom = 0.0;"),
    "attn_scale_dropped": ("sc[j] = scale * dot;", "sc[j] = dot;"),
    "attn_padded_counted": ("      if (pos < 0) continue;\n      const int64_t page = pos / block_size;",
                            "      const int64_t page = (pos < 0 ? 0 : pos) / block_size;"),
    "attn_value_is_query": ("for (int e = 0; e < D; ++e) o[e] += p * x[(size_t)j * D + e];",
                            "for (int e = 0; e < D; ++e) o[e] += p * bf16_value(q[(t * H + h) * D + e]);"),
    "mxfp4_key_scale_row": ("static_cast<const uint8_t*>(k_scale) + row * (D / 32);",
                            "static_cast<const uint8_t*>(k_scale) + 0 * row * (D / 32);"),
}


@pytest.fixture(scope="module")
def mutant_libs():
    src = open(dsa_oracle.SOURCE).read()
    tmp = tempfile.mkdtemp(prefix="oracle_mutants_")

    def make(name):
        old, new = MUTANTS[name]
        assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
        path = os.path.join(tmp, f"{name}.cpp")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        return name, dsa_oracle.build(path, os.path.join(tmp, f"lib{name}.so"), opt="-O1")

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        return dict(ex.map(make, sorted(MUTANTS)))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, mutant_libs):
    mod = dsa_oracle.Oracle(mutant_libs[name])
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(mod)
        except Exception:          # an assertion or a crash both expose the mistake
            failed.append(check.__name__)
    assert failed, f"mutant {name} passes every pin"
