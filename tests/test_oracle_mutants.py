"""Plant plausible mistakes in copies of the oracle (CPU only) and require that
every one of them fails at least one pin.  This is evidence that the pins in
pins.py constrain each part of the oracle, not only that the oracle passes them."""
import os
import types

import pytest

import pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "dsa_oracle.py")

MUTANTS = {
    "relu_dropped": ("relu = np.maximum(s, 0.0)", "relu = s"),
    "relu_after_weighting": ("out[r, :visible] = w[t] @ relu",
                             "out[r, :visible] = np.maximum(w[t] @ s, 0.0)"),
    "head_dropped": ("out[r, :visible] = w[t] @ relu", "out[r, :visible] = w[t][:-1] @ relu[:-1]"),
    "causal_off_by_one": ("(L - next_n + i + 1)", "(L - next_n + i)"),
    "page_offset": ("blocks * block_size + j % block_size", "blocks * block_size + j // block_size"),
    "seq_index": ("b, i = divmod(int(t), next_n)", "i, b = divmod(int(t), next_n)"),
    "k_scale_rows": ("np.asarray(k_scale)[kr]", "np.asarray(k_scale)[:L]"),
    "row_scale_dropped": ("return v * np.asarray(scale, dtype=np.float64)[..., None]", "return v"),
    "e4m3_bias": ("np.exp2((e - 7)", "np.exp2((e - 8)"),
    "e4m3_subnormal": ("(m / 8.0) * 2.0**-6", "(m / 8.0) * 2.0**-7"),
    "tie_order": ("np.lexsort((cand, -v))", "np.lexsort((-cand, -v))"),
    "neg_inf_selected": ("cand = np.nonzero(row != NEG_INF)[0]", "cand = np.arange(row.size)"),
    "no_zero_canon": ("row = x[r] + 0.0", "row = np.where(np.signbit(x[r]) & (x[r] == 0), -1e-300, x[r])"),
    "nibble_order": ("nib[:, 0::2] = fp4_rows & 0xF\n    nib[:, 1::2] = fp4_rows >> 4",
                     "nib[:, 0::2] = fp4_rows >> 4\n    nib[:, 1::2] = fp4_rows & 0xF"),
    "e2m1_table": ("(0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)", "(0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0, 3.5)"),
    "e2m1_sign": ("np.where((n & 8) != 0, -mag, mag)", "np.where((n & 4) != 0, -mag, mag)"),
    "e8m0_ff": ("np.where(b == 0xFF, 0.0,", "np.where(b == 0x100, 0.0,"),
    "e8m0_bias": ("(b - 127).astype(np.int32)", "(b - 128).astype(np.int32)"),
    "scale_group": ("np.repeat(sc, 32, axis=1)", "np.tile(sc, (1, 32))"),
    "bf16_truncate": ("(u + np.uint64(0x7FFF) + keep)", "(u)"),
    "padded_not_zero": ("live = sel >= 0", "live = sel >= -1"),
    "gather_seq_row": ("[b[live], pos // block_size]", "[0 * b[live], pos // block_size]"),
    "gather_offset": ("off = pos % block_size", "off = pos // block_size % block_size"),
    "key_dtype_ignored": ("dequantize(np.asarray(k_data)[kr], ks, k_dtype or dtype)",
                          "dequantize(np.asarray(k_data)[kr], ks, dtype)"),
    "mxfp4_key_scale_ignored": ("return mxfp4_dequant(data, scale)",
                                "return mxfp4_dequant(data, np.full_like(scale, 127))"),
}


def _mutant(name):
    src = open(ORACLE_SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    mod = _mutant(name)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(mod)
        except Exception:          # an assertion or a crash both expose the mistake
            failed.append(check.__name__)
    assert failed, f"mutant {name} passes every pin"
