"""Plant plausible mistakes in copies of oracle.c (on the CPU) and check that the
pins catch every one: a pin set that a wrong oracle passes pins nothing."""
import os
import shutil

import pytest

import oracle as ora
import pins

SRC = os.path.join(os.path.dirname(ora.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
MUTATIONS = [
    ("scatter_sign_of_pad_dim0", "i0 * s[0] - p[0] + (int64_t)k0 * d[0]",
     "i0 * s[0] + p[0] + (int64_t)k0 * d[0]"),
    ("scatter_sign_of_pad_dim2", "i2 * s[2] - p[2] + (int64_t)k2 * d[2]",
     "i2 * s[2] + p[2] + (int64_t)k2 * d[2]"),
    ("flipped_taps_dim2", "wp[(k0 * k[1] + k1) * k[2] + k2]",
     "wp[(k0 * k[1] + k1) * k[2] + (k[2] - 1 - k2)]"),
    ("flipped_taps_dim1", "wp[(k0 * k[1] + k1) * k[2] + k2]",
     "wp[(k0 * k[1] + (k[1] - 1 - k1)) * k[2] + k2]"),
    ("weight_layout_transposed", "w + (ci * cout + co) * (int64_t)k[0] * k[1] * k[2]",
     "w + (co * cin + ci) * (int64_t)k[0] * k[1] * k[2]"),
    ("dilation_dropped", "i2 * s[2] - p[2] + (int64_t)k2 * d[2]",
     "i2 * s[2] - p[2] + (int64_t)k2"),
    ("stride_dropped_dim1", "i1 * s[1] - p[1] + (int64_t)k1 * d[1]",
     "i1 - p[1] + (int64_t)k1 * d[1]"),
    ("bias_dropped", "for (int64_t j = 0; j < osz; ++j) t[j] += bv;",
     "for (int64_t j = 0; j < osz; ++j) t[j] += 0.0 * bv;"),
    ("out_len_off_by_one", "(int64_t)d * (k - 1) + op + 1;", "(int64_t)d * (k - 1) + op;"),
    ("out_pad_ignored", "(int64_t)d * (k - 1) + op + 1;", "(int64_t)d * (k - 1) + 1;"),
    ("pool_len_floor_off_by_one", "n = span / s + 1;", "n = (span + 1) / s + 1;"),
    ("pool_divisor_swapped", "count_include_pad ? padded : inside",
     "count_include_pad ? inside : padded"),
    ("pool_window_shifted", "{a * s[0] - p[0], b * s[1] - p[1], c * s[2] - p[2]}",
     "{a * s[0] - p[0], b * s[1] - p[1], c * s[2] - p[2] + 1}"),
    ("pool_drops_last_tap", "for (int64_t q = st[2]; q < st[2] + k[2]; ++q)",
     "for (int64_t q = st[2]; q < st[2] + k[2] - 1; ++q)"),
    ("fused_scale1_dropped", "t[q] *= scale1;", "t[q] *= 1.0;"),
    ("fused_bias_after_scale2", "out[q] = (out[q] + bv) * scale2;",
     "out[q] = out[q] * scale2 + bv;"),
    ("fused_conv_bias_dropped", "convt_plane(x, in, w, conv_bias, cout,",
     "convt_plane(x, in, w, NULL, cout,"),
    ("fused_pool_stride_one", "avgpool_plane(t, O, pk, pk, pz, 1, P, out);",
     "avgpool_plane(t, O, pk, (const int[3]){1, 1, 1}, pz, 1, P, out);"),
    ("ceil_mode_no_trim", "if ((n - 1) * s >= L + p) n -= 1;", "if ((n - 1) * s > L + p) n -= 1;"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutant = tmp_path / "oracle_mut.c"
    mutant.write_text(src.replace(old, new, 1))
    lib = ora.build(force=True, src=str(mutant), out=str(tmp_path / "liboracle_mut.so"))
    be = ora.load(lib)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(be)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passes every pin"
