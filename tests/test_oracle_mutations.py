"""Plant one plausible mistake at a time in a copy of the oracle (on the
CPU) and check that the pins catch every one of them."""
import pytest

import oracle
import pins

# (id, text in fvif_oracle.c, replacement, pins expected to notice)
MUTATIONS = [
    ("edge_repeat_mirror", "j = 2 * (n - 1) - j;", "j = 2 * n - 1 - j;",
     [pins.pin_mirror_table]),
    ("no_reflect_below", "        j = -j;\n", "        j = 0;\n",
     [pins.pin_mirror_table, pins.pin_filter_brute]),
    ("dropped_last_tap", "for (int k = 0; k < n; ++k) {\n                int jj",
     "for (int k = 0; k < n - 1; ++k) {\n                int jj",
     [pins.pin_filter_brute]),
    ("transposed_vertical_index", "int ii = fvo_mirror(i + k - r, h);",
     "int ii = fvo_mirror(i - k + r - 1, h);", [pins.pin_filter_brute]),
    ("odd_decimation_phase", "f[(size_t)(2 * y) * w + 2 * x]",
     "f[(size_t)(2 * y) * w + 2 * x + 1]", [pins.pin_decimate_brute]),
    ("sigma_from_width", "double sigma = ks * base / 5.0;",
     "double sigma = ks * (2.0 * half + 1.0) / 5.0;",
     [pins.pin_taps_gaussian]),
    ("unnormalised_taps", "taps[k] = (float)(w[k] / sum);",
     "taps[k] = (float)(w[k] / (sum * 1.0001));",
     [pins.pin_taps_symmetric_normalised]),
    ("wrong_sign_sigma12", "float s12 = xy - mu1 * mu2;",
     "float s12 = xy + mu1 * mu2;", [pins.pin_terms_closed_forms]),
    ("nsq_in_fp32", "double d = (double)sv + nsq;",
     "double d = (double)sv + (double)(float)nsq;",
     [pins.pin_num_exact_sequence_random]),
    ("den_in_fp32", "double q2 = (double)s1 / nsq;",
     "double q2 = (double)(s1 / (float)nsq);",
     [pins.pin_terms_exact_sequence_random,
      pins.pin_terms_rounded_once_from_fp64]),
    ("gain_cap_missing", "g = g < gain_limit ? g : gain_limit;", "",
     [pins.pin_terms_closed_forms]),
    ("negative_gain_kept", "if (g < 0.0f) {", "if (g < -1.0e30f) {",
     [pins.pin_terms_closed_forms]),
    ("lowvar_constant", "(float)(4.0 / (255.0 * 255.0))",
     "(float)(4.0 / 255.0)", [pins.pin_terms_closed_forms,
                              pins.pin_flat_ref_closed_form]),
    ("branch_in_fp32", "if ((double)s1 < nsq) {", "if (s1 < (float)nsq) {",
     [pins.pin_branch_is_fp64_compare]),
    ("log2_coefficient", "const float c5 = 1.0f / 5.0f;",
     "const float c5 = 1.0f / 6.0f;", [pins.pin_log2_error_bound]),
    ("log2_no_range_fold", "if (m > sqrt2) {", "if (m > 2.5f) {",
     [pins.pin_log2_error_bound]),
    ("ingest_10bit_halved", "float scaler = (float)(1 << (bd - 8));",
     "float scaler = (float)(1 << (bd - 9));", [pins.pin_ingest]),
    ("rows_summed_twice", "total_num = total_num + row_num;",
     "total_num = total_num + row_num + row_num;",
     [pins.pin_sum_order, pins.pin_identical_frames]),
    ("num_den_swapped_in_score",
     "scores[s] = (double)total_num / (double)total_den;",
     "scores[s] = (double)total_den / (double)total_num;",
     [pins.pin_textbook_vif, pins.pin_sum_order]),
    ("row_sum_right_to_left", "for (int j = 0; j < ws; ++j) {",
     "for (int j = ws - 1; j >= 0; --j) {",
     [pins.pin_row_sums_left_to_right]),
    ("decimate_with_own_scale_taps", "fvo_decimate(x, ws, hs, taps[s + 1], ntaps[s + 1], nx);",
     "fvo_decimate(x, ws, hs, taps[s], ntaps[s], nx);",
     [pins.pin_textbook_vif]),
]


@pytest.mark.parametrize("mid,old,new,catchers", MUTATIONS,
                         ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(mid, old, new, catchers):
    src = oracle.source_text()
    assert src.count(old) == 1, "mutation anchor not found once: %s" % mid
    L = oracle.build_variant(src.replace(old, new), mid)
    caught = []
    for pin in catchers:
        try:
            pin(L)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "no pin noticed the planted mistake %s" % mid


import ssim_pins  # noqa: E402

# (id, text in fssim_oracle.c, replacement, pins expected to notice)
SSIM_MUTATIONS = [
    ("odd_kernel_offsets", "const int hi = k / 2 - ((k % 2 == 0) ? 1 : 0);",
     "const int hi = k / 2;", [ssim_pins.pin_exact_window_sum,
                               ssim_pins.pin_constant_plane]),
    ("mirror_without_edge_repeat", "return r >= n ? p - 1 - r : r;",
     "return r >= n ? (p - 2 - r < 0 ? 0 : p - 2 - r) : r;",
     [ssim_pins.pin_mirror_reflection]),
    ("float_window_sum", "    double sum = 0.0;\n    for (int dy",
     "    float sum = 0.0f;\n    for (int dy", [ssim_pins.pin_exact_window_sum]),
    ("product_not_rounded", "const float prod = img[(size_t)yy * w + xx] * tap;",
     "const double prod = (double)img[(size_t)yy * w + xx] * tap;",
     [ssim_pins.pin_exact_window_sum, ssim_pins.pin_constant_plane]),
    ("size_without_odd_column", "*sw = w / scale + (w & 1);",
     "*sw = w / scale;", [ssim_pins.pin_out_sizes]),
    ("tap_one_over_k", "return 1.0f / (float)(scale * scale);",
     "return 1.0f / (float)scale;", [ssim_pins.pin_tap]),
    ("auto_scale_truncated", "(int)round((double)m / 256.0);",
     "m / 256;", [ssim_pins.pin_auto_scale_rounding]),
    ("centre_off_by_one", "filter_pixel(img, w, h, x * scale, y * scale,",
     "filter_pixel(img, w, h, x * scale + 1, y * scale,",
     [ssim_pins.pin_power_of_two_closed_form,
      ssim_pins.pin_exact_window_sum]),
    ("sixteen_bit_divisor", "const float div = (float)(1 << (bitdepth - 8));",
     "const float div = (float)(1 << (bitdepth - 9));",
     [ssim_pins.pin_scale_one_is_sample_conversion]),
]


@pytest.mark.parametrize("mid,old,new,catchers", SSIM_MUTATIONS,
                         ids=[m[0] for m in SSIM_MUTATIONS])
def test_planted_ssim_mistake_is_caught(mid, old, new, catchers):
    src = oracle.ssim_source()
    assert src.count(old) == 1, "mutation anchor not found once: %s" % mid
    L = oracle.build_variant(oracle.source_text(), "ssim_" + mid,
                             src.replace(old, new))
    caught = []
    for pin in catchers:
        try:
            pin(L)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "no pin noticed the planted mistake %s" % mid
