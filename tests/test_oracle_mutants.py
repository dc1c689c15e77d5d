"""Planted-mistake check of the oracle pins (CPU only).

Each mutant is a copy of the oracle source with one plausible mistake (a
dropped term, a wrong sign or index, a transposed operand, a wrong rounding).
It is compiled into a temporary library and every pin is run against it; at
least one pin must fail, otherwise the pins would not notice that mistake.
"""

import importlib.util
import os
import subprocess
import tempfile

import pytest

import calib_pins
import oracle_pins
from oracle import oracle as O

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "oscar_oracle.cpp")
CALIB_SRC = os.path.join(os.path.dirname(SRC), "calibration.py")

# (name, text in the oracle, replacement, expected number of occurrences)
MUTANTS = [
    ("rotation_transposed",
     "x[i] * static_cast<double>(R[static_cast<size_t>(i) * D + j])",
     "x[i] * static_cast<double>(R[static_cast<size_t>(j) * D + i])", 1),
    ("clip_lower_bound_dropped", "    if (x[j] < -c) x[j] = -c;\n", "", 1),
    ("scale_divisor_4", "(mx - mn) / 3.0", "(mx - mn) / 4.0", 1),
    ("zero_is_max", "const float z32 = static_cast<float>(mn);", "const float z32 = static_cast<float>(mx);", 1),
    ("code_floor_not_rint", "double c = std::nearbyint(u);", "double c = std::floor(u);", 1),
    ("packing_reversed_in_byte", "(c << (2 * (j % 4)))", "(c << (2 * (3 - j % 4)))", 1),
    ("unrotation_not_transposed",
     "acc_rot[j] * static_cast<double>(R_v[static_cast<size_t>(c) * D + j])",
     "acc_rot[j] * static_cast<double>(R_v[static_cast<size_t>(j) * D + c])", 1),
    ("window_ring_index", "* W + (p % W);", "* W + (p - win_begin);", 2),
    ("gqa_mapping_modulo", "const int h = hq / gqa;", "const int h = hq % H;", 2),
    ("dequant_drops_zero", "x[j] = c * s + z;", "x[j] = c * s;", 1),
    ("f16_truncates", "std::nearbyint(a / quantum) * quantum", "std::trunc(a / quantum) * quantum", 1),
    ("default_scale_1_over_D", "sm_scale = 1.0 / std::sqrt(static_cast<double>(D));", "sm_scale = 1.0 / D;", 3),
    ("key_reads_value_codes", "page, h, 0, p % P, kk);", "page, h, 1, p % P, kk);", 1),
    ("softmax_denominator_counts_tokens", "    denom += w;\n", "    denom += 1.0;\n", 1),
    ("query_rotation_transposed",
     "qv[i] * static_cast<double>(Rk[static_cast<size_t>(i) * D + j])",
     "qv[i] * static_cast<double>(Rk[static_cast<size_t>(j) * D + i])", 1),
    ("all_groups_use_group0", "orc_group_params(G, y.data() + g * G, &s_bits, &z_bits);",
     "orc_group_params(G, y.data(), &s_bits, &z_bits);", 1),
    ("scale_zero_swapped", "sz[2 * g + 0] = s_bits;\n          sz[2 * g + 1] = z_bits;",
     "sz[2 * g + 0] = z_bits;\n          sz[2 * g + 1] = s_bits;", 1),
    ("bulk_offset_uses_page_index", "orc_dequant_row(d, int2_pages, scale_zero_pages, page, h, 1, p % P, vv);",
     "orc_dequant_row(d, int2_pages, scale_zero_pages, page, h, 1, (p / P) % P, vv);", 1),
    ("mixed_kv_swapped", "const uint16_t* x = (kv ? v : k) + (static_cast<size_t>(t) * H + h) * D;\n        uint16_t* dst",
     "const uint16_t* x = (kv ? k : v) + (static_cast<size_t>(t) * H + h) * D;\n        uint16_t* dst", 1),
    ("mixed_window_skips_oldest", "} else if (W > 0 && p >= win_begin) {", "} else if (W > 0 && p > win_begin) {", 1),
    ("extend_not_causal", "hq, b, L, pos + 1, R_k", "hq, b, L, L, R_k", 1),
    ("extend_excludes_own_position", "hq, b, L, pos + 1, R_k", "hq, b, L, pos, R_k", 1),
    ("extend_window_of_prefix_length", "const int win_begin = (L - W > S) ? L - W : S;\n  for (int p = 0; p < A; ++p)",
     "const int win_begin = (A - W > S) ? A - W : S;\n  for (int p = 0; p < A; ++p)", 1),
    ("key_offset_added", "orc_bf16_to_f64(k_bf16[i]) - static_cast<double>(c[i])",
     "orc_bf16_to_f64(k_bf16[i]) + static_cast<double>(c[i])", 1),
    ("key_offset_not_rounded_to_f32",
     "out[i] = static_cast<double>(static_cast<float>(orc_bf16_to_f64(k_bf16[i]) - static_cast<double>(c[i])));",
     "out[i] = orc_bf16_to_f64(k_bf16[i]) - static_cast<double>(c[i]);", 1),
    ("key_offset_on_values_too", "if (kv == 0 && offset_k != nullptr) {\n    orc_offset_key",
     "if (offset_k != nullptr) {\n    orc_offset_key", 1),
    ("key_offset_of_head0_for_all", "orc_offset_key(D, x, offset_k + static_cast<size_t>(h) * D, out);",
     "orc_offset_key(D, x, offset_k, out);", 1),
    ("mixed_key_row_not_offset", "if (kv == 0 && offset_k != nullptr) {  // the stored key",
     "if (false) {  // the stored key", 1),
    ("bf16_rounding_truncates", "u += 0x7fffu + lsb;", "u += 0u * lsb;", 1),
    ("extend_row_as_sequence", "const int b = row_seq[r];", "const int b = r < batch ? r : row_seq[r];", 1),
]


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory(prefix="oracle_mutants_") as d:
        yield d


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, count, workdir):
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == count, f"mutation site for {name} not found {count} time(s)"
    path = os.path.join(workdir, f"{name}.cpp")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib_path = os.path.join(workdir, f"lib{name}.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-ffp-contract=off", "-shared", "-fPIC", path, "-o", lib_path],
                   check=True)
    lib = O.load(lib_path)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
            break
    assert caught, f"no pin catches the planted mistake '{name}'"


# Planted mistakes in the calibration oracle (numpy source); same rule: some pin must fail.
CALIB_MUTANTS = [
    ("mean_not_subtracted", "            xh = xh - mu\n", "            xh = xh\n", 1),
    ("divides_by_n_minus_1", "C[h] = (xh.T @ xh) / N", "C[h] = (xh.T @ xh) / (N - 1)", 1),
    ("heads_mixed", "xh = x[:, h, :]", "xh = x[:, 0, :]", 1),
    ("ascending_eigenvalues", 'order = np.argsort(-w, kind="stable")', 'order = np.argsort(w, kind="stable")', 1),
    ("eigenvectors_reordered_by_row", "w, V = w[order], V[:, order]", "w, V = w[order], V[order, :]", 1),
    ("rotation_rows_not_columns", "R[h] = V\n", "R[h] = V.T\n", 1),
    ("sign_rule_negative", "if col[i_big] < 0:", "if col[i_big] > 0:", 1),
    ("sign_rule_last_index", "i_big = int(np.argmax(np.abs(col)))",
     "i_big = int(len(col) - 1 - np.argmax(np.abs(col[::-1])))", 1),
    ("quantile_floor", "k = int(math.ceil(float(q) * float(N)))", "k = int(math.floor(float(q) * float(N)))", 1),
    ("quantile_one_rank_high", "clip[h] = np.sort(y, axis=0)[k - 1]", "clip[h] = np.sort(y, axis=0)[min(k, N - 1)]", 1),
    ("clip_without_magnitude", "y = np.abs(x[:, h, :] @ np.asarray(R[h], dtype=np.float64))",
     "y = (x[:, h, :] @ np.asarray(R[h], dtype=np.float64))", 1),
    ("clip_of_unrotated_samples", "y = np.abs(x[:, h, :] @ np.asarray(R[h], dtype=np.float64))",
     "y = np.abs(x[:, h, :])", 1),
]


@pytest.mark.parametrize("name,old,new,count", CALIB_MUTANTS, ids=[m[0] for m in CALIB_MUTANTS])
def test_calibration_mutant_is_caught(name, old, new, count, workdir):
    with open(CALIB_SRC) as f:
        src = f.read()
    assert src.count(old) == count, f"mutation site for {name} not found {count} time(s)"
    path = os.path.join(workdir, f"calib_{name}.py")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"calib_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = []
    for pin in calib_pins.ALL_PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
            break
    assert caught, f"no pin catches the planted mistake '{name}'"
