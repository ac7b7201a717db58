"""The oracle's pins are strong enough to catch plausible mistakes.

Each case copies oracle.cpp, plants one mistake of the kind an implementation
plausibly makes (a dropped term, a wrong sign, index or tie rule, a transposed
nibble order, a softmax sign or normaliser), builds the copy on the CPU and runs the pin tests against it in
a child process. Every mutant must fail at least one pin.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTANTS = {
    "e2m1_ties_to_odd": ("((i + 1) % 2 == 0)", "((i + 1) % 2 == 1)"),
    "sign_dropped": ("if (k != 0 && x < 0.0f) k |= 8;", ""),
    "nibbles_swapped": ("c[0] | (c[1] << 4)", "c[1] | (c[0] << 4)"),
    "scale_divisor": ("amax / 6.0f", "amax / 4.0f"),
    "e4m3_truncates": ("return std::fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;", "return fl;"),
    "relu_dropped": ("s += w[h] * std::max(0.0, d);", "s += w[h] * d;"),
    "head_weight_index": ("s += w[h] * std::max(0.0, d);", "s += w[(h + 1) % heads] * std::max(0.0, d);"),
    "topk_ties_high_index": ("return s[a] > s[b] || (s[a] == s[b] && a < b);",
                             "return s[a] > s[b] || (s[a] == s[b] && a > b);"),
    "reindex_not_causal": ("if (p <= t) cand.push_back(p);", "cand.push_back(p);"),
    "window_ring_off_by_one": ("n_ctx - window}", "n_ctx - window - 1}"),
    "attention_no_scale": ("logit[i] = tau * d;", "logit[i] = d;"),
    "block_max_shifted": ("for (int64_t p = b * block; p < std::min<int64_t>(n, (b + 1) * block); ++p)",
                          "for (int64_t p = b * block + 1; p < std::min<int64_t>(n, (b + 1) * block); ++p)"),
    "compress_logit_sign": ("const double w = std::exp(static_cast<double>(bf16_value(z[(e * m + i) * dim + c])) - zmax);",
                            "const double w = std::exp(zmax - static_cast<double>(bf16_value(z[(e * m + i) * dim + c])));"),
    "compress_unnormalised": ("out[e * dim + c] = bf16_round(num / den);", "out[e * dim + c] = bf16_round(num);"),
    "compress_ties_away": ("double r = std::nearbyint(std::ldexp(a, -q_exp));",
                           "double r = std::round(std::ldexp(a, -q_exp));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mut = tmp_path / "oracle_mut.cpp"
    mut.write_text(src.replace(old, new, 1))
    lib = tmp_path / "oracle_mut.so"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                           str(mut), "-o", str(lib), "-lpthread"])
    env = dict(os.environ, CSA2_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_formats.py"),
                        os.path.join(ROOT, "tests", "test_oracle_indexer.py"),
                        os.path.join(ROOT, "tests", "test_oracle_attention.py"),
                        os.path.join(ROOT, "tests", "test_oracle_compress.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
