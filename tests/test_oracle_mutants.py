"""Plant plausible mistakes in copies of the oracle's source (CPU only) and
check that at least one pin catches each."""

import os
import shutil
import subprocess

import pytest

import oracle
import pins

# (name, original text, planted mistake)
MUTANTS = [
    ("eps dropped", "acc / d + eps", "acc / d"),
    ("rms over N", "acc / d + eps", "acc / N + eps"),
    ("no sqrt", "1.0 / std::sqrt(acc / d + eps)", "1.0 / (acc / d + eps)"),
    ("w_norm dropped", " *\n                     static_cast<double>(w_norm[i]);", ";"),
    ("rs of stream 0", "rs[t * n + s] * stream_sum", "rs[t * n] * stream_sum"),
    ("W_down transposed", "W_down[(size_t)k * N + i]", "W_down[(size_t)i * K + k]"),
    ("W_up transposed", "W_up[(size_t)i * K + k]", "W_up[(size_t)k * N + i]"),
    ("sigmoid sign", "std::exp(-g)", "std::exp(g)"),
    ("mean over d", "acc / n;", "acc / d;"),
    ("pending ignored", "r + p", "r"),
    ("pending subtracted", "r + p", "r - p"),
    ("epilogue on R", "hc_oracle_epilogue(n, d, T, r_out,", "hc_oracle_epilogue(n, d, T, R,"),
    ("norm on R", "hc_oracle_rms(n, d, T, eps, r_out,", "hc_oracle_rms(n, d, T, eps, R,"),
    ("rms stride", "r_prime[(size_t)t * N + (size_t)s * d + c];", "r_prime[(size_t)t * N + (size_t)c * n + s];"),
    ("gate dropped", "sig * u[", "u["),
    ("lo token stride", "lo[(size_t)t * K + k] = total", "lo[(size_t)k * T + t] = total"),
    ("mean token stride", "mean[(size_t)t * d + c]", "mean[(size_t)c * T + t]"),
    ("x squared", "acc += v * v;", "acc += v;"),
    ("bf16 widening", "<< 16;", "<< 15;"),
    ("q8 scale block", "+ j / 32]", "+ j / 16]"),
    ("q8 scale row stride", "scale[(size_t)r * (cols / 32)", "scale[(size_t)r * (cols / 16)"),
    ("q8 quant transposed", "q[(size_t)r * cols + j]", "q[(size_t)j * cols + r]"),
    ("q8 scale dropped", "return half_to_double(scale[(size_t)r * (cols / 32) + j / 32]) *", "return"),
    ("half exponent bias", "exponent - 25", "exponent - 24"),
    ("half subnormal scale", "fraction), -24)", "fraction), -25)"),
    ("half implicit bit", "1024 + fraction", "fraction"),
    ("half sign", "return sign ? -v : v;", "return v;"),
    ("q2 offset", "static_cast<double>(q - 2)", "static_cast<double>(q - 1)"),
    ("q2 bit order", "(byte >> (2 * (j % 4))) & 3", "(byte >> (6 - 2 * (j % 4))) & 3"),
    ("q2 two-bit mask", "(2 * (j % 4))) & 3;", "(2 * (j % 4))) & 1;"),
    ("q2 block size", "+ j / 64]", "+ j / 32]"),
    ("q2 scale row stride", "scale[(size_t)r * (cols / 64)", "scale[(size_t)r * (cols / 32)"),
    ("q2 code row stride", "codes[(size_t)r * (cols / 4)", "codes[(size_t)r * (cols / 2)"),
    ("q2 input stride", "x[(size_t)c * cols + j]", "x[(size_t)j * ncols + c]"),
    ("q2 output stride", "y[(size_t)c * rows + r]", "y[(size_t)r * ncols + c]"),
    ("q2 scale dropped", "return half_to_double(scale[(size_t)r * (cols / 64) + j / 64]) *", "return"),
    ("q8 down on bf16 path", "hc_oracle_down_q8(n, d, K, T, r_out, w_norm, Wd_q, Wd_scale, rs, lo);", "hc_oracle_down_q8(n, d, K, T, r_out, w_norm, Wd_q, Wu_scale, rs, lo);"),
]


@pytest.fixture(scope="module")
def src():
    with open(oracle.SRC) as f:
        return f.read()


def test_mutants_are_applicable(src):
    for name, old, _ in MUTANTS:
        assert src.count(old) >= 1, f"mutation anchor missing: {name}"


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_caught(tmp_path, src, name, old, new):
    mutated = src.replace(old, new, 1)
    assert mutated != src
    path = os.path.join(tmp_path, "mutant.cpp")
    with open(path, "w") as f:
        f.write(mutated)
    lib = os.path.join(tmp_path, "libmutant.so")
    subprocess.run(oracle.compile_cmd(path, lib), check=True)
    failed = pins.failing_pins(oracle.Oracle(lib))
    assert failed, f"no pin caught the planted mistake '{name}'"
