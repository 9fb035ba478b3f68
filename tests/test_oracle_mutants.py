"""The oracle's pins have teeth: plant plausible mistakes in a temporary copy
of the C oracle and check that every mutant fails at least one pin.

Only in-bounds mutations are planted (each one keeps every array index inside
its buffer), so a mutant can give wrong numbers but cannot crash the test.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import na3d_inputs
from test_oracle import brute_dense, f64

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "na3d_oracle.c")

MUTANTS = {
    "start_off_by_one": ("int64_t s = i - K / 2;", "int64_t s = i - K / 2 + 1;"),
    "window_drops_last_frame": ("kt < st + P->KT; ++kt)\n        for (int64_t kh = sh; kh < sh + P->KH; ++kh)\n            for (int64_t kw = sw; kw < sw + P->KW; ++kw, ++j) {\n                const int64_t tok = ((b * P->T + kt) * P->H + kh) * P->W + kw;\n                const uint16_t* krow",
                                "kt < st + P->KT - (P->KT > 1); ++kt)\n        for (int64_t kh = sh; kh < sh + P->KH; ++kh)\n            for (int64_t kw = sw; kw < sw + P->KW; ++kw, ++j) {\n                const int64_t tok = ((b * P->T + kt) * P->H + kh) * P->W + kw;\n                const uint16_t* krow"),
    "reversed_k_operand": ("acc += qd[d] * bf16_to_f64(krow[d]);",
                           "acc += qd[d] * bf16_to_f64(krow[HD - 1 - d]);"),
    "wrong_head_for_k": ("const uint16_t* krow = P->k + (tok * NH + n) * HD;",
                         "const uint16_t* krow = P->k + (tok * NH + (NH - 1 - n)) * HD;"),
    "batch_zero_for_v": ("const int64_t tok = ((b * P->T + kt) * P->H + kh) * P->W + kw;\n                const uint16_t* vrow",
                         "const int64_t tok = ((0 * P->T + kt) * P->H + kh) * P->W + kw;\n                const uint16_t* vrow"),
    "k_instead_of_v": ("const uint16_t* vrow = P->v +", "const uint16_t* vrow = P->k +"),
    "halved_exponent": ("x[i] = exp(x[i] - xmax);", "x[i] = exp(0.5 * (x[i] - xmax));"),
    "mean_normaliser": ("denom += x[i];", "denom += 1.0;"),
}


def build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O1", "-shared", "-fPIC", "-o", str(so), str(path), "-lm"])
    lib = ctypes.CDLL(str(so))
    I64, P = ctypes.c_int64, ctypes.c_void_p
    lib.na3d_oracle_fwd.argtypes = [P, P, P, P] + [I64] * 9 + [ctypes.c_int]
    lib.na3d_oracle_fwd.restype = ctypes.c_int

    def fwd(q, k, v, kernel):
        out = np.empty(q.shape, dtype=np.float64)
        rc = lib.na3d_oracle_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, out.ctypes.data,
                                 *q.shape, *kernel, 1)
        assert rc == 0
        return out
    return fwd


def pins_pass(fwd):
    """Return True if the candidate oracle passes every pin below."""
    checks = []
    for shape, kernel in [((2, 3, 5, 7, 2, 16), (3, 3, 5)), ((1, 5, 6, 9, 1, 16), (5, 1, 3))]:
        q, k, v = na3d_inputs.make_qkv(*shape, seed=11)
        checks.append(np.allclose(fwd(q, k, v, kernel), brute_dense(q, k, v, kernel),
                                  rtol=1e-11, atol=1e-12))
    B, T, H, W, NH, HD = shape = (2, 3, 4, 5, 2, 16)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=2)

    def heads(x):
        return torch.from_numpy(f64(x)).permute(0, 4, 1, 2, 3, 5).reshape(B, NH, -1, HD)
    ref = torch.nn.functional.scaled_dot_product_attention(heads(q), heads(k), heads(v), scale=1.0)
    ref = ref.reshape(B, NH, T, H, W, HD).permute(0, 2, 3, 4, 1, 5).numpy()
    checks.append(np.allclose(fwd(q, k, v, (T, H, W)), ref, rtol=1e-11, atol=1e-12))
    return all(checks)


def test_unmutated_copy_passes(tmp_path):
    MUTANTS["identity"] = ("denom += x[i];", "denom += x[i];")
    try:
        assert pins_pass(build_mutant(tmp_path, "identity"))
    finally:
        del MUTANTS["identity"]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(tmp_path, name):
    assert not pins_pass(build_mutant(tmp_path, name))
