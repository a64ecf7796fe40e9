"""Pins of the CPU oracle to facts it does not compute itself.

The oracle (oracle/qgemm_oracle.c) is the fp64 definition of the groupwise
dequant-GEMM.  These tests check it against:

* hand-worked cases whose values were derived on paper (tests/golden/);
* exact rational arithmetic (Python integers/Fractions) from the codes as drawn,
  before packing, with numpy's own fp16/bf16 decoding -- the oracle's fp64
  result must lie within the recursive-summation error bound of the exact sum;
* brute force over every int4 byte and every int5 code at every bit offset,
  with the expected codes built by integer arithmetic in the test;
* numpy's float64 matmul on weights dequantised by the test;
* invariants the definition implies: linearity over disjoint supports,
  identity and permutation weights, power-of-two scaling, negated scales,
  int5 restricted to [-8, 7] equal to int4, column independence.

Each pin is a function of the loaded library so that ``test_planted_mistakes``
can re-run the whole set against copies of the oracle with one mistake
planted (a dropped term, a wrong sign extension, swapped nibbles, transposed
scales, ...) and confirm that some pin fails for every one of them.
"""
from __future__ import annotations

import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bit_weight_only_groupwise_gb300 import synth
from tests import golden_io

U = 2.0 ** -53


# ------------------------------------------------------------ independent decoding

def fp16_values(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def exact_gemm(codes, scales_bits, x_bits):
    """Exact Y and A as Fractions, from unpacked integer codes."""
    N, K = codes.shape
    T = x_bits.shape[0]
    s = fp16_values(scales_bits)
    x = bf16_values(x_bits)
    Y = [[None] * N for _ in range(T)]
    A = [[None] * N for _ in range(T)]
    for t in range(T):
        for n in range(N):
            acc = Fraction(0)
            mag = Fraction(0)
            for k in range(K):
                p = Fraction(float(x[t, k])) * Fraction(float(s[n, k // 64])) * int(codes[n, k])
                acc += p
                mag += abs(p)
            Y[t][n] = acc
            A[t][n] = mag
    return Y, A


def small_case(seed, N, K, T, bits):
    w = synth.weights(seed, N, K, bits)
    x = synth.activations(seed, T, K, outliers=True)
    return w, x


# ------------------------------------------------------------ the pins

def pin_golden(lib):
    for fname in ("int4_hand.txt", "int5_hand.txt"):
        for name, c in golden_io.load(fname).items():
            Y, A = oracle.gemm(c["bits"], c["packed"], c["scales"], c["x"], c["N"], c["K"], lib=lib)
            assert np.array_equal(Y, c["y"]), (fname, name, Y, c["y"])
            assert np.array_equal(A, c["a"]), (fname, name, A, c["a"])


def pin_exact_rational(lib):
    shapes = [(1, 2, 1, 4), (3, 8, 2, 5), (5, 64, 3, 4), (4, 100, 2, 5), (7, 128, 4, 4), (2, 192, 3, 5)]
    for seed, (N, K, T, bits) in enumerate(shapes):
        w, x = small_case(seed + 11, N, K, T, bits)
        Y, A = oracle.gemm(bits, w["packed"], w["scales"], x, N, K, lib=lib)
        Ye, Ae = exact_gemm(w["codes"], w["scales"], x)
        for t in range(T):
            for n in range(N):
                bound = K * U * float(Ae[t][n])
                assert abs(Fraction(float(Y[t, n])) - Ye[t][n]) <= Fraction(bound), (N, K, T, bits, t, n)
                assert abs(Fraction(float(A[t, n])) - Ae[t][n]) <= Fraction(bound), (N, K, T, bits, t, n)


def pin_bruteforce_int4(lib):
    # row b holds the single byte b: codes (low nibble, high nibble)
    packed = np.arange(256, dtype=np.uint8).reshape(256, 1)
    scales = np.full((256, 1), 0x3C00, np.uint16)
    x = np.array([[0x3F80, 0], [0, 0x3F80]], np.uint16)           # e_0, e_1
    Y, _ = oracle.gemm(4, packed, scales, x, 256, 2, lib=lib)
    b = np.arange(256, dtype=np.int32)
    lo = ((b << 4).astype(np.uint8).view(np.int8) >> 4).astype(np.float64)   # arithmetic shift
    hi = (b.astype(np.uint8).view(np.int8) >> 4).astype(np.float64)
    assert np.array_equal(Y[0], lo)
    assert np.array_equal(Y[1], hi)
    assert np.array_equal(oracle.unpack(4, packed, 256, 2, lib=lib).astype(np.float64), np.stack([lo, hi], 1))


def pin_bruteforce_int5(lib):
    # K = 8 codes per row (40 bits); row (p, v) holds value v at position p, zeros elsewhere
    rows, want = [], []
    for p in range(8):
        for v in range(-16, 16):
            stream = (v & 31) << (5 * p)
            rows.append(list(stream.to_bytes(5, "little")))
            want.append((p, v))
    packed = np.array(rows, np.uint8)
    N = packed.shape[0]
    codes = oracle.unpack(5, packed, N, 8, lib=lib)
    for r, (p, v) in enumerate(want):
        exp = np.zeros(8, np.int8)
        exp[p] = v
        assert np.array_equal(codes[r], exp), (p, v, codes[r])
    scales = np.full((N, 1), 0x3C00, np.uint16)
    x = np.eye(8, dtype=np.uint16) * np.uint16(0x3F80)
    Y, _ = oracle.gemm(5, packed, scales, x, N, 8, lib=lib)
    for r, (p, v) in enumerate(want):
        col = np.zeros(8)
        col[p] = v
        assert np.array_equal(Y[:, r], col)


def pin_numpy_matmul(lib):
    for seed, (N, K, T, bits) in enumerate([(33, 256, 5, 4), (17, 320, 3, 5), (64, 512, 2, 4)]):
        w, x = small_case(seed + 101, N, K, T, bits)
        W = w["codes"].astype(np.float64) * np.repeat(fp16_values(w["scales"]), 64, axis=1)[:, :K]
        Xd = bf16_values(x)
        ref = Xd @ W.T
        mag = np.abs(Xd) @ np.abs(W).T
        Y, A = oracle.gemm(bits, w["packed"], w["scales"], x, N, K, lib=lib)
        assert np.all(np.abs(Y - ref) <= 2 * K * U * mag), (N, K, T, bits)
        assert np.all(np.abs(A - mag) <= 2 * K * U * mag)
        Wo = oracle.dequant(bits, w["packed"], w["scales"], N, K, lib=lib)
        assert np.array_equal(Wo, W)


def pin_linearity_exact(lib):
    # integer-valued data: every partial sum is exact, so equalities are bitwise
    rng = np.random.default_rng(5)
    N, K, T = 9, 128, 3
    codes = rng.integers(-8, 8, size=(N, K))
    packed = synth.pack_canonical(codes, 4)
    scales = synth.fp64_to_fp16_bits(2.0 ** rng.integers(-2, 3, size=(N, 2)).astype(np.float64))
    xv = rng.integers(-4, 5, size=(T, K)).astype(np.float64)
    x = synth.fp64_to_bf16_bits(xv)
    even = np.zeros_like(xv)
    even[:, 0::2] = xv[:, 0::2]
    odd = xv - even
    Y, _ = oracle.gemm(4, packed, scales, x, N, K, lib=lib)
    Y1, _ = oracle.gemm(4, packed, scales, synth.fp64_to_bf16_bits(even), N, K, lib=lib)
    Y2, _ = oracle.gemm(4, packed, scales, synth.fp64_to_bf16_bits(odd), N, K, lib=lib)
    assert np.array_equal(Y, Y1 + Y2)
    Y3, _ = oracle.gemm(4, packed, scales, synth.fp64_to_bf16_bits(xv * 8.0), N, K, lib=lib)
    assert np.array_equal(Y3, 8.0 * Y)


def pin_identity_and_permutation(lib):
    N = K = 64
    T = 4
    x = synth.activations(3, T, K, outliers=True)
    xv = bf16_values(x)
    eye = np.eye(N, K, dtype=np.int8)
    ones = np.full((N, 1), 0x3C00, np.uint16)
    Y, _ = oracle.gemm(4, synth.pack_canonical(eye, 4), ones, x, N, K, lib=lib)
    assert np.array_equal(Y, xv[:, :N])
    perm = np.random.default_rng(9).permutation(K)[:N]
    P = np.zeros((N, K), np.int8)
    P[np.arange(N), perm] = 1
    for bits in (4, 5):
        Y, _ = oracle.gemm(bits, synth.pack_canonical(P, bits), ones, x, N, K, lib=lib)
        assert np.array_equal(Y, xv[:, perm])


def pin_scaling_and_negation(lib):
    N, K, T = 12, 192, 3
    w, x = small_case(21, N, K, T, 4)
    Y, _ = oracle.gemm(4, w["packed"], w["scales"], x, N, K, lib=lib)
    s2 = w["scales"].copy()
    s2[5] = synth.fp64_to_fp16_bits(fp16_values(s2[5]) * 4.0)        # row 5 scaled by 2^2
    Y2, _ = oracle.gemm(4, w["packed"], s2, x, N, K, lib=lib)
    exp = Y.copy()
    exp[:, 5] *= 4.0
    assert np.array_equal(Y2, exp)
    sneg = w["scales"] ^ np.uint16(0x8000)                           # flip every scale's sign
    Yn, _ = oracle.gemm(4, w["packed"], sneg, x, N, K, lib=lib)
    assert np.array_equal(Yn, -Y)


def pin_int5_contains_int4(lib):
    N, K, T = 10, 128, 2
    codes = synth.uniform_codes(4, 1, N, K, 4)
    scales = synth.group_scales(4, 2, N, K)
    x = synth.activations(4, T, K, outliers=False)
    Y4, _ = oracle.gemm(4, synth.pack_canonical(codes, 4), scales, x, N, K, lib=lib)
    Y5, _ = oracle.gemm(5, synth.pack_canonical(codes, 5), scales, x, N, K, lib=lib)
    assert np.array_equal(Y4, Y5)


def pin_column_independence(lib):
    N, K, T = 8, 128, 5
    w, x = small_case(31, N, K, T, 5)
    Y, _ = oracle.gemm(5, w["packed"], w["scales"], x, N, K, lib=lib)
    for t in range(T):
        Yt, _ = oracle.gemm(5, w["packed"], w["scales"], x[t:t + 1], N, K, lib=lib)
        assert np.array_equal(Yt[0], Y[t])


def pin_swiglu(lib):
    # closed forms: sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4 exactly, so
    # silu(+-ln 3) = +-(3/4 or 1/4) ln 3; silu(0) = 0; silu(z) -> z for large z
    l3 = np.log(3.0)
    g = np.array([0.0, l3, -l3, 40.0, -40.0, 1.5])
    u = np.array([7.0, 2.0, 2.0, 0.5, 1.0, -3.0])
    out = oracle.swiglu(g, u, lib=lib)
    assert out[0] == 0.0
    assert abs(out[1] - 1.5 * l3) <= 4 * U * 1.5 * l3
    assert abs(out[2] + 0.5 * l3) <= 4 * U * 0.5 * l3
    assert abs(out[3] - 20.0) <= 1e-15 * 20.0
    assert abs(out[4]) < 1e-15
    # against scipy's logistic function (a library routine) on random inputs
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(5)
    g = rng.uniform(-30, 30, 257)
    u = rng.normal(0, 3, 257)
    ref = g * special.expit(g) * u
    assert np.allclose(oracle.swiglu(g, u, lib=lib), ref, rtol=1e-13, atol=1e-300)


def pin_linear_add(lib):
    N, K, T = 9, 192, 3
    w, x = small_case(41, N, K, T, 4)
    rng = np.random.default_rng(41)
    R = rng.normal(0, 4, (T, N)).astype(np.float32)
    Rd = R.astype(np.float64)
    # zero scales: the product term vanishes and Y is R itself, A is |R|
    zero = np.zeros_like(w["scales"])
    Y0, A0 = oracle.linear_add(4, w["packed"], zero, x, R, N, K, lib=lib)
    assert np.array_equal(Y0, Rd) and np.array_equal(A0, np.abs(Rd))
    # zero residual: the plain result
    Yg, Ag = oracle.gemm(4, w["packed"], w["scales"], x, N, K, lib=lib)
    Yz, Az = oracle.linear_add(4, w["packed"], w["scales"], x, np.zeros((T, N), np.float32), N, K, lib=lib)
    assert np.array_equal(Yz, Yg) and np.array_equal(Az, Ag)
    # integer-valued weights and activations: every sum is exact, so Y = R + Y0 exactly
    codes = synth.uniform_codes(41, 3, N, K, 4)
    ones = np.full((N, K // 64), 0x3C00, np.uint16)                  # fp16 1.0
    xi = synth.fp64_to_bf16_bits(rng.integers(-3, 4, (T, K)).astype(np.float64))
    Ri = rng.integers(-1000, 1000, (T, N)).astype(np.float32)
    Yi, _ = oracle.linear_add(4, synth.pack_canonical(codes, 4), ones, xi, Ri, N, K, lib=lib)
    exact = Ri.astype(np.int64) + rng_free_dot(xi, codes)
    assert np.array_equal(Yi, exact.astype(np.float64))


def rng_free_dot(x_bits, codes):
    """Integer X . codes^T for integer-valued bf16 activations (exact, in int64)."""
    xv = bf16_values(x_bits).astype(np.int64)
    return xv @ codes.astype(np.int64).T


def fp8_values_torch(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes -> fp64 through torch's float8_e4m3fn type (a library routine)."""
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_fp8_decode(lib):
    # every byte once, unit scales: the dequantised row is the codes' values
    codes = np.arange(256, dtype=np.uint8).reshape(1, 256)
    ones = np.full((1, 4), 0x3C00, np.uint16)
    W = oracle.dequant(8, codes, ones, 1, 256, lib=lib)[0]
    ref = fp8_values_torch(codes[0])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(W), nan) and nan.sum() == 2
    assert np.array_equal(W[~nan], ref[~nan])
    assert np.array_equal(np.signbit(W[~nan]), np.signbit(ref[~nan]))      # -0.0 included
    # closed forms: 1.0, the largest value, the smallest subnormal and normal
    assert (W[0x38], W[0x7E], W[0x01], W[0x08], W[0xB8]) == (1.0, 448.0, 2.0 ** -9, 2.0 ** -6, -1.0)


def pin_fp8_gemm(lib):
    N, K, T = 11, 192, 3
    codes = synth.uniform_codes(51, 1, N, K, 8)
    scales = synth.group_scales(51, 2, N, K)
    x = synth.activations(51, T, K, outliers=True)
    Y, A = oracle.gemm(8, codes, scales, x, N, K, lib=lib)
    w = fp8_values_torch(codes) * np.repeat(fp16_values(scales), 64, axis=1)[:, :K]
    xv = bf16_values(x)
    ref = xv @ w.T
    mag = np.abs(xv) @ np.abs(w).T
    assert np.all(np.abs(Y - ref) <= 2 * K * U * mag)
    assert np.allclose(A, mag, rtol=4 * K * U)


# ------------------------------------------------------------ NVFP4

# E2M1 magnitudes by the code's low three bits (exponent e, mantissa m): the
# format's value set {0, 1/2, 1, 3/2, 2, 3, 4, 6}, written here as twice the
# value, an integer, rather than from the exponent and mantissa fields
E2M1_TWICE = [0, 1, 2, 3, 4, 6, 8, 12]


def e2m1_values_table(codes):
    codes = np.asarray(codes, np.int64)
    mag = np.array(E2M1_TWICE, np.float64)[codes & 7] / 2.0
    return np.where(codes & 8, -mag, mag)


def ue4m3_values_torch(codes):
    # an unsigned E4M3 code is an OCP E4M3 code with the sign bit clear
    return fp8_values_torch(np.asarray(codes, np.uint8) & 0x7F)


def pin_nvfp4_decode(lib):
    # every E2M1 code against the value set, with a unit block and tensor scale
    codes = np.arange(16, dtype=np.uint8).reshape(1, 16)
    W = oracle.dequant_nvfp4(synth.pack_nibbles(codes), np.full((1, 1), 0x38, np.uint8), 1.0, 1, 16, lib=lib)[0]
    assert np.array_equal(W, e2m1_values_table(codes[0]))
    assert np.signbit(W[8]) and W[8] == 0.0                                 # code 8 is -0.0
    # every unsigned E4M3 block scale (the E2M1 code 2 is 1.0) against torch
    bs = np.arange(256, dtype=np.uint8).reshape(256, 1)
    ones = np.full((256, 16), 2, np.uint8)
    Wb = oracle.dequant_nvfp4(synth.pack_nibbles(ones), bs, 1.0, 256, 16, lib=lib)[:, 0]
    ref = ue4m3_values_torch(bs[:, 0])
    outside = (bs[:, 0] >= 0x80) | (bs[:, 0] == 0x7F)
    assert np.all(np.isnan(Wb[outside])) and not np.any(np.isnan(Wb[~outside]))
    assert np.array_equal(Wb[~outside], ref[~outside])
    assert (Wb[0x38], Wb[0x7E], Wb[0x01], Wb[0x08]) == (1.0, 448.0, 2.0 ** -9, 2.0 ** -6)


def pin_nvfp4_gemm(lib):
    # the whole formula against numpy on weights the test dequantises itself:
    # one block scale per 16 columns, the tensor scale, nibble order
    N, K, T = 13, 160, 4
    p = synth.weights(52, N, K, synth.NVFP4)
    x = synth.activations(52, T, K, outliers=True)
    Y, A = oracle.gemm_parent(p, x, lib=lib)
    w = e2m1_values_table(p["codes"]) * np.repeat(ue4m3_values_torch(p["scales"]), 16, axis=1)[:, :K] * p["tscale"]
    xv = bf16_values(x)
    ref = xv @ w.T
    mag = np.abs(xv) @ np.abs(w).T
    assert np.all(np.abs(Y - ref) <= 2 * K * U * mag)
    assert np.allclose(A, mag, rtol=4 * K * U)
    # a power-of-two tensor scale scales the result exactly
    Y2, _ = oracle.gemm_nvfp4(p["packed"], p["scales"], 2 * p["tscale"], x, N, K, lib=lib)
    assert np.array_equal(Y2, 2 * Y)


PINS = [pin_golden, pin_exact_rational, pin_bruteforce_int4, pin_bruteforce_int5, pin_numpy_matmul,
        pin_linearity_exact, pin_identity_and_permutation, pin_scaling_and_negation,
        pin_int5_contains_int4, pin_column_independence, pin_swiglu, pin_linear_add, pin_fp8_decode,
        pin_fp8_gemm, pin_nvfp4_decode, pin_nvfp4_gemm]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.load())


# ------------------------------------------------------------ planted mistakes

MUTANTS = {
    "dropped_last_term": ("for (int k = 0; k < K; ++k) {\n                double p",
                          "for (int k = 0; k < K - 1; ++k) {\n                double p"),
    "sign_extension": ("return nib >= 8 ? nib - 16 : nib;", "return nib > 8 ? nib - 16 : nib;"),
    "nibble_order": ("(k & 1) ? (byte >> 4) : (byte & 0x0f)", "(k & 1) ? (byte & 0x0f) : (byte >> 4)"),
    "transposed_scales": ("w[k] = s * oracle_value(bits, row, k);",
                          "w[k] = oracle_half_to_double(scales[(size_t)(k / ORACLE_GROUP) * N + n])"
                          " * oracle_value(bits, row, k); (void)s;"),
    "int5_sign": ("return v >= 16 ? v - 32 : v;", "return v >= 16 ? v - 31 : v;"),
    "int5_bit_order": ("& 1) << b;", "& 1) << (4 - b);"),
    "abs_sum": ("mag += fabs(p);", "mag += p;"),
    "x_stride": ("const uint16_t *xr = X + (size_t)t * K;", "const uint16_t *xr = X + (size_t)t;"),
    "half_bias": ("expo - 25);", "expo - 24);"),
    "half_subnormal": ("ldexp((double)mant, -24);", "ldexp((double)mant, -25);"),
    "group_width": ("#define ORACLE_GROUP 64", "#define ORACLE_GROUP 128"),
    "silu_sign": ("out[i] = g[i] / (1.0 + exp(-g[i])) * u[i];", "out[i] = g[i] / (1.0 + exp(g[i])) * u[i];"),
    "silu_gate_up_swapped": ("out[i] = g[i] / (1.0 + exp(-g[i])) * u[i];",
                             "out[i] = u[i] / (1.0 + exp(-u[i])) * g[i];"),
    "residual_dropped": ("Y[i] = (double)R[i] + Y[i];", "Y[i] = Y[i];"),
    "residual_abs": ("A[i] = fabs((double)R[i]) + A[i];", "A[i] = (double)R[i] + A[i];"),
    "e4m3_bias": ("ldexp((double)(8 + mant), expo - 10);", "ldexp((double)(8 + mant), expo - 9);"),
    "e4m3_subnormal": ("ldexp((double)mant, -9);", "ldexp((double)mant, -10);"),
    "e4m3_nan": ("if (expo == 15 && mant == 7)", "if (expo == 15)"),
    "e4m3_sign": ("int sign = b >> 7;", "int sign = (b >> 6) & 1;"),
    "e2m1_bias": ("ldexp(1.0 + 0.5 * mant, expo - 1);", "ldexp(1.0 + 0.5 * mant, expo);"),
    "e2m1_subnormal": ("expo == 0 ? 0.5 * mant", "expo == 0 ? 1.0 * mant"),
    "e2m1_sign": ("int sign = (nib >> 3) & 1;", "int sign = (nib >> 2) & 1;"),
    "nvfp4_block_width": ("#define ORACLE_NVFP4_BLOCK 16", "#define ORACLE_NVFP4_BLOCK 32"),
    "nvfp4_tensor_scale_dropped": ("* oracle_ue4m3_to_double(bs_row[k / ORACLE_NVFP4_BLOCK]) * ts;",
                                   "* oracle_ue4m3_to_double(bs_row[k / ORACLE_NVFP4_BLOCK]);"),
    "ue4m3_signed": ("if ((b & 0x80) || (expo == 15 && mant == 7))", "if (expo == 15 && mant == 7)"),
    "nvfp4_nibble_order": ("int nib = (k & 1) ? (byte >> 4) : (byte & 0x0f);\n        w[k]",
                           "int nib = (k & 1) ? (byte & 0x0f) : (byte >> 4);\n        w[k]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new)
    cpath = tmp_path / "mutant.c"
    cpath.write_text(mutated)
    so = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", so, str(cpath), "-lm"], check=True)
    lib = oracle.load(so)
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
