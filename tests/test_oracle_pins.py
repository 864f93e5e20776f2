"""Pins for the CPU oracle: checks against facts that do not come from the oracle.

Each test ties the oracle to something independent of its own code: the
IEEE/bfloat16 bit layouts as decoded by numpy, hand-written packed words,
exact rational arithmetic (Python ``fractions``), a dense numpy float64
product, closed forms of degenerate inputs, and the worked example printed on
the "15 year old GPU" page.  ``test_pins_catch_planted_mistakes`` compiles
deliberately broken copies of the oracle and checks that these pins fail.
"""
import math
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

from quantized_weight_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- decoders

def test_half_decoder_matches_numpy_for_every_pattern(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_double(int(p)) for p in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zero survives decoding
    assert math.copysign(1.0, oracle_mod.half_to_double(0x8000)) == -1.0


def test_bf16_decoder_matches_upper_half_of_binary32(oracle_mod):
    # bfloat16 is, by definition, the upper 16 bits of an IEEE binary32.
    pats = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (pats << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([oracle_mod.bf16_to_double(int(p)) for p in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- packing

def test_pack_known_words(oracle_mod):
    # INT4: codes k mod 16 -> lowest nibble holds the lowest k.
    c4 = (np.arange(64) % 16).astype(np.uint8)[None, :]
    w4 = oracle_mod.pack(c4, 4)
    assert [hex(v) for v in w4[0, :2]] == ["0x76543210", "0xfedcba98"]
    # INT8: one byte per code, little-endian in the word, two's complement.
    c8 = np.zeros((1, 32), dtype=np.uint8)
    c8[0, :4] = [1, 2, 3, 0xFF]          # 0xFF is the int8 value -1
    assert oracle_mod.pack(c8, 8)[0, 0] == 0xFF030201
    # Q1: bit (k mod 32) of word k/32.
    c1 = np.zeros((1, 64), dtype=np.uint8)
    c1[0, 0] = 1
    c1[0, 33] = 1
    c1[0, 63] = 1
    w1 = oracle_mod.pack(c1, 1)
    assert w1[0, 0] == 0x1 and w1[0, 1] == 0x80000002
    alt = (np.arange(32) % 2 == 0).astype(np.uint8)[None, :]
    assert oracle_mod.pack(alt, 1)[0, 0] == 0x55555555


@pytest.mark.parametrize("bits", [1, 4, 8])
def test_pack_unpack_roundtrip(oracle_mod, bits):
    d = inputs.make(1, 7, 256, bits, 64 if bits != 1 else 128, seed=3)
    p = oracle_mod.pack(d["codes"], bits)
    assert p.shape == (7, 256 * bits // 32)
    assert np.array_equal(oracle_mod.unpack(p, 7, 256, bits), d["codes"])


def test_pack_rejects_codes_that_do_not_fit(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.pack(np.full((1, 32), 16, dtype=np.uint8), 4)
    with pytest.raises(ValueError):
        oracle_mod.pack(np.full((1, 32), 2, dtype=np.uint8), 1)


# ---------------------------------------------------------------- exact rationals

def _frac_half(u16):
    return Fraction(float(np.uint16(u16).view(np.float16)))


def _exact_y(d, bits, group):
    """y = x . dequant(W)^T in exact rational arithmetic, from the unpacked codes."""
    codes, sc, bi, x = d["codes"], d["scales"], d["biases"], d["x"]
    N, K = codes.shape
    M = x.shape[0]
    W = []
    for n in range(N):
        row = []
        for k in range(K):
            s = _frac_half(sc[n, k // group])
            c = int(codes[n, k])
            if bits == 4:
                row.append(s * c + _frac_half(bi[n, k // group]))
            elif bits == 8:
                row.append(s * (c - 256 if c >= 128 else c))
            else:
                row.append(s * (2 * c - 1))
        W.append(row)
    X = [[Fraction(float(v)) for v in x[m]] for m in range(M)]
    y = [[sum(W[n][k] * X[m][k] for k in range(K)) for n in range(N)] for m in range(M)]
    absum = [[sum(abs(W[n][k] * X[m][k]) for k in range(K)) for n in range(N)] for m in range(M)]
    return y, absum


TINY = [(bits, group, K, M, N, seed)
        for bits, group in [(4, 64), (4, 32), (8, 64), (1, 128), (1, 32)]
        for (K, M, N, seed) in [(128, 2, 3, 0), (64 if group <= 64 else 128, 1, 2, 1)]]


@pytest.mark.parametrize("bits,group,K,M,N,seed", TINY)
def test_oracle_equals_exact_rationals_within_rounding_bound(oracle_mod, bits, group, K, M, N, seed):
    d = inputs.make(M, N, K, bits, group, seed=seed)
    p = oracle_mod.pack(d["codes"], bits)
    got = oracle_mod.qmm_f32x(d["x"], p, d["scales"], d["biases"], N, K, bits, group)
    y, absum = _exact_y(d, bits, group)
    # Rounding bound for a length-K dot product of exact weights in double:
    # |fl(sum) - sum| <= gamma_{K+1} * sum |w_k x_k|,  gamma_n = n u / (1 - n u).
    u = 2.0 ** -53
    gamma = (K + 1) * u / (1 - (K + 1) * u)
    for m in range(M):
        for n in range(N):
            err = abs(Fraction(got[m, n]) - y[m][n])
            assert err <= Fraction(gamma) * absum[m][n], (m, n, float(err))


def test_bf16_activations_decode_exactly(oracle_mod):
    d = inputs.make(2, 3, 128, 4, 64, seed=5, prefill=True)
    p = oracle_mod.pack(d["codes"], 4)
    xb = d["x_bf16"]
    got = oracle_mod.qmm_bf16x(xb, p, d["scales"], d["biases"], 3, 128, 4, 64)
    # the same activations given as float32 (bf16 widened exactly) give the same y
    xf = (xb.astype(np.uint32) << 16).view(np.float32)
    ref = oracle_mod.qmm_f32x(xf, p, d["scales"], d["biases"], 3, 128, 4, 64)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- library cross-check

@pytest.mark.parametrize("bits,group", [(4, 64), (8, 64), (1, 128)])
def test_oracle_matches_dense_numpy_product(oracle_mod, bits, group):
    M, N, K = 3, 37, 512
    d = inputs.make(M, N, K, bits, group, seed=11)
    s = d["scales"].view(np.float16).astype(np.float64).repeat(group, axis=1)
    c = d["codes"]
    if bits == 4:
        W = s * c.astype(np.float64) + d["biases"].view(np.float16).astype(np.float64).repeat(group, axis=1)
    elif bits == 8:
        W = s * c.view(np.int8).astype(np.float64)
    else:
        W = s * (2.0 * c.astype(np.float64) - 1.0)
    ref = d["x"].astype(np.float64) @ W.T
    p = oracle_mod.pack(c, bits)
    got = oracle_mod.qmm_f32x(d["x"], p, d["scales"], d["biases"], N, K, bits, group)
    rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert rel.max() <= 1e-12
    wd = oracle_mod.dequant(p, d["scales"], d["biases"], N, K, bits, group)
    assert np.array_equal(wd, W)   # dequantization is exact in double


def test_sampled_outputs_equal_full_product(oracle_mod):
    d = inputs.make(4, 50, 256, 4, 64, seed=2, prefill=True)
    p = oracle_mod.pack(d["codes"], 4)
    full = oracle_mod.qmm_bf16x(d["x_bf16"], p, d["scales"], d["biases"], 50, 256, 4, 64, nthreads=3)
    ms, ns = np.array([0, 3, 2, 1]), np.array([0, 49, 17, 5])
    got = oracle_mod.qmm_sampled(d["x_bf16"], p, d["scales"], d["biases"], ms, ns, 50, 256, 4, 64)
    assert np.array_equal(got, full[ms, ns])
    full1 = oracle_mod.qmm_bf16x(d["x_bf16"], p, d["scales"], d["biases"], 50, 256, 4, 64, nthreads=1)
    assert np.array_equal(full, full1)   # thread count does not change any output


# ---------------------------------------------------------------- closed forms and invariants

def _groupsum(x, group):
    M, K = x.shape
    return x.astype(np.float64).reshape(M, K // group, group).sum(axis=2)


def test_zero_codes_int4_give_bias_times_group_sums(oracle_mod):
    M, N, K, g = 2, 9, 256, 64
    d = inputs.make(M, N, K, 4, g, seed=4, codes="zeros")
    p = oracle_mod.pack(d["codes"], 4)
    y = oracle_mod.qmm_f32x(d["x"], p, d["scales"], d["biases"], N, K, 4, g)
    b = d["biases"].view(np.float16).astype(np.float64)
    ref = _groupsum(d["x"], g) @ b.T            # y = sum_g b_g * X_g
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13)


def test_zero_codes_int8_give_exact_zero(oracle_mod):
    d = inputs.make(2, 5, 128, 8, 64, seed=4, codes="zeros")
    p = oracle_mod.pack(d["codes"], 8)
    y = oracle_mod.qmm_f32x(d["x"], p, d["scales"], None, 5, 128, 8, 64)
    assert np.all(y == 0.0)


def test_q1_all_plus_one_is_scale_times_group_sums_and_flip_negates(oracle_mod):
    M, N, K, g = 2, 6, 512, 128
    d = inputs.make(M, N, K, 1, g, seed=6, codes="ones")
    p = oracle_mod.pack(d["codes"], 1)
    y = oracle_mod.qmm_f32x(d["x"], p, d["scales"], None, N, K, 1, g)
    s = d["scales"].view(np.float16).astype(np.float64)
    assert np.allclose(y, _groupsum(d["x"], g) @ s.T, rtol=1e-13, atol=1e-13)
    # all bits 0 gives exactly the negation
    p0 = oracle_mod.pack(np.zeros_like(d["codes"]), 1)
    y0 = oracle_mod.qmm_f32x(d["x"], p0, d["scales"], None, N, K, 1, g)
    assert np.array_equal(y0, -y)
    # flipping every bit of random signs negates y exactly
    r = inputs.make(M, N, K, 1, g, seed=7)
    pr = oracle_mod.pack(r["codes"], 1)
    pf = oracle_mod.pack(1 - r["codes"], 1)
    yr = oracle_mod.qmm_f32x(r["x"], pr, r["scales"], None, N, K, 1, g)
    yf = oracle_mod.qmm_f32x(r["x"], pf, r["scales"], None, N, K, 1, g)
    assert np.array_equal(yf, -yr)


@pytest.mark.parametrize("bits,group", [(4, 64), (8, 64), (1, 128)])
def test_doubling_coefficients_doubles_y_exactly(oracle_mod, bits, group):
    d = inputs.make(2, 8, 256, bits, group, seed=8)
    p = oracle_mod.pack(d["codes"], bits)
    y = oracle_mod.qmm_f32x(d["x"], p, d["scales"], d["biases"], 8, 256, bits, group)
    dbl = lambda a: None if a is None else (a.view(np.float16).astype(np.float64) * 2).astype(np.float16).view(np.uint16)
    y2 = oracle_mod.qmm_f32x(d["x"], p, dbl(d["scales"]), dbl(d["biases"]), 8, 256, bits, group)
    assert np.array_equal(y2, 2.0 * y)


@pytest.mark.parametrize("bits,group", [(4, 64), (8, 64), (1, 128)])
def test_linearity_in_x(oracle_mod, bits, group):
    d1 = inputs.make(2, 8, 256, bits, group, seed=9)
    d2 = inputs.make(2, 8, 256, bits, group, seed=10)
    p = oracle_mod.pack(d1["codes"], bits)
    f = lambda x: oracle_mod.qmm_f32x(x, p, d1["scales"], d1["biases"], 8, 256, bits, group)
    xs = (d1["x"].astype(np.float64) + d2["x"].astype(np.float64)).astype(np.float32)
    # float32 sum may round; compare with the sum of parts within that rounding
    lhs = f(xs)
    rhs = f(d1["x"]) + f(d2["x"])
    scale = np.abs(f(np.abs(xs))).max() + 1.0
    assert np.abs(lhs - rhs).max() <= 1e-6 * scale


def test_permuting_groups_consistently_keeps_y(oracle_mod):
    M, N, K, g = 2, 5, 256, 64
    d = inputs.make(M, N, K, 4, g, seed=12)
    perm = np.array([2, 0, 3, 1])
    kperm = (perm[:, None] * g + np.arange(g)[None, :]).ravel()
    p = oracle_mod.pack(d["codes"], 4)
    pp = oracle_mod.pack(np.ascontiguousarray(d["codes"][:, kperm]), 4)
    y = oracle_mod.qmm_f32x(d["x"], p, d["scales"], d["biases"], N, K, 4, g)
    yp = oracle_mod.qmm_f32x(np.ascontiguousarray(d["x"][:, kperm]), pp,
                             np.ascontiguousarray(d["scales"][:, perm]),
                             np.ascontiguousarray(d["biases"][:, perm]), N, K, 4, g)
    assert np.allclose(y, yp, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- the page's worked example

def _golden(name):
    vals = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (t.strip() for t in line.split("="))
                vals[k] = float(v)
    return vals


def test_affine_worked_example_from_the_page(oracle_mod):
    g = _golden("affine_worked_example.txt")
    block = np.array([g["block_min"], g["block_max"], g["weight"]])
    q, scale, mn = oracle_mod.quantize_affine4(block)
    assert round(scale, 4) == g["scale"]
    assert round((g["weight"] - mn) / scale, 2) == g["quotient"]
    assert q[2] == g["code"] and q[0] == g["code_of_min"] and q[1] == g["code_of_max"]
    # dequantized = q * scale + min, through the oracle's INT4 path, with the
    # coefficients stored as binary16 the way the library stores them
    codes = np.zeros((1, 64), dtype=np.uint8)
    codes[0, 5] = q[2]
    s16 = np.array([[scale]], dtype=np.float16).view(np.uint16)
    b16 = np.array([[mn]], dtype=np.float16).view(np.uint16)
    w = oracle_mod.dequant(oracle_mod.pack(codes, 4), s16, b16, 1, 64, 4, 64)
    assert round(w[0, 5], 2) == g["dequantized"]
    assert w[0, 0] == mn


# ---------------------------------------------------------------- the pins catch mistakes

MUTANTS = {
    "dropped bias": ("return s * (double)q + b;", "return s * (double)q;"),
    "Q1 polarity": ("return s * (double)(2 * q - 1);", "return s * (double)(1 - 2 * q);"),
    "int8 unsigned": ("if (bits == 8 && u >= 128) u -= 256;", ";"),
    "nibble order": ("int shift = (int)(bits * (k % per_word));",
                     "int shift = (int)(bits * (per_word - 1 - k % per_word));"),
    "group index": ("int64_t g = k / group;", "int64_t g = (k / group) % 2;"),
    "half subnormal": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "last group skipped": ("for (int64_t g0 = 0; g0 < K; g0 += group)",
                           "for (int64_t g0 = 0; g0 + group < K; g0 += group)"),
    "binary16 ties round up": ("if (rem > half || (rem == half && (q & 1u))) q++;", "if (rem >= half) q++;"),
    "quantizer truncates": ("float r = roundf(t);", "float r = truncf(t);"),
    "quantizer ignores the bias": ("volatile float d = v[i] - b;", "volatile float d = v[i];"),
    "quantizer max skipped": ("if (isnan(hi) || x > hi || (x == hi && !signbit(x) && signbit(hi))) hi = x;",
                              "if (isnan(hi)) hi = x;"),
}


def _checks_fail_with(lib_file):
    """Run a compact set of the pins above against another build of the oracle."""
    import importlib
    import oracle.oracle as om
    saved = (om._lib, om._LIB)
    om._lib, om._LIB = None, lib_file
    try:
        fails = 0
        for bits, group in [(4, 64), (8, 64), (1, 128), (4, 32)]:
            d = inputs.make(2, 3, 128, bits, group, seed=1)
            p = om.pack(d["codes"], bits)
            got = om.qmm_f32x(d["x"], p, d["scales"], d["biases"], 3, 128, bits, group)
            y, absum = _exact_y(d, bits, group)
            u = 2.0 ** -53
            gamma = 129 * u / (1 - 129 * u)
            for m in range(2):
                for n in range(3):
                    if abs(Fraction(got[m, n]) - y[m][n]) > Fraction(gamma) * absum[m][n]:
                        fails += 1
        sub = np.array([om.half_to_double(v) for v in range(1, 1024)])
        if not np.array_equal(sub, np.arange(1, 1024, dtype=np.uint16).view(np.float16).astype(np.float64)):
            fails += 1
        # binary16 encoder: ties to even, overflow, the subnormal edge
        for v, want in [(1.0 + 2.0 ** -11, 0x3C00), (1.0 + 3 * 2.0 ** -11, 0x3C02), (65520.0, 0x7C00),
                        (2.0 ** -25, 0x0000), (3 * 2.0 ** -26, 0x0001)]:
            if om.float_to_half(v) != want:
                fails += 1
        # stored-format quantizer: an exact grid, and half a step of error at most
        j = np.arange(64) % 16
        j[1] = 15
        w = (np.float32(-1.0) + j.astype(np.float32) * np.float32(0.0625))[None, :]
        c, sh, bh = om.quantize_affine4_f32(np.ascontiguousarray(w), 64)
        if not np.array_equal(c[0], j):
            fails += 1
        wr = np.random.default_rng(3).standard_normal((8, 128)).astype(np.float32)
        c, sh, bh = om.quantize_affine4_f32(wr, 64)
        s = sh.view(np.float16).astype(np.float64).repeat(64, axis=1)
        if (np.abs(_dq(c, sh, bh, 64) - wr) > s * 0.5 + 2.0 ** -10).any():
            fails += 1
        return fails > 0
    finally:
        om._lib, om._LIB = saved


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(tmp_path, name):
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "qmm_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name!r} not found"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    from oracle.oracle import CFLAGS
    subprocess.run(["gcc", *CFLAGS, str(mut), "-o", str(so), "-lm"], check=True)
    assert _checks_fail_with(str(so)), f"planted mistake {name!r} passed every pin"


# ---------------------------------------------------------------- binary16 encoder and stored-format quantizer

def test_float_to_half_rounds_like_numpy_at_every_boundary(oracle_mod):
    """The oracle's own float32 -> binary16 encoder against numpy's cast (IEEE
    round to nearest even) at every tie between adjacent binary16 values and
    one float32 step on either side of it, plus the overflow edge."""
    h = np.arange(0, 0x7C00, dtype=np.uint16)                # finite non-negative halves
    lo = h[:-1].view(np.float16).astype(np.float64)
    hi = h[1:].view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)                  # exact: 11 bits fit in 24
    cand = np.concatenate([mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0)),
                           h.view(np.float16).astype(np.float32),
                           np.array([65504.0, 65519.996, 65520.0, 1e9, 2.0 ** -25, 2.0 ** -26, 1e-30],
                                    dtype=np.float32)])
    cand = np.concatenate([cand, -cand])
    rng = np.random.default_rng(7)
    cand = cand[rng.permutation(cand.size)[:60000]]
    with np.errstate(over="ignore"):
        ref = cand.astype(np.float16).view(np.uint16)
    got = np.array([oracle_mod.float_to_half(float(v)) for v in cand], dtype=np.uint16)
    assert np.array_equal(got, ref)
    assert oracle_mod.float_to_half(float("nan")) == 0x7E00
    assert oracle_mod.float_to_half(float("inf")) == 0x7C00
    assert oracle_mod.float_to_half(-0.0) == 0x8000


def _dq(codes, sh, bh, group):
    s = sh.view(np.float16).astype(np.float64).repeat(group, axis=1)
    b = bh.view(np.float16).astype(np.float64).repeat(group, axis=1)
    return codes.astype(np.float64) * s + b


def test_stored_quantizer_reproduces_the_worked_example(oracle_mod):
    g = _golden("affine_worked_example.txt")
    w = np.full((1, 64), g["weight"], dtype=np.float32)
    w[0, 0], w[0, 1] = g["block_min"], g["block_max"]
    codes, sh, bh = oracle_mod.quantize_affine4_f32(w, 64)
    assert round(float(sh.view(np.float16)[0, 0]), 4) == g["scale"]
    assert bh.view(np.float16)[0, 0] == np.float16(g["block_min"])
    assert codes[0, 0] == g["code_of_min"] and codes[0, 1] == g["code_of_max"] and codes[0, 2] == g["code"]
    assert round(_dq(codes, sh, bh, 64)[0, 2], 2) == g["dequantized"]


def test_stored_quantizer_on_an_exact_grid(oracle_mod):
    """Values lo + j*s with s and lo exact in binary16 and every step exact in
    float32 quantize to q = j exactly, for every group size."""
    for group in (32, 64, 128):
        j = np.arange(group) % 16
        j[0], j[1] = 0, 15                                    # the range is exactly 15 steps
        w = (np.float32(-1.0) + j.astype(np.float32) * np.float32(0.0625))[None, :].repeat(3, axis=0)
        w[1] *= np.float32(4.0)                              # s = 0.25, lo = -4
        w[2] += np.float32(3.0)                              # lo = 2
        codes, sh, bh = oracle_mod.quantize_affine4_f32(np.ascontiguousarray(w), group)
        assert np.array_equal(codes, np.broadcast_to(j, w.shape))
        assert list(sh.view(np.float16)[:, 0]) == [0.0625, 0.25, 0.0625]
        assert list(bh.view(np.float16)[:, 0]) == [-1.0, -4.0, 2.0]


def test_stored_quantizer_constant_nan_and_bounds(oracle_mod):
    rng = np.random.default_rng(3)
    w = rng.standard_normal((64, 256)).astype(np.float32)
    w[0, :64] = 0.75                                          # constant group: scale 0, codes 0
    w[1, 5] = np.nan                                          # NaN is skipped, coded 0
    codes, sh, bh = oracle_mod.quantize_affine4_f32(w, 64)
    assert sh[0, 0] == 0 and (codes[0, :64] == 0).all() and bh.view(np.float16)[0, 0] == 0.75
    assert codes[1, 5] == 0
    assert codes.max() <= 15
    # every weight within half a step of its level (plus the binary16 rounding of the bias)
    s = sh.view(np.float16).astype(np.float64).repeat(64, axis=1)
    err = np.abs(_dq(codes, sh, bh, 64) - w)
    ok = ~np.isnan(w)
    ok[0, :64] = False
    assert (err[ok] <= s[ok] * 0.5 + 2.0 ** -10).all()
    # monotone: a sorted group gets non-decreasing codes
    ws = np.sort(w[2:3], axis=1)
    c2, _, _ = oracle_mod.quantize_affine4_f32(ws, 64)
    assert (np.diff(c2.reshape(-1, 64), axis=1) >= 0).all()
