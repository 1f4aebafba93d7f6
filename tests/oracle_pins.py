"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin takes an ``oracle.Oracle`` and returns ``(ok, detail)``. The pins use
library routines (torch's bf16 rounding, numpy's float64 matmul), exact
rational arithmetic (``fractions.Fraction``), closed forms of special cases,
the float-floor field chain of llama.cpp PR #159 "How", hand-worked
fixtures of the field order (``tests/golden/field_order.txt``) and, for the
mxfp4 mode, ml_dtypes' E2M1 and torch's E8M0 decoders.

``test_oracle.py`` asserts every pin passes on the real oracle, and that every
oracle build with a planted mistake (``-DORACLE_MUTANT=k``) fails at least one.
"""

from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "field_order.txt")


def _f64(bits16: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits16).astype(np.float64)


def _problem(N, K, M, bits, gs, seed):
    inp = synth.make_inputs(N, K, M, bits, gs, seed)
    return inp


def _numpy_dequant(inp) -> np.ndarray:
    """Dense fp64 W = s*q + b from the UNPACKED q, then numpy's matmul."""
    gs = inp.problem.group_size
    s = np.repeat(_f64(inp.scales), gs, axis=1)
    b = np.repeat(_f64(inp.biases), gs, axis=1)
    w = s * inp.q.astype(np.float64) + b
    return _f64(inp.x) @ w.T


# ------------------------------------------------------------------ bf16 --
def pin_bf16_rounding(o):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        # exact ties: bf16 value + half an ulp, both parities of the kept bit
        ((np.arange(1, 2000, dtype=np.uint32) << 16) | 0x8000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38, 1e-45], dtype=np.float32),
    ])
    ours = o.f32_to_bf16(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad = int(np.sum(ours != ref))
    return bad == 0, f"{bad} mismatches vs torch bf16 rounding"


def pin_bf16_widen(o):
    rng = np.random.default_rng(2)
    h = rng.integers(0, 1 << 16, 4000, dtype=np.uint32).astype(np.uint16)
    h = h[(h & 0x7F80) != 0x7F80]  # finite only
    ours = o.bf16_to_f64(h)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return bool(np.array_equal(ours, ref)), "bf16 widening vs torch"


# ---------------------------------------------------------------- fields --
def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            kind, bits, val, *fields = line.split()
            rows.append((kind, int(bits), int(val, 16), [int(v) for v in fields]))
    return rows


def pin_golden_field_order(o):
    for kind, bits, val, fields in _golden_rows():
        if kind == "byte":
            got = o.byte_fields(val, bits)
            if got != fields:
                return False, f"byte {val:#x} bits {bits}: {got} != {fields}"
        elif kind == "word":
            w = np.array([val], dtype=np.uint32)
            got = [o.field(w, i, bits) for i in range(32 // bits)]
            if got != fields:
                return False, f"word {val:#x} bits {bits}: {got} != {fields}"
            # packing the listed fields must give back the word
            q = np.array([fields], dtype=np.uint8)
            packed = o.pack(q, bits)
            if int(packed[0, 0]) != val:
                return False, f"pack {fields} -> {int(packed[0, 0]):#x} != {val:#x}"
        elif kind == "masked":
            # element k of a 16-bit word, scaled by 16**k, is (w & (0xf << 4k))
            w = np.array([val], dtype=np.uint32)
            got = [o.field(w, k, bits) * 16 ** k for k in range(4)]
            if got != fields:
                return False, f"masked {val:#x}: {got} != {fields}"
    return True, "golden field order"


def pin_floatfloor_exhaustive(o):
    for bits in (2, 4):
        for byte in range(256):
            a = o.byte_fields(byte, bits)
            b = o.byte_fields_floatfloor(byte, bits)
            if a != b:
                return False, f"byte {byte:#x} bits {bits}: shift/mask {a} != float-floor {b}"
    return True, "256 bytes x {2,4} bits agree with the float-floor chain"


def pin_pack_roundtrip(o):
    for bits in (2, 4):
        inp = _problem(5, 256, 1, bits, 64, 11)
        w = o.pack(inp.q, bits)
        for n in range(5):
            got = np.array([o.field(w[n], i, bits) for i in range(256)], dtype=np.uint8)
            if not np.array_equal(got, inp.q[n]):
                return False, f"bits {bits} row {n}: unpack(pack(q)) != q"
    return True, "pack/field round trip"


# ------------------------------------------------------------ arithmetic --
_SHAPES = [(7, 256, 2, 4, 64), (5, 384, 3, 2, 64), (6, 512, 1, 4, 128), (4, 256, 2, 2, 128)]


def pin_dequant_vs_numpy(o):
    for N, K, M, bits, gs in _SHAPES:
        inp = _problem(N, K, M, bits, gs, 3)
        w = o.pack(inp.q, bits)
        y = o.qmv_f64_dequant(w, inp.scales, inp.biases, inp.x, bits, gs)
        T = o.abs_terms(w, inp.scales, inp.biases, inp.x, bits, gs)
        ref = _numpy_dequant(inp)
        tref = np.abs(_f64(inp.x)) @ np.abs(
            np.repeat(_f64(inp.scales), gs, 1) * inp.q + np.repeat(_f64(inp.biases), gs, 1)).T
        if not np.all(np.abs(y - ref) <= 1e-12 * tref + 1e-300):
            return False, f"dequant vs numpy {(N, K, M, bits, gs)}: max {np.max(np.abs(y - ref))}"
        if not np.allclose(T, tref, rtol=1e-12, atol=0):
            return False, f"abs terms vs numpy {(N, K, M, bits, gs)}"
    return True, "fp64 dequantize-then-dot agrees with numpy's matmul of s*q+b"


def pin_factored_vs_dequant(o):
    for N, K, M, bits, gs in _SHAPES:
        inp = _problem(N, K, M, bits, gs, 4)
        w = o.pack(inp.q, bits)
        y1 = o.qmv_f64_dequant(w, inp.scales, inp.biases, inp.x, bits, gs)
        y2 = o.qmv_f64_factored(w, inp.scales, inp.biases, inp.x, bits, gs)
        T = o.abs_terms(w, inp.scales, inp.biases, inp.x, bits, gs)
        if not np.all(np.abs(y1 - y2) <= 1e-12 * T):
            return False, f"factored vs dequant {(N, K, M, bits, gs)}"
    return True, "factored and dequantized forms agree within 1e-12 * sum|w x|"


def _exact(inp, m, n):
    gs = inp.problem.group_size
    s = _f64(inp.scales[n])
    b = _f64(inp.biases[n])
    x = _f64(inp.x[m])
    tot = Fraction(0)
    for i in range(inp.problem.K):
        g = i // gs
        tot += (Fraction(float(s[g])) * int(inp.q[n, i]) + Fraction(float(b[g]))) * Fraction(float(x[i]))
    return tot


def pin_fraction_bruteforce(o):
    for K in (64, 128, 256):
        for bits in (2, 4):
            for gs in (64, 128):
                if K % gs:
                    continue
                inp = _problem(3, K, 2, bits, gs, 5 + K + bits + gs)
                w = o.pack(inp.q, bits)
                y1 = o.qmv_f64_dequant(w, inp.scales, inp.biases, inp.x, bits, gs)
                y2 = o.qmv_f64_factored(w, inp.scales, inp.biases, inp.x, bits, gs)
                T = o.abs_terms(w, inp.scales, inp.biases, inp.x, bits, gs)
                for m in range(2):
                    for n in range(3):
                        ex = _exact(inp, m, n)
                        for y in (y1, y2):
                            if abs(Fraction(float(y[m, n])) - ex) > Fraction(1e-13) * Fraction(float(T[m, n])):
                                return False, f"brute force K={K} bits={bits} gs={gs} ({m},{n})"
    return True, "both fp64 forms match exact rational arithmetic"


def _bf16(vals) -> np.ndarray:
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def pin_closed_forms(o):
    for bits in (2, 4):
        for gs in (64, 128):
            N, K = 6, 256
            G = K // gs
            inp = _problem(N, K, 1, bits, gs, 21 + bits + gs)
            w = o.pack(inp.q, bits)
            s, b = _f64(inp.scales), _f64(inp.biases)
            forms = (o.qmv_f64_dequant, o.qmv_f64_factored)
            # x == 1: y_n = sum_g (s_g * sum_t q + gs * b_g)
            ones = _bf16(np.ones((1, K)))
            qs = inp.q.astype(np.float64).reshape(N, G, gs).sum(-1)
            expect = (s * qs + gs * b).sum(1)
            for f in forms:
                y = f(w, inp.scales, inp.biases, ones, bits, gs)[0]
                if not np.allclose(y, expect, rtol=1e-13, atol=1e-15):
                    return False, f"x==1 closed form bits={bits} gs={gs}"
            # q == 0: y_n = sum_g b_g * sum_{i in g} x_i
            w0 = np.zeros_like(w)
            xs = _f64(inp.x).reshape(G, gs).sum(-1)
            expect = (b * xs[None, :]).sum(1)
            for f in forms:
                y = f(w0, inp.scales, inp.biases, inp.x, bits, gs)[0]
                if not np.allclose(y, expect, rtol=1e-12, atol=1e-14):
                    return False, f"q==0 closed form bits={bits} gs={gs}"
            # s == 0: bias-only, the same closed form
            s0 = np.zeros_like(inp.scales)
            for f in forms:
                y = f(w, s0, inp.biases, inp.x, bits, gs)[0]
                if not np.allclose(y, expect, rtol=1e-12, atol=1e-14):
                    return False, f"s==0 closed form bits={bits} gs={gs}"
            # one-hot x at column i: the dequantized column s*q + b, exactly
            for i in (0, 1, gs - 1, gs, K - 1):
                e = np.zeros((1, K), dtype=np.float32)
                e[0, i] = 1.0
                col = s[:, i // gs] * inp.q[:, i] + b[:, i // gs]
                for f in forms:
                    y = f(w, inp.scales, inp.biases, _bf16(e), bits, gs)[0]
                    if not np.array_equal(y, col):
                        return False, f"one-hot column {i} bits={bits} gs={gs}"
            # linearity in x (small integers are exact in bf16)
            rng = np.random.default_rng(bits * 1000 + gs)
            x1 = rng.integers(-8, 9, (1, K)).astype(np.float32)
            x2 = rng.integers(-8, 9, (1, K)).astype(np.float32)
            for f in forms:
                ya = f(w, inp.scales, inp.biases, _bf16(x1), bits, gs)
                yb = f(w, inp.scales, inp.biases, _bf16(x2), bits, gs)
                yab = f(w, inp.scales, inp.biases, _bf16(x1 + x2), bits, gs)
                T = o.abs_terms(w, inp.scales, inp.biases, _bf16(np.abs(x1) + np.abs(x2)), bits, gs)
                if not np.all(np.abs(yab - (ya + yb)) <= 1e-12 * T):
                    return False, f"linearity bits={bits} gs={gs}"
            # row permutation equivariance (rows are independent)
            perm = rng.permutation(N)
            for f in forms:
                y = f(w, inp.scales, inp.biases, inp.x, bits, gs)
                yp = f(w[perm], inp.scales[perm], inp.biases[perm], inp.x, bits, gs)
                if not np.array_equal(yp, y[:, perm]):
                    return False, f"row permutation bits={bits} gs={gs}"
    return True, "closed forms: x==1, q==0, s==0, one-hot x, linearity, row permutation"


def pin_f32_form(o):
    for N, K, M, bits, gs in _SHAPES:
        inp = _problem(N, K, M, bits, gs, 8)
        w = o.pack(inp.q, bits)
        yb, y32, _ = o.qmv_f32_factored(w, inp.scales, inp.biases, inp.x, bits, gs, nthreads=2, want_f32=True)
        ref = o.qmv_f64_dequant(w, inp.scales, inp.biases, inp.x, bits, gs)
        T = o.abs_terms(w, inp.scales, inp.biases, inp.x, bits, gs)
        # fp32 accumulation error is far below bf16 output rounding
        if not np.all(np.abs(y32 - ref) <= 1e-5 * T + 1e-7):
            return False, f"fp32 form vs fp64 {(N, K, M, bits, gs)}"
        rne = torch.from_numpy(y32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        if not np.array_equal(yb, rne):
            return False, f"fp32 form's bf16 output is not RNE of its fp32 value {(N, K, M, bits, gs)}"
    return True, "fp32 factored form within 1e-5*sum|wx| of fp64; bf16 output = RNE(fp32)"


# ----------------------------------------------------------------- mxfp4 --
# The fp mode: E2M1 codes, one E8M0 scale byte per 32 elements along K (the
# OCP MX v1.0 MXFP4 format, the reading taken for the pages' "mxfp4").
_MX_SHAPES = [(5, 32, 1), (6, 96, 2), (3, 256, 3), (4, 1024, 1)]


def _mx_decode_numpy(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dense fp64 weights through library decoders: ml_dtypes' float4_e2m1fn for
    the elements, torch's float8_e8m0fnu for the block scales."""
    import pytest
    ml_dtypes = pytest.importorskip("ml_dtypes")
    v = np.ascontiguousarray(codes, dtype=np.uint8).view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    sc = torch.from_numpy(np.ascontiguousarray(scales, dtype=np.uint8)).view(torch.float8_e8m0fnu)
    sc = sc.to(torch.float64).numpy()
    return v * np.repeat(sc, 32, axis=1)


def pin_mx_e2m1_value_set(o):
    """What the E2M1 layout fixes without any table: +0 at code 0, -0 at code 8,
    the sign bit negates exactly, magnitudes rise strictly with the code, the
    subnormal code 1 is half the smallest normal code 2, and each normal binade
    holds two values, the upper one 1.5 times the lower."""
    v = o.e2m1_to_f64(np.arange(16))
    if v[0] != 0.0 or np.signbit(v[0]) or v[8] != 0.0 or not np.signbit(v[8]):
        return False, f"zeros: {v[0]!r}, {v[8]!r}"
    if not np.array_equal(v[8:], -v[:8]):
        return False, f"sign bit does not negate: {v.tolist()}"
    if not np.all(np.diff(v[:8]) > 0):
        return False, f"magnitudes not increasing: {v[:8].tolist()}"
    if v[1] * 2 != v[2]:
        return False, f"subnormal {v[1]} is not half the smallest normal {v[2]}"
    for e in (1, 2, 3):
        lo, hi = v[2 * e], v[2 * e + 1]
        if hi != 1.5 * lo or (e > 1 and lo != 2 * v[2 * e - 2]):
            return False, f"binade {e}: {lo}, {hi}"
    return True, "E2M1 value set has the layout's structure"


def pin_mx_e2m1_vs_ml_dtypes(o):
    import pytest
    ml_dtypes = pytest.importorskip("ml_dtypes")
    ours = o.e2m1_to_f64(np.arange(16))
    ref = np.arange(16, dtype=np.uint8).view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    same = np.array_equal(ours, ref) and np.array_equal(np.signbit(ours), np.signbit(ref))
    return same, f"oracle {ours.tolist()} vs ml_dtypes {ref.tolist()}"


def pin_mx_e8m0_vs_torch(o):
    ours = o.e8m0_to_f64(np.arange(256))
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    same = np.array_equal(ours, ref, equal_nan=True) and np.isnan(ours[255])
    bad = np.nonzero(~((ours == ref) | (np.isnan(ours) & np.isnan(ref))))[0]
    return bool(same), f"{bad.size} of 256 scale bytes differ from torch float8_e8m0fnu (first {bad[:4].tolist()})"


def pin_mx_dequant_vs_numpy(o):
    for N, K, M in _MX_SHAPES:
        inp = synth.make_mxfp4_inputs(N, K, M, seed=5)
        w = o.pack(inp.codes, 4)
        y = o.mxfp4_qmv_f64(w, inp.scales, inp.x)
        T = o.mxfp4_abs_terms(w, inp.scales, inp.x)
        W = _mx_decode_numpy(inp.codes, inp.scales)
        ref = _f64(inp.x) @ W.T
        tref = np.abs(_f64(inp.x)) @ np.abs(W).T
        if not np.all(np.abs(y - ref) <= 1e-12 * tref + 1e-300):
            return False, f"mxfp4 dequant vs numpy {(N, K, M)}: max {np.max(np.abs(y - ref))}"
        if not np.allclose(T, tref, rtol=1e-12, atol=0):
            return False, f"mxfp4 abs terms vs numpy {(N, K, M)}"
    return True, "mxfp4 fp64 dequantize-then-dot agrees with numpy over library-decoded weights"


def pin_mx_fraction_bruteforce(o):
    """Exact rational sums over library-decoded weights on tiny shapes: the fp64
    oracle must sit within 1e-13 * sum|w x| of them."""
    for K in (32, 64, 160):
        inp = synth.make_mxfp4_inputs(3, K, 2, seed=50 + K)
        W = _mx_decode_numpy(inp.codes, inp.scales)
        xf = _f64(inp.x)
        w = o.pack(inp.codes, 4)
        y = o.mxfp4_qmv_f64(w, inp.scales, inp.x)
        T = o.mxfp4_abs_terms(w, inp.scales, inp.x)
        for m in range(2):
            for n in range(3):
                ex = sum((Fraction(float(W[n, i])) * Fraction(float(xf[m, i])) for i in range(K)), Fraction(0))
                if abs(Fraction(float(y[m, n])) - ex) > Fraction(1e-13) * Fraction(float(T[m, n])):
                    return False, f"mxfp4 brute force K={K} ({m},{n})"
    return True, "mxfp4 fp64 oracle matches exact rational arithmetic"


def pin_mx_closed_forms(o):
    import math
    N, K = 3, 128
    x = synth.make_mxfp4_inputs(1, K, 2, seed=6).x
    xf = _f64(x)
    ones = np.full((N, K), 0b0010, dtype=np.uint8)      # E2M1 +1.0
    unit = np.full((N, K // 32), 127, dtype=np.uint8)   # E8M0 2^0
    y = o.mxfp4_qmv_f64(o.pack(ones, 4), unit, x)
    for m in range(2):
        if not np.all(y[m] == math.fsum(xf[m].tolist())):
            return False, "codes +1.0 with unit scales must give sum(x)"
    zeros = np.where(np.arange(K) % 2 == 0, 0, 8).astype(np.uint8)[None].repeat(N, 0)
    if np.any(o.mxfp4_qmv_f64(o.pack(zeros, 4), unit, x) != 0.0):
        return False, "codes +-0 must give 0"
    inp = synth.make_mxfp4_inputs(N, K, 2, seed=7)
    w = o.pack(inp.codes, 4)
    y0 = o.mxfp4_qmv_f64(w, inp.scales, inp.x)
    # flipping every sign bit negates y exactly
    if not np.array_equal(o.mxfp4_qmv_f64(o.pack(inp.codes ^ 8, 4), inp.scales, inp.x), -y0):
        return False, "sign flip of every code must negate y"
    # one more in every scale exponent doubles y exactly
    if not np.array_equal(o.mxfp4_qmv_f64(w, inp.scales + 1, inp.x), 2 * y0):
        return False, "scale exponent + 1 must double y"
    # a scale byte of 255 (NaN) poisons its row only
    s = inp.scales.copy()
    s[1, 2] = 255
    yn = o.mxfp4_qmv_f64(w, s, inp.x)
    if not (np.all(np.isnan(yn[:, 1])) and np.array_equal(yn[:, [0, 2]], y0[:, [0, 2]])):
        return False, "scale byte 255 must make its row NaN and leave the others"
    # one-hot x reads one weight: scale * e2m1(code)
    v = o.e2m1_to_f64(np.arange(16))
    for k in (0, 31, 32, 77, K - 1):
        xk = np.zeros((1, K), dtype=np.uint16)
        xk[0, k] = 0x3F80  # bf16 1.0
        got = o.mxfp4_qmv_f64(w, inp.scales, xk)[0]
        want = v[inp.codes[:, k]] * np.ldexp(1.0, inp.scales[:, k // 32].astype(np.int64) - 127)
        if not np.array_equal(got, want):
            return False, f"one-hot x at {k}: {got} != {want}"
    return True, "mxfp4 closed forms: sum(x), zeros, sign flip, scale step, NaN scale, one-hot x"


PINS = {
    "bf16_rounding": pin_bf16_rounding,
    "bf16_widen": pin_bf16_widen,
    "golden_field_order": pin_golden_field_order,
    "floatfloor_exhaustive": pin_floatfloor_exhaustive,
    "pack_roundtrip": pin_pack_roundtrip,
    "dequant_vs_numpy": pin_dequant_vs_numpy,
    "factored_vs_dequant": pin_factored_vs_dequant,
    "fraction_bruteforce": pin_fraction_bruteforce,
    "closed_forms": pin_closed_forms,
    "f32_form": pin_f32_form,
    "mx_e2m1_value_set": pin_mx_e2m1_value_set,
    "mx_e2m1_vs_ml_dtypes": pin_mx_e2m1_vs_ml_dtypes,
    "mx_e8m0_vs_torch": pin_mx_e8m0_vs_torch,
    "mx_dequant_vs_numpy": pin_mx_dequant_vs_numpy,
    "mx_fraction_bruteforce": pin_mx_fraction_bruteforce,
    "mx_closed_forms": pin_mx_closed_forms,
}

MUTANTS = tuple(range(1, 12))
