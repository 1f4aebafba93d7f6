"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin takes an ``oracle.Oracle`` and returns ``(ok, detail)``. The pins use
library routines (torch's bf16 rounding, numpy's float64 matmul), exact
rational arithmetic (``fractions.Fraction``), closed forms of special cases,
the float-floor field chain of llama.cpp PR #159 "How", and hand-worked
fixtures of the field order (``tests/golden/field_order.txt``).

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
}

MUTANTS = tuple(range(1, 8))
