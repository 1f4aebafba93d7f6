"""Seeded synthetic inputs for group-quantized mat-vec (qmv): affine and mxfp4.

This module only draws random numbers. It holds none of the method's
arithmetic (no packing, no extraction, no dot products), so both the CUDA
path and the CPU oracle can take their inputs from it.

Distributions (the workloads of the group_quantized_mat pages; the pages
measure on trained checkpoints, which these stand in for):

* ``q``      uniform integers 0 .. 2**bits - 1, one per weight, ``uint8 [N, K]``
* ``scales`` fp32 U(0.001, 0.02) rounded to bf16, ``[N, K // group_size]``
* ``biases`` ``-2**(bits-1) * scale_bf16 + N(0, 1e-3)`` computed in fp32, rounded
  to bf16 (for 4-bit this is ``-8 * scale``, the integer midpoint; for 2-bit
  ``-2 * scale``), same shape as ``scales``
* ``x``      N(0, 1) rounded to bf16, ``[M, K]``

All bf16 arrays are returned as ``uint16`` bit patterns (numpy has no bf16).
Draw order is fixed: q, scales, bias noise, x, from one
``torch.Generator(device="cpu")`` seeded with ``seed``.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class QmvProblem:
    N: int
    K: int
    M: int
    bits: int
    group_size: int
    seed: int


@dataclass
class QmvInputs:
    problem: QmvProblem
    q: np.ndarray        # uint8  [N, K]   quantized fields, < 2**bits
    scales: np.ndarray   # uint16 [N, G]   bf16 bit patterns
    biases: np.ndarray   # uint16 [N, G]   bf16 bit patterns
    x: np.ndarray        # uint16 [M, K]   bf16 bit patterns


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def make_weights(N: int, K: int, bits: int, group_size: int, seed: int):
    """q, scales, biases for one weight matrix (see module docstring)."""
    if K % group_size:
        raise ValueError("K must be a multiple of group_size")
    G = K // group_size
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randint(0, 1 << bits, (N, K), generator=g, dtype=torch.uint8)
    s32 = torch.rand((N, G), generator=g, dtype=torch.float32) * (0.02 - 0.001) + 0.001
    s_bf = s32.to(torch.bfloat16)
    noise = torch.randn((N, G), generator=g, dtype=torch.float32) * 1e-3
    b32 = -float(1 << (bits - 1)) * s_bf.to(torch.float32) + noise
    return q.numpy().copy(), _bf16_bits(s_bf), _bf16_bits(b32), g


def make_activations(M: int, K: int, seed: int, generator: torch.Generator | None = None):
    g = generator if generator is not None else torch.Generator(device="cpu").manual_seed(int(seed))
    x = torch.randn((M, K), generator=g, dtype=torch.float32)
    return _bf16_bits(x)


def make_inputs(N: int, K: int, M: int, bits: int = 4, group_size: int = 64, seed: int = 0) -> QmvInputs:
    q, s, b, g = make_weights(N, K, bits, group_size, seed)
    x = make_activations(M, K, seed, generator=g)
    return QmvInputs(QmvProblem(N, K, M, bits, group_size, seed), q, s, b, x)


@dataclass
class MxInputs:
    N: int
    K: int
    M: int
    seed: int
    codes: np.ndarray    # uint8  [N, K]      E2M1 codes, 0 .. 15
    scales: np.ndarray   # uint8  [N, K // 32] E8M0 exponent bytes
    x: np.ndarray        # uint16 [M, K]      bf16 bit patterns


def make_mxfp4_inputs(N: int, K: int, M: int, seed: int = 0, scale_lo: int = 118, scale_hi: int = 122) -> MxInputs:
    """Seeded inputs of the mxfp4 mode (E2M1 codes, one E8M0 byte per 32 along K).

    * ``codes``  uniform over all 16 E2M1 codes (both zeros, both signs, up to +-6)
    * ``scales`` uniform integer exponent bytes in [scale_lo, scale_hi] (2^-9 .. 2^-5
      by default: weights up to about 0.19 in magnitude, as for a checkpoint's
      projection matrices)
    * ``x``      N(0, 1) rounded to bf16

    Draw order: codes, scales, x, from one ``torch.Generator(device="cpu")``.
    """
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    codes = torch.randint(0, 16, (N, K), generator=g, dtype=torch.uint8)
    scales = torch.randint(scale_lo, scale_hi + 1, (N, K // 32), generator=g, dtype=torch.int32).to(torch.uint8)
    x = make_activations(M, K, seed, generator=g)
    return MxInputs(N, K, M, seed, codes.numpy().copy(), scales.numpy().copy(), x)


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact: bf16 is the top half of binary32)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


# The workloads named for this method, by what they are.
WORKLOADS = {
    # tiny parity case: 256 x 1024, 4-bit, group 64, one vector
    "tiny_256x1024_4b_g64": dict(N=256, K=1024, bits=4, group_size=64, Ms=(1,)),
    # 12B-class decode up/gate projection
    "proj_15360x3840_4b_g64": dict(N=15360, K=3840, bits=4, group_size=64, Ms=(1, 2, 4, 5, 10, 13, 16)),
    # 12B-class down projection
    "down_3840x15360_4b_g64": dict(N=3840, K=15360, bits=4, group_size=64, Ms=(1, 2, 4, 5, 10, 13, 16)),
    # 27B-class layer stack
    "l27b_5120x5120_4b_g64": dict(N=5120, K=5120, bits=4, group_size=64, Ms=(1, 13)),
    "l27b_1024x5120_4b_g64": dict(N=1024, K=5120, bits=4, group_size=64, Ms=(1, 13)),
    "l27b_17408x5120_4b_g64": dict(N=17408, K=5120, bits=4, group_size=64, Ms=(1, 13)),
    "l27b_5120x17408_4b_g64": dict(N=5120, K=17408, bits=4, group_size=64, Ms=(1, 13)),
    # 2-bit variant of the projection
    "proj_15360x3840_2b_g64": dict(N=15360, K=3840, bits=2, group_size=64, Ms=(1, 13)),
    "proj_15360x3840_2b_g128": dict(N=15360, K=3840, bits=2, group_size=128, Ms=(1, 13)),
}

# The same shapes in the mxfp4 mode (E2M1 codes, 32-element E8M0 blocks).
MX_WORKLOADS = {
    "proj_15360x3840_mxfp4": dict(N=15360, K=3840, Ms=(1, 13)),
    "down_3840x15360_mxfp4": dict(N=3840, K=15360, Ms=(1, 13)),
}
