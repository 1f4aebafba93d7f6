"""GPU tests of the mxfp4 mode through the C ABI (qmv_mxfp4_run): parity with
the CPU oracle's fp64 dequantize-then-dot, and bitwise identity of every
column of an M-vector call with the M = 1 call on that column.

Acceptance per output element, as for the affine mode:
|y_gpu - y_oracle| <= 8e-3 * sum_i |w_i x_i| + 1e-5 for bf16 output; the fp32
output (QMV_F32_OUT) is held to 1e-5 * sum_i |w_i x_i| (the fp32 summation
error of at most ~60 roundings of sums bounded by that scale).
"""

import numpy as np
import pytest
import torch

import group_quantized_mat_gb300 as g
import synth
from gpu_helpers import dev, threaded_rows
from oracle import Oracle, tolerance_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from group_quantized_mat_gb300 import build
    build.build()
    g.load()


@pytest.fixture(scope="module")
def o():
    return Oracle(0)


class MxDevice:
    """Seeded mxfp4 inputs packed by the library codec and resident on the GPU."""

    def __init__(self, inp: synth.MxInputs):
        self.inp = inp
        self.N, self.K, self.M = inp.N, inp.K, inp.M
        self.w = dev(g.qmv_pack(inp.codes, 4))
        self.s = torch.from_numpy(np.ascontiguousarray(inp.scales)).cuda()
        self.x = dev(inp.x)

    def run(self, x=None, M=None, flags=0) -> np.ndarray:
        x = self.x if x is None else x
        M = self.M if M is None else M
        f32 = bool(flags & g.F32_OUT)
        y = torch.empty((M, self.N), dtype=torch.float32 if f32 else torch.int16, device="cuda")
        g.qmv_mxfp4_run(self.w, self.s, x, y, M, self.N, self.K, flags=flags)
        torch.cuda.synchronize()
        out = y.cpu().numpy()
        return out if f32 else out.view(np.uint16)


def oracle_rows(o, inp, rows=None, codes=None, scales=None, x=None):
    codes = inp.codes if codes is None else codes
    scales = inp.scales if scales is None else scales
    x = inp.x if x is None else x
    if rows is not None:
        codes, scales = codes[rows], scales[rows]
    w = o.pack(codes, 4)
    return o.mxfp4_qmv_f64(w, scales, x), o.mxfp4_abs_terms(w, scales, x)


def check(y_bits, y_ref, terms, what):
    y = synth.bf16_bits_to_f32(y_bits).astype(np.float64)
    ok, worst = tolerance_ok(y, y_ref, terms)
    assert ok, f"{what}: worst |dy| / (8e-3*sum|wx| + 1e-5) = {worst:.3f}"


# Sizes the oracle finishes in seconds: one and several 1024-element K-chunks
# (a short last chunk), row counts that leave the last 32-row CTA partial, and
# every launch-width regime (1, 2..4, 5..8, 9..16, and M > 16 in two launches).
MEDIUM = [
    (37, 32, 1),        # a single block per row, 37 rows (two CTAs, the second with 5 rows)
    (64, 1056, 3),      # two chunks, the second one block long
    (100, 3072, 5),     # three whole chunks
    (33, 3840, 13),     # K of the 12B projection: 4 chunks, the last 24 blocks long
    (70, 2080, 16),     # widest launch
    (20, 1024, 17),     # launches of 16 and 1
    (9, 4096, 33),      # launches of 16, 16 and 1
    (1, 64, 8),         # one row
    (250, 15360, 2),    # K of the down projection
]


@pytest.mark.parametrize("N,K,M", MEDIUM)
def test_mxfp4_parity_full_output(o, N, K, M):
    inp = synth.make_mxfp4_inputs(N, K, M, seed=N * 7 + K + M)
    d = MxDevice(inp)
    y = d.run()
    y_ref, terms = oracle_rows(o, inp)
    check(y, y_ref, terms, f"mxfp4 {N}x{K} M={M}")


@pytest.mark.parametrize("N,K,M", [(100, 3072, 5), (33, 3840, 13)])
def test_mxfp4_f32_output(o, N, K, M):
    inp = synth.make_mxfp4_inputs(N, K, M, seed=3)
    d = MxDevice(inp)
    y32 = d.run(flags=g.F32_OUT)
    y_ref, terms = oracle_rows(o, inp)
    err = np.abs(y32.astype(np.float64) - y_ref)
    assert np.all(err <= 1e-5 * terms), f"worst {np.max(err / terms):.3g} of sum|wx|"
    # the bf16 output is the nearest-even rounding of the fp32 value
    yb = d.run()
    rne = torch.from_numpy(y32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(yb, rne)


@pytest.mark.parametrize("M", [2, 3, 4, 5, 8, 9, 13, 16, 20])
def test_mxfp4_columns_bit_identical_to_one_vector(M):
    """Column j of an M-vector call equals the M = 1 call on x[j], bit for bit
    (fp32 output, so that no rounding to bf16 can hide a difference)."""
    inp = synth.make_mxfp4_inputs(96, 3840, M, seed=40 + M)
    d = MxDevice(inp)
    y = d.run(flags=g.F32_OUT)
    for j in range(M):
        yj = d.run(x=d.x[j:j + 1].contiguous(), M=1, flags=g.F32_OUT)
        assert np.array_equal(y[j].view(np.uint32), yj[0].view(np.uint32)), f"column {j} of M={M}"
    # and the library's own per-column mode agrees
    yf = d.run(flags=g.F32_OUT | g.FORCE_M1_PER_COLUMN)
    assert np.array_equal(y.view(np.uint32), yf.view(np.uint32))


def test_mxfp4_special_values(o):
    N, K, M = 40, 2048, 3
    inp = synth.make_mxfp4_inputs(N, K, M, seed=11)
    codes, scales = inp.codes.copy(), inp.scales.copy()
    codes[0] = np.where(np.arange(K) % 2 == 0, 0, 8)   # +0 / -0 everywhere: y = 0
    scales[1, 5] = 255                                  # NaN scale: the row is NaN
    scales[2] = 0                                       # 2^-127: tiny but finite
    scales[3] = 140                                     # 2^13: large but finite
    codes[4] = 0b0111                                   # +6 everywhere
    codes[5] = 0b1111                                   # -6 everywhere, with row 4's scales
    scales[5] = scales[4]
    d = MxDevice(synth.MxInputs(N, K, M, 11, codes, scales, inp.x))
    y32 = d.run(flags=g.F32_OUT)
    assert np.all(y32[:, 0] == 0.0)
    assert np.all(np.isnan(y32[:, 1]))
    y_ref, terms = oracle_rows(o, inp, codes=codes, scales=scales)
    keep = np.ones(N, dtype=bool)
    keep[1] = False
    err = np.abs(y32[:, keep].astype(np.float64) - y_ref[:, keep])
    assert np.all(err <= 1e-5 * terms[:, keep] + 1e-44)
    assert np.array_equal(y32[:, 4], -y32[:, 5])


def test_mxfp4_one_hot_x_reads_single_weights(o):
    N, K = 64, 1024
    inp = synth.make_mxfp4_inputs(N, K, 1, seed=12)
    ks = [0, 1, 31, 32, 33, 511, 1000, 1023]
    x = np.zeros((len(ks), K), dtype=np.uint16)
    for j, k in enumerate(ks):
        x[j, k] = 0x3F80  # bf16 1.0
    d = MxDevice(inp)
    y32 = d.run(x=dev(x), M=len(ks), flags=g.F32_OUT)
    vals = o.e2m1_to_f64(np.arange(16))
    for j, k in enumerate(ks):
        want = vals[inp.codes[:, k]] * np.ldexp(1.0, inp.scales[:, k // 32].astype(np.int64) - 127)
        assert np.array_equal(y32[j].astype(np.float64), want), f"one-hot x at {k}"


@pytest.mark.parametrize("N,K,M", [(15360, 3840, 1), (15360, 3840, 13), (3840, 15360, 13)])
def test_mxfp4_full_size_all_rows(o, N, K, M):
    """The bench's shapes: every output element against the oracle (computed
    over row slices on host threads)."""
    inp = synth.make_mxfp4_inputs(N, K, M, seed=21)
    d = MxDevice(inp)
    y = d.run()
    w = o.pack(inp.codes, 4)
    y_ref = threaded_rows(lambda lo, hi: o.mxfp4_qmv_f64(w[lo:hi], inp.scales[lo:hi], inp.x), N, M)
    terms = threaded_rows(lambda lo, hi: o.mxfp4_abs_terms(w[lo:hi], inp.scales[lo:hi], inp.x), N, M)
    check(y, y_ref, terms, f"mxfp4 {N}x{K} M={M}")


@pytest.mark.parametrize("M", [1, 3])
def test_mxfp4_long_rows(o, M):
    """K = 2^22: 4096 chunks per row; every column still equals its one-vector
    call bit for bit."""
    N, K = 5, 1 << 22
    inp = synth.make_mxfp4_inputs(N, K, M, seed=90 + M)
    d = MxDevice(inp)
    y = d.run(flags=g.F32_OUT)
    if M > 1:
        singles = np.stack([d.run(x=d.x[m:m + 1].contiguous(), M=1, flags=g.F32_OUT)[0] for m in range(M)])
        assert np.array_equal(y.view(np.uint32), singles.view(np.uint32))
    y_ref, terms = oracle_rows(o, inp)
    check(d.run(), y_ref, terms, f"mxfp4 K=2^22 M={M}")


def test_mxfp4_graph_capture_replays_identically():
    inp = synth.make_mxfp4_inputs(512, 3840, 13, seed=30)
    d = MxDevice(inp)
    ref = d.run()
    y = torch.empty((13, 512), dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.qmv_mxfp4_run(d.w, d.s, d.x, y, 13, 512, 3840, stream=s)  # warm-up outside the capture
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            g.qmv_mxfp4_run(d.w, d.s, d.x, y, 13, 512, 3840, stream=s)
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint16), ref)
