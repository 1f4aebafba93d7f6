"""GPU tests through the C ABI: parity with the CPU oracle and bitwise
identity of the streamed kernel's columns with the M = 1 kernel.

Acceptance (per output element): |y_gpu - y_oracle| <= 8e-3 * sum_i |w_i x_i| + 1e-5,
y_oracle the fp64 dequantize-then-dot form. Streamed columns must equal the
M = 1 result bit for bit (mlxcel issue #1289, "The observation this rests on":
"bit-identical to qmv at M = 1 by construction, not by tolerance").
"""

import numpy as np
import pytest
import torch

import group_quantized_mat_gb300 as g
import synth
from gpu_helpers import DeviceProblem, check_parity, dev, oracle_rows
from oracle import Oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from group_quantized_mat_gb300 import build
    build.build()
    g.load()
    yield
    assert g.qmv_device_error() == 0, "a kernel reported a timed-out wait"


@pytest.fixture(scope="module")
def o():
    return Oracle(0)


# ----------------------------------------------------------- full parity --
# Sizes the oracle finishes in seconds that span several row blocks, several
# K-chunks and ragged tails (N not a multiple of 8; partial last stage).
MEDIUM = [
    (256, 1024, 1, 4, 64),      # the tiny workload
    (200, 3840, 3, 4, 64),      # K of the 12B projection: 2 chunks, 7.5 stages
    (130, 15360, 2, 4, 64),     # K of the down projection: 8 chunks
    (77, 5120, 16, 4, 64),      # widest M
    (90, 3840, 14, 4, 64),      # two passes, each its own work item
    (300, 3840, 13, 2, 64),
    (150, 3840, 5, 2, 128),
    (129, 2048, 4, 4, 128),
    (9, 384, 1, 4, 128),        # one partial box per row
    (1, 64, 1, 4, 64),          # a single group and a single row
    (65, 128, 7, 2, 128),
    (64, 17408, 2, 4, 64),      # 9 chunks, the last one short
]


@pytest.mark.parametrize("N,K,M,bits,gs", MEDIUM)
def test_parity_full_output(o, N, K, M, bits, gs):
    inp = synth.make_inputs(N, K, M, bits, gs, seed=N + K + M)
    dp = DeviceProblem(inp)
    y = dp.run()
    ref, terms = oracle_rows(o, inp)
    check_parity(y, ref, terms, f"{(N, K, M, bits, gs)}")
    # the fp32 value before rounding is far closer than the bf16 tolerance
    y32 = dp.run(flags=g.F32_OUT)
    assert np.all(np.abs(y32 - ref) <= 1e-4 * terms + 1e-6)
    # and the bf16 output is its round-to-nearest-even
    rne = torch.from_numpy(y32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(rne, y)


# ----------------------------------------------------------- full sizes --
# Every workload at its full size, in the launch configuration the bench
# times; every output element is checked against the oracle.
FULL = [
    ("proj_15360x3840_4b_g64", 1), ("proj_15360x3840_4b_g64", 13),
    ("down_3840x15360_4b_g64", 1), ("down_3840x15360_4b_g64", 16),
    ("l27b_5120x5120_4b_g64", 13), ("l27b_1024x5120_4b_g64", 1),
    ("l27b_17408x5120_4b_g64", 1), ("l27b_5120x17408_4b_g64", 13),
    ("proj_15360x3840_2b_g64", 13), ("proj_15360x3840_2b_g128", 1),
]


@pytest.mark.parametrize("name,M", FULL)
def test_parity_full_size_all_rows(o, name, M):
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w["N"], w["K"], M, w["bits"], w["group_size"], seed=0)
    y = DeviceProblem(inp).run()
    ref, terms = oracle_rows(o, inp)
    check_parity(y, ref, terms, f"{name} M={M}")


# Rows whose four-row unit is 8-10 KB go to the ring (one copy of whole rows)
# when every consumer warp gets two units, else to the direct-load kernel: both
# sides of that rule, at 4 and 2 bits, every row against the oracle.
@pytest.mark.parametrize("N,K,bits,gs", [(9728, 9216, 2, 64), (12288, 5120, 4, 128), (2048, 4608, 4, 64)])
def test_parity_long_whole_row_units(o, N, K, bits, gs):
    inp = synth.make_inputs(N, K, 1, bits, gs, seed=N + K)
    y = DeviceProblem(inp).run()
    ref, terms = oracle_rows(o, inp)
    check_parity(y, ref, terms, f"{N}x{K} {bits}-bit g{gs}")


# ------------------------------------------------------- bit identity --
IDENT = [
    (15360, 3840, 4, 64), (3840, 15360, 4, 64), (1000, 5120, 4, 64),
    (15360, 3840, 2, 64), (15360, 3840, 2, 128), (333, 1024, 4, 128),
]


@pytest.mark.parametrize("N,K,bits,gs", IDENT)
def test_streamed_columns_bit_identical_to_m1(N, K, bits, gs):
    inp = synth.make_inputs(N, K, 16, bits, gs, seed=7)
    dp = DeviceProblem(inp)
    singles_bf = np.stack([dp.run(x=dp.x[m:m + 1].contiguous(), M=1)[0] for m in range(16)])
    singles_32 = np.stack([dp.run(x=dp.x[m:m + 1].contiguous(), M=1, flags=g.F32_OUT)[0] for m in range(16)])
    # every pass structure: one pass (2..8), two unequal (9, 13), two equal in
    # one work item (10), two equal passes as separate work items (14, 16)
    for M in (2, 4, 5, 9, 10, 13, 14, 16):
        x = dp.x[:M].contiguous()
        y_bf = dp.run(x=x, M=M)
        y_32 = dp.run(x=x, M=M, flags=g.F32_OUT)
        assert np.array_equal(y_bf, singles_bf[:M]), f"M={M}: bf16 columns differ from M=1"
        assert np.array_equal(y_32.view(np.uint32), singles_32[:M].view(np.uint32)), f"M={M}: fp32 columns differ"
        per_col = dp.run(x=x, M=M, flags=g.F32_OUT | g.FORCE_M1_PER_COLUMN)
        assert np.array_equal(per_col.view(np.uint32), y_32.view(np.uint32))


def _wide_range_x(M: int, K: int, seed: int) -> np.ndarray:
    """bf16 x whose subgroups mix a large element with ones up to 240 binades
    smaller, around the point (231 binades) past which the staging makes an
    element a zero of its sign."""
    rng = np.random.default_rng(seed)
    top = rng.integers(236, 246, size=(M, K // 64))
    gap = rng.choice(np.array([0, 1, 3, 7, 100, 200, 228, 229, 230, 231, 232, 233, 234, 236, 238, 240]), size=(M, K))
    ex = np.clip(np.repeat(top, 64, axis=1) - gap, 0, 254)
    ex[:, ::64] = np.repeat(top[:, :, None], 1, axis=2)[:, :, 0]   # the subgroup's largest
    mant = rng.integers(0, 128, size=(M, K))
    sign = rng.integers(0, 2, size=(M, K))
    return ((sign << 15) | (ex << 7) | mant).astype(np.uint16)


@pytest.mark.parametrize("bits", [4, 2])
def test_wide_exponent_range(o, bits):
    """Subgroups spanning more than 231 binades: the two field readings still
    agree bit for bit, and the result stays within the tolerance."""
    N, K = 96, 4096
    inp = synth.make_inputs(N, K, 6, bits, 64, seed=31)
    inp.x = _wide_range_x(6, K, 5 + bits)
    dp = DeviceProblem(inp)
    y6 = dp.run(flags=g.F32_OUT)
    singles = np.stack([dp.run(x=dp.x[m:m + 1].contiguous(), M=1, flags=g.F32_OUT)[0] for m in range(6)])
    assert np.array_equal(y6.view(np.uint32), singles.view(np.uint32))
    assert np.array_equal(dp.run(), np.stack([dp.run(x=dp.x[m:m + 1].contiguous(), M=1)[0] for m in range(6)]))
    ref, terms = oracle_rows(o, inp)
    assert np.all(np.abs(y6 - ref) <= 1e-4 * terms + 1e-6)


@pytest.mark.parametrize("M", [17, 20, 33])
def test_more_than_sixteen_vectors(o, M):
    """M above 16 runs in launches of 16 and the remainder: every column still
    equals the M = 1 result bit for bit and meets the tolerance."""
    N, K = 700, 3840
    inp = synth.make_inputs(N, K, M, 4, 64, seed=40 + M)
    dp = DeviceProblem(inp)
    y = dp.run(flags=g.F32_OUT)
    singles = np.stack([dp.run(x=dp.x[m:m + 1].contiguous(), M=1, flags=g.F32_OUT)[0] for m in range(M)])
    assert np.array_equal(y.view(np.uint32), singles.view(np.uint32))
    ref, terms = oracle_rows(o, inp)
    check_parity(dp.run(), ref, terms, f"M={M}")


@pytest.mark.parametrize("N,K,bits,gs", [
    (15360, 3840, 4, 64),   # whole-row units, one metadata box per unit
    (3840, 15360, 4, 64),   # 2-D tile units
    (100, 4160, 4, 64),     # per-row pieces (G = 65)
    (300, 3840, 2, 128),
    (70, 11264, 4, 128),    # G = 88: tiles
])
def test_interleaved_metadata_gives_identical_results(o, N, K, bits, gs):
    """QMV_SB_INTERLEAVED changes how scales and biases travel, not the
    arithmetic: the results equal the separate layout's bit for bit, and the
    interleaved call's bf16 output meets the oracle's tolerance."""
    inp = synth.make_inputs(N, K, 13, bits, gs, seed=60 + K)
    dp = DeviceProblem(inp)
    sb = dev(g.qmv_pack_sb(inp.scales, inp.biases))
    ref, terms = oracle_rows(o, inp)
    for M in (1, 4, 13):
        x = dp.x[:M].contiguous()
        want = dp.run(x=x, M=M, flags=g.F32_OUT)
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        g.qmv_run_ex(dp.w, sb, None, x, y, M, N, K, bits, gs, flags=g.F32_OUT | g.SB_INTERLEAVED)
        yb = torch.empty((M, N), dtype=torch.int16, device="cuda")
        g.qmv_run_ex(dp.w, sb, None, x, yb, M, N, K, bits, gs, flags=g.SB_INTERLEAVED)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32)), f"M={M}"
        # the interleaved layout's own output against the oracle
        check_parity(yb.cpu().numpy().view(np.uint16), ref[:M], terms[:M], f"interleaved {N}x{K} M={M}")


@pytest.mark.parametrize("M,N,K", [(1, 15360, 3840), (4, 2048, 3840), (13, 3840, 15360), (20, 1000, 5120)])
def test_pdl_launches_wait_for_the_producer_of_x(M, N, K):
    """With QMV_PDL a launch may start while the preceding kernel runs; x is
    written by exactly such a kernel here, so reading it before the
    dependency wait would give other results than the plain launch."""
    inp = synth.make_inputs(N, K, M, 4, 64, seed=70 + M)
    dp = DeviceProblem(inp)
    rng = np.random.default_rng(M)
    xs = [dp.x[rng.permutation(M)].contiguous() for _ in range(4)]
    want = [dp.run(x=x, flags=g.F32_OUT) for x in xs]
    x_buf = torch.empty_like(dp.x)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for x in xs:
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            x_buf.zero_()
            x_buf.copy_(x)  # the kernel right before the call writes x
            g.qmv_run_ex(dp.w, dp.s, dp.b, x_buf, y, M, N, K, 4, 64, flags=g.F32_OUT | g.PDL, stream=s)
            outs.append(y)
    torch.cuda.synchronize()
    for got, ref in zip(outs, want):
        assert np.array_equal(got.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("case", ["x_zero", "s_zero", "q_zero", "q_max"])
def test_degenerate_inputs(o, case):
    """The method's degenerate cases: zero activations (y = 0), zero scales
    (bias terms only), all-zero and all-maximum fields. Parity with the
    oracle, and streamed columns equal to M = 1 bit for bit."""
    N, K = 260, 5120
    inp = synth.make_inputs(N, K, 4, 4, 64, seed=81)
    if case == "x_zero":
        inp.x = np.zeros_like(inp.x)
    elif case == "s_zero":
        inp.scales = np.zeros_like(inp.scales)
    elif case == "q_zero":
        inp.q = np.zeros_like(inp.q)
    else:
        inp.q = np.full_like(inp.q, 15)
    dp = DeviceProblem(inp)
    y = dp.run(flags=g.F32_OUT)
    singles = np.stack([dp.run(x=dp.x[m:m + 1].contiguous(), M=1, flags=g.F32_OUT)[0] for m in range(4)])
    assert np.array_equal(y.view(np.uint32), singles.view(np.uint32))
    ref, terms = oracle_rows(o, inp)
    check_parity(dp.run(), ref, terms, case)
    if case == "x_zero":
        assert np.all(y == 0.0)


@pytest.mark.parametrize("M", [1, 3])
def test_long_rows(o, M):
    """K = 2^22: thousands of chunks per row, hundreds of K-ranges meeting in
    the workspace."""
    N, K = 5, 1 << 22
    inp = synth.make_inputs(N, K, M, 4, 64, seed=90 + M)
    dp = DeviceProblem(inp)
    y = dp.run(flags=g.F32_OUT)
    if M > 1:
        singles = np.stack([dp.run(x=dp.x[m:m + 1].contiguous(), M=1, flags=g.F32_OUT)[0] for m in range(M)])
        assert np.array_equal(y.view(np.uint32), singles.view(np.uint32))
    ref, terms = oracle_rows(o, inp)
    check_parity(dp.run(), ref, terms, f"K=2^22 M={M}")


def test_position_invariance():
    inp = synth.make_inputs(3840, 3840, 13, 4, 64, seed=11)
    dp = DeviceProblem(inp)
    x = dp.x
    perm = list(range(1, 13)) + [0]          # vector 0 moves to the last column
    ya = dp.run(x=x, M=13, flags=g.F32_OUT)
    yb = dp.run(x=x[perm].contiguous(), M=13, flags=g.F32_OUT)
    assert np.array_equal(ya[0].view(np.uint32), yb[12].view(np.uint32))
    assert np.array_equal(ya[perm].view(np.uint32), yb.view(np.uint32))


def test_mutated_order_is_detected(o, tmp_path):
    """A build whose streamed kernel folds in a different order still passes
    the tolerance, and the bit-identity check must reject it."""
    from group_quantized_mat_gb300 import build
    path = build.build(extra_defines=("QMV_TEST_MUTATE_ORDER=1",),
                       out=str(build.LIB).replace("libqmv.so", "libqmv_mutant.so"))
    mut = g.load(path)
    inp = synth.make_inputs(512, 3840, 4, 4, 64, seed=3)
    dp = DeviceProblem(inp)
    y4 = dp.run(M=4, flags=g.F32_OUT, lib=mut)
    singles = np.stack([dp.run(x=dp.x[m:m + 1].contiguous(), M=1, flags=g.F32_OUT, lib=mut)[0] for m in range(4)])
    ref, terms = oracle_rows(o, inp)
    assert np.all(np.abs(y4 - ref) <= 1e-4 * terms + 1e-6)
    assert not np.array_equal(y4.view(np.uint32), singles.view(np.uint32))


# ----------------------------------------------------------- workspace --
def test_explicit_workspace_matches_library_workspace():
    inp = synth.make_inputs(1000, 15360, 13, 4, 64, seed=5)
    dp = DeviceProblem(inp)
    y_lib = dp.run(flags=g.F32_OUT)
    nbytes = g.qmv_workspace_size(13, 1000, 15360, 4, 64)
    assert nbytes > 0
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.int32, device="cuda")
    g.qmv_workspace_init(ws, nbytes)
    for _ in range(3):  # the counters return to zero after every call
        y = dp.run(flags=g.F32_OUT, workspace=ws, workspace_bytes=nbytes)
        assert np.array_equal(y.view(np.uint32), y_lib.view(np.uint32))
    with pytest.raises(g.QmvError) as e:
        dp.run(flags=g.F32_OUT, workspace=ws, workspace_bytes=nbytes - 4)
    assert e.value.code == 8


def test_streams_and_back_to_back_calls():
    """Different problems alternating on one stream share the library workspace."""
    a = DeviceProblem(synth.make_inputs(640, 15360, 3, 4, 64, seed=1))
    b = DeviceProblem(synth.make_inputs(700, 3840, 9, 4, 64, seed=2))
    ya, yb = a.run(), b.run()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            assert np.array_equal(a.run(), ya)
            assert np.array_equal(b.run(), yb)


def test_cuda_graph_capture_replays_identically():
    dp = DeviceProblem(synth.make_inputs(2048, 3840, 5, 4, 64, seed=4))
    y_ref = dp.run()  # first call sizes the library workspace outside capture
    y = torch.empty((5, 2048), dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            g.qmv_run(dp.w, dp.s, dp.b, dp.x, y, 5, 2048, 3840, 4, 64, stream=s)
    for _ in range(3):
        y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().view(np.uint16), y_ref)


def test_workspace_serves_any_shape_sequence():
    """One workspace, problems of different N / K / M in turn: every call must
    match a fresh-workspace result whatever the workspace held before."""
    probs = [DeviceProblem(synth.make_inputs(3840, 15360, 16, 4, 64, seed=21)),
             DeviceProblem(synth.make_inputs(5120, 5120, 13, 4, 64, seed=22)),
             DeviceProblem(synth.make_inputs(1000, 3840, 3, 2, 128, seed=23))]
    need = max(g.qmv_workspace_size(p.M, p.N, p.K, p.bits, p.gs) for p in probs)
    refs = []
    for p in probs:
        nb = g.qmv_workspace_size(p.M, p.N, p.K, p.bits, p.gs)
        fresh = torch.zeros(nb // 4 + 4, dtype=torch.int32, device="cuda")
        refs.append(p.run(flags=g.F32_OUT, workspace=fresh, workspace_bytes=nb))
    # the workspace is scratch: garbage left in it (here, random words) must
    # not change any result
    ws = torch.randint(-2**31, 2**31 - 1, (need // 4 + 4,), dtype=torch.int32, device="cuda")
    for rnd in range(2):
        for p, ref in zip(probs, refs):
            y = p.run(flags=g.F32_OUT, workspace=ws, workspace_bytes=need)
            assert np.array_equal(y.view(np.uint32), ref.view(np.uint32)), f"round {rnd} N={p.N}"
        ws.random_(-2**31, 2**31 - 1)
