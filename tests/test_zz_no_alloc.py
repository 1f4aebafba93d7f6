"""qmv_run_noalloc: the entry point for callers that cannot allocate device
memory (pool-owned memory, latency-bound loops). It must give
the same output as the existing qmv_run_ex path, call after call, while its
scratch lives in a fixed array inside the library.

This file is collected last on purpose, so a failure here stops a
``-x`` run only after every other test has run."""

import numpy as np
import pytest
import torch

import group_quantized_mat_gb300 as g
import synth
from gpu_helpers import DeviceProblem, oracle_rows
from oracle import Oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from group_quantized_mat_gb300 import build
    build.build()
    return g.load()


# (N, K, M): the streamed kernel with a K split; a one-vector launch whose
# CTAs split K (its tickets live in the array and are cleared on the stream);
# more than 16 vectors, which run as two launches sharing the array.
CASES = [(3840, 15360, 13), (64, 65536, 1), (3840, 15360, 17)]


@pytest.mark.parametrize("N,K,M", CASES)
def test_noalloc_matches_existing_entry_point_twice(lib, N, K, M):
    bits, gs = 4, 64
    need = g.qmv_workspace_size(M, N, K, bits, gs)
    assert 0 < need <= g.NOALLOC_SCRATCH_BYTES  # this problem uses scratch
    inp = synth.make_inputs(N, K, M, bits, gs, seed=41 + M)
    dp = DeviceProblem(inp)

    ws = torch.zeros(need // 4 + 4, dtype=torch.int32, device="cuda")
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    g.qmv_run_ex(dp.w, dp.s, dp.b, dp.x, ref, M, N, K, bits, gs, workspace=ws, workspace_bytes=need)
    torch.cuda.synchronize()
    ref_bits = ref.cpu().numpy().view(np.uint16)

    rows = np.unique(np.concatenate([np.random.default_rng(5).choice(N, min(N, 64), replace=False), [0, N - 1]]))
    _, terms = oracle_rows(Oracle(0), inp, rows)
    y_ref = synth.bf16_bits_to_f32(ref_bits).astype(np.float64)

    outs = [torch.full((M, N), -1, dtype=torch.int16, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    free_before = None
    for call, y in enumerate(outs):
        code = lib.qmv_run_noalloc(dp.w.data_ptr(), dp.s.data_ptr(), dp.b.data_ptr(), dp.x.data_ptr(),
                                   y.data_ptr(), M, N, K, bits, gs, torch.cuda.current_stream().cuda_stream)
        assert code == 0, g.qmv_status_string(code)
        torch.cuda.synchronize()
        if call == 0:
            # the first call may load the kernels; the next one adds nothing
            free_before = torch.cuda.mem_get_info()[0]
        got_bits = y.cpu().numpy().view(np.uint16)
        got = synth.bf16_bits_to_f32(got_bits).astype(np.float64)
        # within the acceptance tolerance of the existing entry point's output ...
        assert np.all(np.abs(got[:, rows] - y_ref[:, rows]) <= 8e-3 * terms + 1e-5), f"call {call}"
        # ... and, since the arithmetic is the same, bit for bit
        assert np.array_equal(got_bits, ref_bits), f"call {call}"
    assert torch.cuda.mem_get_info()[0] == free_before, "a call took device memory"


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    N, K, M = 65536, 15360, 16
    assert g.qmv_workspace_size(M, N, K, 4, 64) > g.NOALLOC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first
    code = lib.qmv_run_noalloc(fake, fake, fake, fake, fake, M, N, K, 4, 64, None)
    assert code == 8, g.qmv_status_string(code)
