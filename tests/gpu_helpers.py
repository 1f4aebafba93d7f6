"""Helpers for the GPU tests: device buffers from seeded inputs, calls through
the C ABI, and oracle references for selected rows."""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import group_quantized_mat_gb300 as g
import synth
from oracle import Oracle, tolerance_ok


def dev(a: np.ndarray) -> torch.Tensor:
    """numpy -> CUDA tensor with the same bytes (uint16/uint32 viewed as signed)."""
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class DeviceProblem:
    """Seeded inputs packed by the library codec and resident on the GPU."""

    def __init__(self, inp: synth.QmvInputs):
        self.inp = inp
        pr = inp.problem
        self.N, self.K, self.M, self.bits, self.gs = pr.N, pr.K, pr.M, pr.bits, pr.group_size
        self.w_host = g.qmv_pack(inp.q, pr.bits)
        self.w = dev(self.w_host)
        self.s = dev(inp.scales)
        self.b = dev(inp.biases)
        self.x = dev(inp.x)

    def run(self, x: torch.Tensor | None = None, M: int | None = None, flags: int = 0, workspace=None,
            workspace_bytes: int = 0, lib=None) -> np.ndarray:
        x = self.x if x is None else x
        M = self.M if M is None else M
        f32 = bool(flags & g.F32_OUT)
        y = torch.empty((M, self.N), dtype=torch.float32 if f32 else torch.int16, device="cuda")
        if lib is None:
            if flags == 0 and workspace is None:
                g.qmv_run(self.w, self.s, self.b, x, y, M, self.N, self.K, self.bits, self.gs)
            else:
                g.qmv_run_ex(self.w, self.s, self.b, x, y, M, self.N, self.K, self.bits, self.gs,
                             workspace=workspace, workspace_bytes=workspace_bytes, flags=flags)
        else:
            code = lib.qmv_run_ex(self.w.data_ptr(), self.s.data_ptr(), self.b.data_ptr(), x.data_ptr(),
                                  y.data_ptr(), M, self.N, self.K, self.bits, self.gs, None, 0, flags,
                                  torch.cuda.current_stream().cuda_stream)
            assert code == 0, g.qmv_status_string(code)
        torch.cuda.synchronize()
        out = y.cpu().numpy()
        return out if f32 else out.view(np.uint16)


def row_slices(n: int, parts: int):
    """[lo, hi) bounds splitting n rows into at most `parts` contiguous slices."""
    step = max(1, -(-n // parts))
    return [(lo, min(n, lo + step)) for lo in range(0, n, step)]


def threaded_rows(fn, n: int, M: int, threads: int | None = None) -> np.ndarray:
    """fn(lo, hi) -> [M, hi - lo] evaluated over row slices on a thread pool
    (the oracle's C calls release the GIL) and joined along the rows. Rows are
    independent outputs, so slicing changes no value."""
    threads = threads or min(16, os.cpu_count() or 1)
    parts = row_slices(n, threads)
    out = np.empty((M, n), dtype=np.float64)
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        for (lo, hi), blk in zip(parts, ex.map(lambda b: fn(*b), parts)):
            out[:, lo:hi] = blk
    return out


def oracle_rows(o: Oracle, inp: synth.QmvInputs, rows: np.ndarray | None = None):
    """fp64 reference y and sum|w x| for the given rows (all rows when None),
    computed from the oracle's own packing of q; large problems are split
    over host threads by rows."""
    pr = inp.problem
    q = inp.q if rows is None else inp.q[rows]
    s = inp.scales if rows is None else inp.scales[rows]
    b = inp.biases if rows is None else inp.biases[rows]
    w = o.pack(q, pr.bits)
    n, M = w.shape[0], np.atleast_2d(inp.x).shape[0]
    y = threaded_rows(lambda lo, hi: o.qmv_f64_dequant(w[lo:hi], s[lo:hi], b[lo:hi], inp.x, pr.bits,
                                                       pr.group_size), n, M)
    t = threaded_rows(lambda lo, hi: o.abs_terms(w[lo:hi], s[lo:hi], b[lo:hi], inp.x, pr.bits, pr.group_size),
                      n, M)
    return y, t


def check_parity(y_gpu_bits: np.ndarray, y_ref: np.ndarray, terms: np.ndarray, what: str):
    y = synth.bf16_bits_to_f32(y_gpu_bits).astype(np.float64)
    ok, worst = tolerance_ok(y, y_ref, terms)
    assert ok, f"{what}: worst |dy| / (8e-3*sum|wx| + 1e-5) = {worst:.3f}"
    return worst
