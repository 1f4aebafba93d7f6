"""Host-side checks of the C-ABI library (no GPU needed): it loads, it exports
every symbol the header declares, the codec matches the oracle's packing bit
for bit, and argument validation rejects bad calls before touching a GPU."""

import os
import re
import subprocess

import numpy as np
import pytest

import group_quantized_mat_gb300 as g
import synth
from oracle import Oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmv.h")


@pytest.fixture(scope="module")
def lib():
    from group_quantized_mat_gb300 import build
    build.build()
    return g.load()


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"QMV_API\s+[\w\s\*]+?\b(qmv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = header_functions()
    assert set(names) == set(g.EXPORTED), names


def test_library_exports_every_header_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in header_functions() if n not in exported]
    assert not missing, missing
    for n in header_functions():
        assert hasattr(lib, n)


def test_library_has_no_torch_dependency(lib):
    out = subprocess.run(["ldd", g.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in out and "libcudart.so" not in out


@pytest.mark.parametrize("bits", [2, 4])
def test_pack_matches_oracle_and_roundtrips(lib, bits):
    o = Oracle(0)
    for N, K, seed in [(3, 64, 1), (17, 384, 2), (64, 1024, 3)]:
        inp = synth.make_inputs(N, K, 1, bits, 64, seed)
        ours = g.qmv_pack(inp.q, bits)
        ref = o.pack(inp.q, bits)
        assert ours.dtype == np.uint32 and np.array_equal(ours, ref)
        assert np.array_equal(g.qmv_unpack(ours, K, bits), inp.q)
        assert g.qmv_packed_words(N, K, bits) == ours.size


@pytest.mark.parametrize("bits", [2, 4])
def test_pack_every_byte_value(lib, bits):
    """All 256 byte values through the library codec against the oracle's
    shift/mask fields and the float-floor chain (llama.cpp PR #159, "How")."""
    o = Oracle(0)
    per_byte = 8 // bits
    fields = np.array([o.byte_fields(b, bits) for b in range(256)], dtype=np.uint8)  # [256, per_byte]
    ff = np.array([o.byte_fields_floatfloor(b, bits) for b in range(256)], dtype=np.uint8)
    assert np.array_equal(fields, ff)
    q = fields.reshape(1, 256 * per_byte)
    w = g.qmv_pack(q, bits)
    assert np.array_equal(w.view(np.uint8).ravel(), np.arange(256, dtype=np.uint8))
    assert np.array_equal(g.qmv_unpack(w, 256 * per_byte, bits), q)


def test_pack_rejects_bad_input(lib):
    with pytest.raises(g.QmvError) as e:
        g.qmv_pack(np.full((2, 64), 16, np.uint8), 4)
    assert e.value.code == 9
    with pytest.raises(g.QmvError) as e:
        g.qmv_pack(np.zeros((2, 64), np.uint8), 3)
    assert e.value.code == 2
    with pytest.raises(g.QmvError) as e:
        g.qmv_pack(np.zeros((2, 12), np.uint8), 4)
    assert e.value.code == 4
    assert lib.qmv_pack(None, None, 1, 64, 4) == 1
    assert g.qmv_packed_words(1, 12, 4) == 0


def test_split_plan(lib):
    # K-chunks of 2048 elements: a function of K only
    assert g.qmv_split_count(15360, 3840, 4, 64) == g.qmv_split_count(7, 3840, 4, 64) == 2
    assert g.qmv_split_count(15360, 3840, 2, 64) == 2
    assert g.qmv_split_count(15360, 3840, 2, 128) == 2
    assert g.qmv_split_count(256, 1024, 4, 64) == 1
    assert g.qmv_split_count(3840, 15360, 4, 64) == 8
    assert g.qmv_split_count(5120, 17408, 4, 64) == 9
    assert g.qmv_split_count(1, 1000, 4, 64) == 0
    a256 = lambda b: (b + 255) // 256 * 256
    # M = 1: no workspace while one CTA covers all chunks of its rows
    assert g.qmv_workspace_size(1, 256, 1024, 4, 64) == 0
    assert g.qmv_workspace_size(1, 15360, 3840, 4, 64) == 0
    assert g.qmv_workspace_size(1, 3840, 15360, 4, 64) == 0
    # M >= 2: the call's staged x cells [M][K/64], 272 bytes each (fp32 x'
    # and the subgroup's meta). On K = 3840 the cells of all of K fit a CTA's
    # shared memory up to M = 10; from M = 11 CTAs split K in two.
    assert g.qmv_workspace_size(2, 15360, 3840, 4, 64) == a256(2 * 60 * 272)
    assert g.qmv_workspace_size(10, 15360, 3840, 4, 64) == a256(10 * 60 * 272)
    split_p = lambda M: a256(3840 * 4) + 2 * M * 15360 * 4
    assert g.qmv_workspace_size(11, 15360, 3840, 4, 64) == a256(split_p(11)) + a256(11 * 60 * 272)
    assert g.qmv_workspace_size(13, 15360, 3840, 4, 64) == a256(split_p(13)) + a256(13 * 60 * 272)
    # K = 15360 splits; chunk values meet in the
    # workspace first: a 256-byte-aligned block of one counter per 4-row
    # block, then ks x M x N fp32 partials, then the cells
    split13 = (960 * 4 + 255) // 256 * 256 + 8 * 13 * 3840 * 4
    w13 = g.qmv_workspace_size(13, 3840, 15360, 4, 64)
    assert w13 == a256(split13) + a256(13 * 240 * 272)
    w16 = g.qmv_workspace_size(16, 3840, 15360, 4, 64)
    assert w16 == a256(split13 + 8 * 3 * 3840 * 4) + a256(16 * 240 * 272)
    # M above 16 runs as launches of 16 vectors and one of the remainder: the
    # widest of those decides
    assert g.qmv_workspace_size(17, 15360, 3840, 4, 64) == a256(split_p(16)) + a256(16 * 60 * 272)
    assert g.qmv_workspace_size(20, 3840, 15360, 4, 64) == w16
    assert g.qmv_workspace_size(33, 3840, 15360, 4, 64) == w16
    assert g.qmv_workspace_size(256, 3840, 15360, 4, 64) == w16
    assert g.qmv_workspace_size(257, 3840, 15360, 4, 64) == 0
    # sizes whose scale index would pass 2^31 are refused
    assert g.qmv_split_count(1 << 30, 1 << 13, 4, 64) == 0


FAKE = 1 << 20  # an aligned address that validation must reject before any use


@pytest.mark.parametrize("kw,code", [
    (dict(w_q=0), 1), (dict(y=0), 1),
    (dict(bits=3), 2), (dict(group_size=32), 3),
    (dict(K=1000), 4), (dict(N=0), 4), (dict(K=0), 4),
    (dict(M=0), 5), (dict(M=257), 5),
    (dict(w_q=FAKE + 8), 6), (dict(x=FAKE + 2), 6), (dict(scales=FAKE + 1), 6),
    (dict(scales=FAKE + 8), 6), (dict(biases=FAKE + 2), 6),
])
def test_run_validation_before_gpu(lib, kw, code):
    args = dict(w_q=FAKE, scales=FAKE, biases=FAKE, x=FAKE, y=FAKE, M=1, N=64, K=1024, bits=4, group_size=64)
    args.update(kw)
    r = lib.qmv_run(args["w_q"] or None, args["scales"], args["biases"], args["x"], args["y"] or None,
                    args["M"], args["N"], args["K"], args["bits"], args["group_size"], None)
    assert r == code, g.qmv_status_string(r)


def test_run_ex_rejects_flags(lib):
    r = lib.qmv_run_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 1024, 4, 64, None, 0, 0x100, None)
    assert r == 10
    r = lib.qmv_run_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 1024, 4, 64, None, 0, 0x10, None)
    assert r == 10
    r = lib.qmv_run_ex(FAKE, FAKE, FAKE, FAKE, FAKE + 2, 1, 64, 1024, 4, 64, None, 0, g.F32_OUT, None)
    assert r == 6


def test_run_ex_interleaved_metadata_validation(lib):
    # with QMV_SB_INTERLEAVED the biases pointer is not read (NULL allowed) ...
    r = lib.qmv_run_ex(FAKE, FAKE + 8, None, FAKE, FAKE, 1, 64, 1024, 4, 64, None, 0, g.SB_INTERLEAVED, None)
    assert r == 6  # ... and the interleaved array must be 16-byte aligned
    r = lib.qmv_run_ex(FAKE, None, None, FAKE, FAKE, 1, 64, 1024, 4, 64, None, 0, g.SB_INTERLEAVED, None)
    assert r == 1
    r = lib.qmv_run_ex(FAKE, FAKE, None, FAKE, FAKE, 1, 64, 1024, 4, 64, None, 0, 0, None)
    assert r == 1  # without the flag the biases are required


def test_pack_sb_interleaves_scale_low_bias_high(lib):
    rng = np.random.default_rng(3)
    s = rng.integers(0, 1 << 16, size=(5, 7), dtype=np.uint16)
    b = rng.integers(0, 1 << 16, size=(5, 7), dtype=np.uint16)
    sb = g.qmv_pack_sb(s, b)
    assert sb.dtype == np.uint32 and sb.shape == (5, 7)
    assert np.array_equal(sb & 0xFFFF, s) and np.array_equal(sb >> 16, b)
    out = np.empty(4, dtype=np.uint32)
    assert lib.qmv_pack_sb(None, b.ctypes.data, out.ctypes.data, 1, 4) == 1
    assert lib.qmv_pack_sb(s.ctypes.data, b.ctypes.data, out.ctypes.data, 0, 4) == 4
    assert lib.qmv_pack_sb(s.ctypes.data, b.ctypes.data, out.ctypes.data, 4, 0) == 4


def test_status_strings(lib):
    for code in range(11):
        s = g.qmv_status_string(code)
        assert s.startswith(g.STATUS[code])
    assert "unknown" in g.qmv_status_string(99)


@pytest.mark.parametrize("kw,code", [
    (dict(w_q=0), 1), (dict(scales=0), 1), (dict(x=0), 1), (dict(y=0), 1),
    (dict(K=48), 4), (dict(K=0), 4), (dict(N=0), 4), (dict(K=1 << 25), 4), (dict(N=(1 << 30) + 1), 4),
    (dict(N=1 << 26, K=1 << 10), 4),  # N * K/32 = 2^31 scale bytes
    (dict(M=0), 5), (dict(M=257), 5),
    (dict(w_q=FAKE + 8), 6), (dict(x=FAKE + 2), 6), (dict(y=FAKE + 1), 6),
    (dict(flags=0x4), 10), (dict(flags=0x8), 10), (dict(flags=0x100), 10),
])
def test_mxfp4_run_validation_before_gpu(lib, kw, code):
    args = dict(w_q=FAKE, scales=FAKE + 3, x=FAKE, y=FAKE, M=1, N=64, K=1024, flags=0)
    args.update(kw)
    r = lib.qmv_mxfp4_run(args["w_q"] or None, args["scales"] or None, args["x"] or None, args["y"] or None,
                          args["M"], args["N"], args["K"], args["flags"], None)
    assert r == code, g.qmv_status_string(r)
    # an fp32 y needs 4-byte alignment
    assert lib.qmv_mxfp4_run(FAKE, FAKE, FAKE, FAKE + 2, 1, 64, 1024, g.F32_OUT, None) == 6


def test_header_compiles_as_c_and_links(tmp_path, lib):
    """include/qmv.h is a plain C header: a C99 program that includes it,
    calls the host-only entry points and links against libqmv.so runs
    without a GPU."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "use_qmv.c"
    src.write_text(r'''
#include <stdio.h>
#include "qmv.h"
int main(void) {
    uint8_t q[64];
    uint32_t w[8];
    for (int i = 0; i < 64; ++i) q[i] = (uint8_t)(i % 16);
    if (qmv_packed_words(1, 64, 4) != 8) return 1;
    if (qmv_pack(q, w, 1, 64, 4) != QMV_OK) return 2;
    if (w[0] != 0x76543210u) return 3;
    if (qmv_mxfp4_run(NULL, NULL, NULL, NULL, 1, 1, 32, 0u, NULL) != QMV_ERR_NULL) return 4;
    printf("%s\n", qmv_status_string(QMV_ERR_SHAPE));
    return 0;
}
''')
    inc = os.path.join(ROOT, "include")
    libdir = os.path.dirname(g.LIB_PATH)
    exe = tmp_path / "use_qmv"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), "-L", libdir, "-lqmv",
                        f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.strip() != ""
