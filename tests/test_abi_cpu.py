"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, and rejects bad arguments synchronously with the documented status."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def lib():
    import io_aware_exact_fwd_gb300 as fa

    if not os.path.exists(fa.library_path()):
        from io_aware_exact_fwd_gb300 import _build

        _build.build()
    return fa.load_library()


def _declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^FA_API\s+[^;(]*?\b(fa_\w+)\s*\(", src, re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert "fa_fwd" in names and "fa_sync_check" in names
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_and_version(lib):
    import io_aware_exact_fwd_gb300 as fa

    for code in range(0, 7):
        assert fa.fa_strerror(code)
    assert fa.fa_strerror(99) == "unknown status"
    assert fa.fa_version() >= 1


FAKE = 0x10000  # 16-byte aligned fake device address: never dereferenced on these paths


def _fwd(lib, B=1, H=1, N=128, d=64, causal=0, scale=0.125, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE):
    vp = ctypes.c_void_p
    return lib.fa_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, N, d, causal, scale, vp(0))


def test_forward_validation_statuses(lib):
    assert _fwd(lib, B=-1) == 1
    assert _fwd(lib, N=-5) == 1
    assert _fwd(lib, causal=2) == 1
    for s in (0.0, -0.1, float("nan"), float("inf")):
        assert _fwd(lib, scale=s) == 1
    assert _fwd(lib, d=96) == 2
    assert _fwd(lib, d=256) == 2
    assert _fwd(lib, q=0) == 1
    assert _fwd(lib, lse=0) == 1
    assert _fwd(lib, o=FAKE + 8) == 3
    assert _fwd(lib, lse=FAKE + 2) == 3
    # Empty problems are valid no-ops, even with NULL pointers.
    assert _fwd(lib, B=0, q=0, k=0, v=0, o=0, lse=0) == 0
    assert _fwd(lib, N=0, q=0, k=0, v=0, o=0, lse=0) == 0
    # Sizes beyond the kernel's index range are refused before any device work.
    assert _fwd(lib, B=1 << 16, H=1 << 16, N=128) == 2


def test_binding_raises_without_gpu_work(lib):
    import torch

    import io_aware_exact_fwd_gb300 as fa

    with pytest.raises(TypeError):
        fa.fa_fwd(torch.zeros(1, 1, 8, 64), torch.zeros(1, 1, 8, 64), torch.zeros(1, 1, 8, 64))


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "io_aware_exact_fwd_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, fn), encoding="utf-8").read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, re.M), fn
                assert "oracle/" not in src, fn


def _part(lib, B=1, H=1, Nq=1, Nk=1000, d=128, n=4, causal=0, scale=0.125, q=FAKE, k=FAKE, v=FAKE, o=FAKE,
          lse=FAKE):
    vp = ctypes.c_void_p
    return lib.fa_fwd_splitkv_partial(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, Nq, Nk, d, n, causal, scale,
                                      vp(0))


def test_splitkv_validation_statuses(lib):
    assert _part(lib, n=0) == 1
    assert _part(lib, n=1025) == 1
    assert _part(lib, Nk=0) == 1
    assert _part(lib, Nq=-1) == 1
    assert _part(lib, causal=1, Nq=2000, Nk=1000) == 1   # causal needs Nq <= Nk
    assert _part(lib, d=96) == 2
    assert _part(lib, q=0) == 1
    assert _part(lib, o=FAKE + 4) == 3
    assert _part(lib, Nq=0, q=0, k=0, v=0, o=0, lse=0) == 0  # empty: no-op
    vp = ctypes.c_void_p
    assert lib.fa_merge_partials(vp(FAKE), vp(FAKE), vp(FAKE + 8), vp(FAKE), 2, 1, 1, 4, 64, vp(0)) == 3
    assert lib.fa_merge_partials(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 0, 1, 1, 4, 64, vp(0)) == 1
    # The combined call refuses a short workspace before any device work.
    need = lib.fa_splitkv_workspace_size(2, 3, 5, 64, 7)
    assert need >= 7 * 2 * 3 * 5 * (64 + 1) * 4
    assert lib.fa_fwd_splitkv(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), need - 1, 2, 3, 5, 900, 64,
                              7, 0, 0.125, vp(0)) == 6
    assert lib.fa_splitkv_workspace_size(1, 1, 1, 96, 1) == 0


def test_splitkv_default_split_rule(lib):
    # fa_splitkv_default_splits (include/fa.h): the fewest splits n in 1 .. min(64, max(1,
    # nkb / 4)) whose busiest-slot load ceil(units n / slots) / n is within 2 % of the
    # best; 1 when Nq > 128 and the units already cover the SMs; slots = SMs, times the
    # one-row kernel's resident CTAs for Nq == 1 at d == 64.  Without a GPU the library
    # assumes 148 SMs and 4 resident CTAs.
    import torch
    if torch.cuda.is_available():
        pytest.skip("checked on the device by the GPU tests")
    sms = 148

    def expected(B, H, Nq, Nk, d):
        units = B * H * ((Nq + 255) // 256)
        nkb = (Nk + 127) // 128
        if Nq > 128 and units >= sms:
            return 1
        slots = sms * 4 if (Nq == 1 and d == 64) else sms
        n_max = min(max(1, nkb // 4), 64)
        cost = lambda n: ((units * n + slots - 1) // slots) / n
        best = min(cost(n) for n in range(1, n_max + 1))
        return next(n for n in range(1, n_max + 1) if cost(n) <= best * 1.02)

    for B, H, Nq, Nk, d in [(8, 16, 1, 32768, 128), (1, 16, 1, 131072, 128), (8, 32, 1, 32768, 64),
                            (4, 16, 16, 32768, 128), (1, 16, 128, 65536, 128), (1, 2, 1, 300, 64),
                            (2, 3, 5, 1500, 64), (4, 16, 2048, 2048, 128), (1, 1, 200, 100000, 128)]:
        assert lib.fa_splitkv_default_splits(B, H, Nq, Nk, d) == expected(B, H, Nq, Nk, d), (B, H, Nq, Nk, d)
    assert lib.fa_splitkv_default_splits(1, 1, 1, 1000, 96) == 0


def test_strided_validation_statuses(lib):
    vp = ctypes.c_void_p
    good = (ctypes.c_int64 * 3)(128, 128 * 64, 128 * 64 * 2)
    odd = (ctypes.c_int64 * 3)(132, 132 * 64, 132 * 64 * 2)
    short = (ctypes.c_int64 * 3)(64, 128 * 64, 128 * 64 * 2)
    def fwd(qs):
        return lib.fa_fwd_strided(vp(FAKE), ctypes.cast(qs, vp) if qs is not None else None, vp(FAKE), None,
                                  vp(FAKE), None, vp(FAKE), None, vp(FAKE), 2, 2, 64, 128, 0, 0.1, vp(0))
    assert fwd(odd) == 3      # row stride of 132 elements is not 16-byte aligned
    assert fwd(short) == 1    # rows of one head would overlap
    neg = (ctypes.c_int64 * 3)(128, -1, 1)
    assert fwd(neg) == 1


def test_w4a16_validation_statuses(lib):
    vp = ctypes.c_void_p
    def g(M=4, N=128, K=256, n=1, y=FAKE, ws=0, wsb=0):
        return lib.fa_w4a16_gemm(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(y), vp(ws), wsb, M, N, K, n, vp(0))
    assert g(M=129) == 2
    assert g(N=120) == 2
    assert g(K=384) == 2
    assert g(M=-1) == 1
    assert g(M=0) == 0
    assert g(y=FAKE + 8) == 3
    assert g(M=2, K=1024, n=4) == 6               # splits of the tensor-core path need a workspace
    assert lib.fa_w4a16_workspace_size(8, 128, 1024, 4) == 4 * 8 * 128 * 4
    assert lib.fa_w4a16_workspace_size(8, 128, 1024, 1) == 0
    # M = 1: the matrix-vector path, one pass over K per row, never a workspace.
    assert lib.fa_w4a16_workspace_size(1, 128, 1024, 4) == 0
    assert lib.fa_w4a16_default_splits(1, 28672, 8192) == 1
    # Tensor-core path: splits of at least 4 chunks of 256, never more than K allows.
    for M, N, K in ((16, 28672, 8192), (16, 8192, 28672), (128, 4096, 4096), (2, 256, 1024)):
        n = lib.fa_w4a16_default_splits(M, N, K)
        assert 1 <= n <= max(1, K // 1024), (M, N, K, n)
    assert lib.fa_w4a16_default_splits(0, 128, 256) == 0
    assert lib.fa_w4a16_default_splits(4, 120, 256) == 0


def test_fp8_backward_validation_statuses(lib):
    vp = ctypes.c_void_p
    B, H, N, d = 1, 2, 100, 128
    f8 = lib.fa_fp8_workspace_size(B, H, N, d)
    need = lib.fa_bwd_fp8_workspace_size(B, H, N, d)
    assert need >= lib.fa_bwd_workspace_size(B, H, N, d) + 4 * B * H * N * d * 2 + B * H * N * 4
    # d = 64 is supported; other head dims are not.
    assert lib.fa_bwd_fp8_workspace_size(B, H, N, 64) >= lib.fa_bwd_workspace_size(B, H, N, 64)
    assert lib.fa_bwd_fp8_workspace_size(B, H, N, 96) == 0

    def g(det=0, rec=0, dd=d, ws8=FAKE, f8b=f8, signs=FAKE, ws=FAKE, wsb=need, n=N):
        return lib.fa_bwd_fp8(vp(ws8), f8b, vp(signs), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                              vp(ws), wsb, B, H, n, dd, 0, 0.1, det, rec, vp(0))
    assert g(det=2) == 1
    assert g(rec=-1) == 1
    assert g(dd=96) == 2
    assert g(ws8=0) == 6
    assert g(f8b=f8 - 1) == 6
    assert g(signs=0) == 1
    assert g(wsb=need - 1) == 6
    assert g(ws=FAKE + 16) == 3
    assert g(n=0) == 0
    assert lib.fa_fp8_dequantize(vp(FAKE), f8, vp(FAKE + 8), vp(FAKE), vp(FAKE), B, H, N, d, vp(0)) == 3
    assert lib.fa_fp8_dequantize(vp(0), f8, vp(FAKE), vp(FAKE), vp(FAKE), B, H, N, d, vp(0)) == 6


def test_header_is_plain_c(tmp_path):
    # The boundary is a C ABI: the header must compile as strict C99 with no C++.
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_fa.c"
    src.write_text('#include "fa.h"\nint main(void) { return fa_version() == 0; }\n')
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-c", str(src), "-o", str(tmp_path / "use_fa.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_seeded_rotation_signs_match_the_oracle(lib):
    # The library's host copy of the seeded sign rule against the oracle's SplitMix64
    # (itself pinned by published outputs); pure host code, no GPU needed.
    import numpy as np

    from oracle import seeded_rotation_signs

    for seed in (0, 1, 5, 1234567, 2 ** 63, 2 ** 64 - 1):
        for d in (1, 64, 128):
            out = (ctypes.c_int8 * d)()
            assert lib.fa_fp8_rotation_signs(ctypes.c_uint64(seed), d, out) == 0
            assert np.array_equal(np.frombuffer(out, dtype=np.int8), seeded_rotation_signs(seed, d)), (seed, d)
    assert lib.fa_fp8_rotation_signs(ctypes.c_uint64(1), 0, (ctypes.c_int8 * 1)()) == 1
    assert lib.fa_fp8_rotation_signs(ctypes.c_uint64(1), 64, None) == 1


def test_fp8_prepare_validation_statuses(lib):
    vp = ctypes.c_void_p
    B, H, N, d = 1, 2, 100, 128
    need = lib.fa_fp8_workspace_size(B, H, N, d)
    seeded = lambda q=FAKE, ws=FAKE, nb=need, dt=0, dd=d: lib.fa_fp8_prepare_seeded(
        vp(q), vp(FAKE), vp(FAKE), dt, ctypes.c_uint64(7), vp(ws), nb, B, H, N, dd, vp(0))
    assert seeded(q=0) == 1
    assert seeded(dt=2) == 1
    assert seeded(ws=0) == 6
    assert seeded(nb=need - 1) == 6
    assert seeded(q=FAKE + 8) == 3
    assert seeded(ws=FAKE + 16) == 3          # workspace must be 256-byte aligned
    assert seeded(dd=96) == 2
    # The signs-array form needs its signs.
    assert lib.fa_fp8_prepare(vp(FAKE), vp(FAKE), vp(FAKE), 0, vp(0), vp(FAKE), need, B, H, N, d, vp(0)) == 1
