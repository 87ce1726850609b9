"""W4A16 GEMM (fa_w4a16_gemm through the C ABI) against the float64 oracle.

Tolerance, per output element: the exact product of the fp16 weights and
activations rounded once to fp16 (half an fp16 ulp of |Y_ref|), plus the
worst-case error of an fp32 sum of K products, K * 2^-24 * sum_k |x_k w_k|
(doubled for the sum of split partials).  Every weight must be dequantised
exactly as the oracle rounds it, or the error would exceed this at once.
"""

import numpy as np
import pytest
import torch

import io_aware_exact_fwd_gb300 as fa
from oracle import w4a16_abs_sum, w4a16_gemm
from synth import w4a16_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.fa_debug_set_fault(0)
    fa.fa_debug_set_wait_limit_ns(0)


def _half_ulp_fp16(y):
    ay = np.abs(y)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ay > 0, ay, 1.0)))
    e = np.maximum(e, -14)  # subnormal spacing below 2^-14
    return np.where(ay > 0, 2.0 ** (e - 11), 2.0 ** -25)


def _check(y, d, K, rows=None):
    x, wq, s, z = d["x"], d["wq"], d["scales"], d["zeros"]
    if rows is not None:
        wq, s, z = wq[rows], s[:, rows], z[:, rows]
        y = y[:, rows]
    ref = w4a16_gemm(x, wq, s, z)
    bound = _half_ulp_fp16(ref) * 1.001 + 2.0 * K * 2.0 ** -24 * w4a16_abs_sum(x, wq, s, z)
    err = np.abs(y.float().cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), float((err - bound).max())


def _run(M, N, K, seed, n_split=0):
    d = w4a16_inputs(M, N, K, seed)
    dev = {k: v.cuda() for k, v in d.items()}
    y = fa.fa_w4a16_gemm(dev["x"], dev["wq"], dev["scales"], dev["zeros"], n_split=n_split)
    fa.fa_sync_check()
    return y, d


@pytest.mark.parametrize("M,N,K", [(1, 128, 256), (5, 256, 512), (32, 384, 1024), (33, 144, 768), (64, 512, 2048),
                                   (100, 256, 512), (128, 1024, 4096)])
@pytest.mark.parametrize("n_split", [1, 3, 0])
def test_matches_oracle(M, N, K, n_split):
    y, d = _run(M, N, K, M + N + K, n_split)
    _check(y, d, K)


@pytest.mark.parametrize("M,N,K", [(1, 16, 256), (1, 48, 768), (1, 272, 1280), (1, 1024, 4096), (1, 32, 65536),
                                   (2, 80, 65536), (1, 96, 65792), (3, 272, 1280), (4, 48, 768)])
def test_matrix_vector_path_matches_oracle(M, N, K):
    # M = 1 runs on the CUDA cores (K <= 65536): ragged last row block (N % 32 == 16),
    # rows shorter than one 128-word step (K = 256, 768) and of one step plus a part
    # (K = 1280), the largest K of the path and one K just past it (tensor-core path);
    # small M > 1 on the tensor-core path beside them.
    y, d = _run(M, N, K, 7 * M + N + K)
    _check(y, d, K)


def test_matrix_vector_path_is_deterministic():
    d = w4a16_inputs(1, 4096, 8192, 9)
    dev = {k: v.cuda() for k, v in d.items()}
    a = fa.fa_w4a16_gemm(dev["x"], dev["wq"], dev["scales"], dev["zeros"])
    b = fa.fa_w4a16_gemm(dev["x"], dev["wq"], dev["scales"], dev["zeros"], n_split=5)
    fa.fa_sync_check()
    assert torch.equal(a, b)


def test_deterministic_with_splits():
    d = w4a16_inputs(16, 1024, 8192, 7)
    dev = {k: v.cuda() for k, v in d.items()}
    a = fa.fa_w4a16_gemm(dev["x"], dev["wq"], dev["scales"], dev["zeros"], n_split=8)
    b = fa.fa_w4a16_gemm(dev["x"], dev["wq"], dev["scales"], dev["zeros"], n_split=8)
    fa.fa_sync_check()
    assert torch.equal(a, b)
    _check(a, d, 8192, rows=np.arange(0, 1024, 37))


@pytest.mark.parametrize("M", [1, 16])
def test_decode_workload_sampled_columns(M):
    # The decode workload at full size: a 28672 x 8192 weight matrix (a 70B-class
    # MLP projection), default split count; output columns sampled for the oracle.
    N, K = 28672, 8192
    y, d = _run(M, N, K, 2026 + M)
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 60)]))
    _check(y, d, K, rows=rows)


def test_zero_point_equal_codes_give_zero():
    M, N, K = 4, 128, 256
    d = w4a16_inputs(M, N, K, 3)
    word = 0
    for j in range(8):
        word |= 5 << (4 * (j // 2) + 16 * (j % 2))
    wq = torch.full((N, K // 8), word, dtype=torch.int64).to(torch.int32)
    zeros = torch.full((K // 128, N), 5, dtype=torch.uint8)
    y = fa.fa_w4a16_gemm(d["x"].cuda(), wq.cuda(), d["scales"].cuda(), zeros.cuda())
    fa.fa_sync_check()
    assert torch.count_nonzero(y) == 0


def test_rejects_unsupported_sizes():
    x = torch.zeros((129, 256), dtype=torch.float16, device="cuda")
    wq = torch.zeros((128, 32), dtype=torch.int32, device="cuda")
    s = torch.zeros((2, 128), dtype=torch.float16, device="cuda")
    z = torch.zeros((2, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_w4a16_gemm(x, wq, s, z)
    assert e.value.status == 2
