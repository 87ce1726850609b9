"""Split-KV forward and merge: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances are those of the bf16 forward: max|LSE - LSE_ref| <= 1e-3 for every
finite partial and merged LSE, 1e-2 on O (fp32 partials: absolute; merged bf16 O:
beyond the rounding of the exact result to bf16).  An empty split (no visible key)
must give LSE = -inf exactly, where the oracle does.  The oracle sees the same bf16
input values as the GPU.
"""

import numpy as np
import pytest
import torch

import io_aware_exact_fwd_gb300 as fa
from oracle import attention_general, attention_splitkv, merge_partials
from synth import normal_qkv

from gpu_util import FWD_LSE_ATOL, FWD_O_ATOL, max_abs, o_excess

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.fa_debug_set_fault(0)
    fa.fa_debug_set_wait_limit_ns(0)


def _inputs(B, H, Nq, Nk, d, seed):
    kv = normal_qkv(B, H, Nk, d, seed)
    q = normal_qkv(B, H, Nq, d, seed + 7)["q"]
    return q.to(torch.bfloat16).cuda(), kv["k"].to(torch.bfloat16).cuda(), kv["v"].to(torch.bfloat16).cuda()


def _check_partials(op, lp, op_ref, lp_ref):
    lp, op = lp.cpu().numpy().astype(np.float64), op.cpu().numpy().astype(np.float64)
    empty_ref = np.isneginf(lp_ref)
    assert np.array_equal(np.isneginf(lp), empty_ref), "empty-split pattern differs"
    fin = ~empty_ref
    if fin.any():
        assert np.abs(lp[fin] - lp_ref[fin]).max() <= FWD_LSE_ATOL
        assert np.abs(op[fin] - op_ref[fin]).max() <= FWD_O_ATOL


CASES = [
    # B, H, Nq, Nk, d, n_split, causal
    (1, 2, 1, 1000, 128, 3, False),
    (1, 2, 1, 1000, 128, 3, True),
    (2, 2, 7, 777, 64, 4, False),
    (2, 2, 7, 777, 64, 4, True),
    (1, 2, 300, 1300, 128, 5, True),
    (1, 2, 513, 513, 128, 2, True),
    (1, 1, 129, 900, 64, 2, False),
    (1, 2, 5, 300, 128, 40, False),   # 3 key blocks: 37 trailing splits are empty
    (1, 1, 600, 600, 128, 1, False),  # several 256-row query units, one split
    # One query row: at d = 64 the CUDA-core partials (32-key chunks over four warps).
    (2, 3, 1, 777, 64, 4, False),     # a ragged last chunk
    (1, 2, 1, 300, 64, 40, True),     # 37 trailing splits empty
    (1, 1, 1, 33, 64, 1, False),      # one full chunk and one key
    (1, 1, 1, 5, 64, 1, False),       # fewer keys than lanes, three warps idle
    (3, 2, 1, 4500, 64, 2, True),     # many chunks per warp
    (1, 2, 1, 300, 128, 40, True),    # d = 128: the tensor-core kernel with one row
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,n,causal", CASES)
def test_partials_match_oracle(B, H, Nq, Nk, d, n, causal):
    q, k, v = _inputs(B, H, Nq, Nk, d, 31 + Nq + Nk)
    scale = d ** -0.5
    op, lp = fa.fa_fwd_splitkv_partial(q, k, v, n, causal=causal, scale=scale)
    fa.fa_sync_check()
    op_ref, lp_ref = attention_splitkv(q, k, v, scale, causal, n)
    _check_partials(op, lp, op_ref, lp_ref)


@pytest.mark.parametrize("B,H,Nq,Nk,d,n,causal", CASES)
def test_split_forward_matches_oracle(B, H, Nq, Nk, d, n, causal):
    q, k, v = _inputs(B, H, Nq, Nk, d, 57 + Nq + Nk)
    scale = d ** -0.5
    o, lse = fa.fa_fwd_splitkv(q, k, v, n_split=n, causal=causal, scale=scale)
    fa.fa_sync_check()
    o_ref, lse_ref = attention_general(q, k, v, scale, causal)
    assert o_excess(o, o_ref) <= FWD_O_ATOL
    assert max_abs(lse, lse_ref) <= FWD_LSE_ATOL


def test_merge_kernel_alone_is_exact_to_fp32():
    # Partials from the oracle (float64 -> fp32), including empty splits whose O is
    # garbage: the merge must not read it.  Only fp32 arithmetic and the final bf16
    # rounding of O separate the kernel from the float64 merge.
    B, H, Nq, Nk, d, n = 2, 3, 40, 700, 128, 9
    q, k, v = _inputs(B, H, Nq, Nk, d, 5)
    op_ref, lp_ref = attention_splitkv(q, k, v, 0.1, True, n)
    op32 = op_ref.astype(np.float32)
    lp32 = lp_ref.astype(np.float32)
    op32[np.isneginf(lp32)] = np.nan
    o, lse = fa.fa_merge_partials(torch.from_numpy(op32).cuda(), torch.from_numpy(lp32).cuda())
    fa.fa_sync_check()
    o_m, lse_m = merge_partials(op32.astype(np.float64), lp32.astype(np.float64))
    assert o_excess(o, o_m) <= 1e-5
    assert max_abs(lse, lse_m) <= 1e-5


def test_all_splits_empty_row():
    # A row with no visible key in any split: O = 0, LSE = -inf.
    op = torch.full((3, 1, 1, 2, 64), float("nan"), device="cuda")
    lp = torch.full((3, 1, 1, 2), float("-inf"), device="cuda")
    lp[1, 0, 0, 1] = 0.5
    op[1, 0, 0, 1] = 2.0
    o, lse = fa.fa_merge_partials(op, lp)
    fa.fa_sync_check()
    assert torch.all(o[0, 0, 0] == 0) and torch.isneginf(lse[0, 0, 0])
    assert torch.all(o[0, 0, 1] == 2.0) and abs(float(lse[0, 0, 1]) - 0.5) < 1e-6


def _fwd_takes_whole_units(B, H, N, causal):
    # fa_fwd deals a partial last pass of R <= SMs / 2 non-causal units (after at
    # most 4 full passes) out as 2R shared tiles (two warpgroups on one tile,
    # partial softmaxes merged): the same values up to rounding, but not bitwise
    # those of one whole-key split.
    units = B * H * ((N + 255) // 256)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rem = units % sms
    return causal or N <= 128 or rem == 0 or 2 * rem > sms or units // sms > 4


@pytest.mark.parametrize("B, N", [(2, 700), (40, 700)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_one_split_equals_fa_fwd(B, N, causal, d):
    # With one split and Nq == Nk the partial is the forward's O and LSE before
    # the bf16 rounding; the merge of one split multiplies by exactly 1.  Bitwise
    # when fa_fwd takes whole units; otherwise within one bf16 rounding of O.
    H = 2
    q, k, v = _inputs(B, H, N, N, d, 9)
    o1, l1 = fa.fa_fwd(q, k, v, causal=causal)
    o2, l2 = fa.fa_fwd_splitkv(q, k, v, n_split=1, causal=causal)
    fa.fa_sync_check()
    if _fwd_takes_whole_units(B, H, N, causal):
        assert torch.equal(o1, o2)
        assert torch.equal(l1, l2)
    else:
        # Both round the same exact values to bf16: at most one bf16 step apart
        # (2^-7 relative), plus a small absolute slack where |O| is tiny.
        a, b = o1.float(), o2.float()
        assert bool(((a - b).abs() <= 2.0 ** -7 * torch.maximum(a.abs(), b.abs()) + 1e-3).all())
        assert float((l1 - l2).abs().max()) <= 1e-5


@pytest.mark.parametrize("causal", [False, True])
def test_default_split_count(causal):
    B, H, Nq, Nk, d = 1, 4, 3, 5000, 128
    n = fa.fa_splitkv_default_splits(B, H, Nq, Nk, d)
    assert 1 <= n <= -(-Nk // 128)
    q, k, v = _inputs(B, H, Nq, Nk, d, 77)
    o, lse = fa.fa_fwd_splitkv(q, k, v, causal=causal)
    fa.fa_sync_check()
    o_ref, lse_ref = attention_general(q, k, v, d ** -0.5, causal)
    assert o_excess(o, o_ref) <= FWD_O_ATOL
    assert max_abs(lse, lse_ref) <= FWD_LSE_ATOL


@pytest.mark.parametrize("H, d", [(16, 128), (32, 64)])
def test_decode_workload_sampled_heads(H, d):
    # The decode workloads at full size (B=8, one query, Nk=32768; H=16 at d=128 on the
    # tensor cores, H=32 at d=64 on the CUDA cores) in the launch configuration the
    # benchmark uses; heads sampled for the oracle.
    B, Nq, Nk = 8, 1, 32768
    q, k, v = _inputs(B, H, Nq, Nk, d, 2024)
    o, lse = fa.fa_fwd_splitkv(q, k, v)
    fa.fa_sync_check()
    rng = np.random.default_rng(0)
    for b, h in [(0, 0), (B - 1, H - 1)] + [tuple(x) for x in rng.integers(0, [B, H], size=(4, 2))]:
        o_ref, lse_ref = attention_general(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1],
                                           d ** -0.5, False)
        assert o_excess(o[b:b + 1, h:h + 1], o_ref) <= FWD_O_ATOL
        assert max_abs(lse[b:b + 1, h:h + 1], lse_ref) <= FWD_LSE_ATOL


def test_splits_are_deterministic():
    q, k, v = _inputs(1, 2, 4, 3000, 128, 3)
    a = fa.fa_fwd_splitkv(q, k, v, n_split=6)
    b = fa.fa_fwd_splitkv(q, k, v, n_split=6)
    fa.fa_sync_check()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
