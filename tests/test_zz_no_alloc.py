"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (a plugin inside a framework that owns all device memory, or a
loop where cudaMalloc's possible device-wide synchronisation is not allowed)
pass inputs and outputs only; the library supplies the scratch from a fixed
per-device buffer.  These tests call the entry point through the C ABI and
check it against the float64 oracle, and against fa_bwd (the entry point with a
caller workspace) on two calls in a row (the buffer keeps the previous call's contents, so the second call
also shows that everything that must start at zero is cleared).  This file is
collected last so that a run stopping at its first failure has already run
every other test; it also passes alone in a fresh process.
"""

import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import io_aware_exact_fwd_gb300 as fa
from synth import normal_qkv

from gpu_util import BWD_REL

pytestmark = pytest.mark.gpu


def _rel(x, ref):
    x = x.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-4))


def test_noalloc_backward_matches_fa_bwd_on_two_calls():
    fa.load_library()
    fa.fa_debug_set_fault(0)
    fa.fa_debug_set_wait_limit_ns(0)
    for call, (N, causal) in enumerate(((777, False), (1030, True))):
        x = normal_qkv(2, 3, N, 128, 300 + call, with_do=True)
        q, k, v, g = (x[n].to(torch.bfloat16).cuda() for n in ("q", "k", "v", "do"))
        o, lse = fa.fa_fwd(q, k, v, causal=causal)
        ref = fa.fa_bwd(q, k, v, o, g, lse, causal=causal)
        got = tuple(torch.empty_like(q) for _ in range(3))
        fa.fa_bwd_noalloc(q, k, v, o, g, lse, *got, causal=causal)
        fa.fa_sync_check()
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert _rel(a, b) <= BWD_REL, (call, name, _rel(a, b))
        # dK and dV involve no atomics: identical to the workspace entry point.
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_backward_matches_the_oracle(d):
    # The same entry point against the float64 oracle directly (ragged N, causal),
    # every head, at the backward's bar: max|dX - dX_ref| <= 2e-2 max|dX_ref|.
    from oracle import attention_backward

    fa.load_library()
    fa.fa_debug_set_fault(0)
    fa.fa_debug_set_wait_limit_ns(0)
    B, H, N = 1, 2, 333
    x = normal_qkv(B, H, N, d, 311, with_do=True)
    q, k, v, g = (x[n].to(torch.bfloat16).cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v, causal=True)
    got = tuple(torch.empty_like(q) for _ in range(3))
    fa.fa_bwd_noalloc(q, k, v, o, g, lse, *got, causal=True)
    fa.fa_sync_check()
    ref = attention_backward(q, k, v, g, d ** -0.5, True)
    for name, a, r in zip(("dq", "dk", "dv"), got, ref):
        err = float(np.abs(a.double().cpu().numpy() - r).max() / max(np.abs(r).max(), 1e-4))
        assert err <= BWD_REL, (d, name, err)


def test_noalloc_rejects_problems_beyond_its_buffer():
    lib = fa.load_library()
    limit = fa.fa_bwd_noalloc_max_workspace()
    assert limit == 64 << 20
    B, H, N, d = 1, 64, 8192, 128
    assert fa.fa_bwd_workspace_size(B, H, N, d) > limit
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check comes first
    st = lib.fa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, B, H, N, d, 0, 0.088,
                            ctypes.c_void_p(0))
    assert st == 6


def test_noalloc_validates_arguments_before_its_buffer():
    # A bad call gets fa_bwd's status (here: a NULL q), whatever its size.
    lib = fa.load_library()
    fake = ctypes.c_void_p(0x10000)
    null = ctypes.c_void_p(0)
    st = lib.fa_bwd_noalloc(null, fake, fake, fake, fake, fake, fake, fake, fake, 1, 2, 300, 128, 0, 0.088,
                            ctypes.c_void_p(0))
    assert st == 1
    st = lib.fa_bwd_noalloc(ctypes.c_void_p(0x10008), fake, fake, fake, fake, fake, fake, fake, fake, 1, 2, 300, 128,
                            0, 0.088, ctypes.c_void_p(0))
    assert st == 3  # q not 16-byte aligned


# The child process below uses the CUDA driver API through ctypes (no torch): it
# allocates device memory in the device's primary context, runs the forward, the
# backward with a workspace and fa_bwd_noalloc, then creates a second context on
# the same device, makes it current and does the same there.  The scratch array
# and the error word are different memory in each context, so their addresses
# must be looked up in the context that is current at each call; an address
# carried over from the first context would not be valid in the second.
_CHILD = r"""
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import io_aware_exact_fwd_gb300 as fa
lib = fa.load_library()
cu = ctypes.CDLL("libcuda.so.1")
def ck(r, what):
    if r != 0:
        raise SystemExit(f"{what}: CUresult {r}")
ck(cu.cuInit(0), "cuInit")
dev = ctypes.c_int()
ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
B, H, N, d, causal = 1, 2, 700, 128, 1
scale = d ** -0.5
rng = np.random.default_rng(77)
def bf16_bits(x):
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
def bf16_val(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
host = {n: bf16_bits(rng.standard_normal((B, H, N, d))) for n in ("q", "k", "v", "do")}
nel = B * H * N * d
ws_bytes = lib.fa_bwd_workspace_size(B, H, N, d)
def alloc(nbytes):
    p = ctypes.c_uint64()
    ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc")
    return p.value
def run_in_current_context():
    buf = {n: alloc(nel * 2) for n in ("q", "k", "v", "do", "o", "dq", "dk", "dv", "dq2", "dk2", "dv2")}
    buf["lse"] = alloc(B * H * N * 4)
    ws = alloc(ws_bytes)
    for n in ("q", "k", "v", "do"):
        ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(buf[n]), host[n].ctypes.data_as(ctypes.c_void_p),
                              ctypes.c_size_t(nel * 2)), "HtoD")
    P = lambda n: ctypes.c_void_p(buf[n])
    F = ctypes.c_float
    S = ctypes.c_void_p(0)
    assert lib.fa_fwd(P("q"), P("k"), P("v"), P("o"), P("lse"), B, H, N, d, causal, F(scale), S) == 0
    assert lib.fa_bwd(P("q"), P("k"), P("v"), P("o"), P("do"), P("lse"), P("dq"), P("dk"), P("dv"),
                      ctypes.c_void_p(ws), ctypes.c_size_t(ws_bytes), B, H, N, d, causal, F(scale), S) == 0
    for _ in range(2):  # two calls in a row on the shared scratch
        assert lib.fa_bwd_noalloc(P("q"), P("k"), P("v"), P("o"), P("do"), P("lse"), P("dq2"), P("dk2"),
                                  P("dv2"), B, H, N, d, causal, F(scale), S) == 0
    assert lib.fa_sync_check(S) == 0
    out = {}
    for n in ("dq", "dk", "dv", "dq2", "dk2", "dv2"):
        h = np.empty(nel, np.uint16)
        ck(cu.cuMemcpyDtoH_v2(h.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(buf[n]),
                              ctypes.c_size_t(nel * 2)), "DtoH")
        out[n] = h
    for p in list(buf.values()) + [ws]:
        ck(cu.cuMemFree_v2(ctypes.c_uint64(p)), "cuMemFree")
    return out
def check(out, tag):
    assert np.array_equal(out["dk"], out["dk2"]) and np.array_equal(out["dv"], out["dv2"]), tag
    a, b = bf16_val(out["dq2"]), bf16_val(out["dq"])
    assert np.abs(a - b).max() <= 2e-2 * max(np.abs(b).max(), 1e-4), tag
primary = ctypes.c_void_p()
ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "cuDevicePrimaryCtxRetain")
ck(cu.cuCtxPushCurrent_v2(primary), "push primary")
first = run_in_current_context()
check(first, "primary context")
second = ctypes.c_void_p()
create = getattr(cu, "cuCtxCreate_v4", None)
if create is not None:
    ck(create(ctypes.byref(second), None, 0, dev), "cuCtxCreate")   # pushed: now current
else:
    ck(cu.cuCtxCreate_v2(ctypes.byref(second), 0, dev), "cuCtxCreate")
again = run_in_current_context()
check(again, "second context")
assert np.array_equal(first["dk2"], again["dk2"]) and np.array_equal(first["dv2"], again["dv2"])
ck(cu.cuCtxSynchronize(), "sync")
ck(cu.cuCtxPopCurrent_v2(ctypes.byref(ctypes.c_void_p())), "pop second")   # left to process exit
ck(cu.cuCtxPopCurrent_v2(ctypes.byref(ctypes.c_void_p())), "pop primary")
print("contexts ok")
"""


def test_noalloc_in_a_second_context_of_the_same_device():
    # A caller may run the library under a context of its own (a host framework's
    # non-primary context): the scratch address must be the one of that context.
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CHILD, root], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "contexts ok" in r.stdout, (r.stdout[-2000:], r.stderr[-2000:])
