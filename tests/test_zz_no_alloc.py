"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (a plugin inside a framework that owns all device memory, or a
loop where cudaMalloc's possible device-wide synchronisation is not allowed)
pass inputs and outputs only; the library supplies the scratch from a fixed
per-device buffer.  This test calls the new entry point through the C ABI and
checks it against fa_bwd, the entry point with a caller workspace, on two calls
in a row (the buffer keeps the previous call's contents, so the second call
also shows that everything that must start at zero is cleared).  This file is
collected last so that a run stopping at its first failure has already run
every other test; it also passes alone in a fresh process.
"""

import ctypes

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
