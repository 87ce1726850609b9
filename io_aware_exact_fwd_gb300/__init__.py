"""GB300 (sm_103a) exact attention: thin Python binding over the C ABI of libfa.so.

Every function here has the name of the C entry point it calls (include/fa.h)
and only marshals arguments: it checks dtypes, shapes and devices of torch
tensors, passes their device pointers and the current CUDA stream, and raises
``FAError`` on a nonzero status.  All arithmetic runs in the library's CUDA
kernels; there is no fallback.  If libfa.so is missing, importing the binding
still works but every call raises, so a missing build is never silent.

PyTorch is used only as device-memory and stream plumbing.
"""

from __future__ import annotations

import ctypes
import os

__all__ = [
    "FAError", "load_library", "library_path", "fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_bwd_noalloc",
    "fa_bwd_noalloc_max_workspace", "fa_bwd_prep", "fa_bwd_main", "fa_bwd_dq", "fa_fp8_workspace_size",
    "fa_fp8_workspace_offsets", "fa_fp8_prepare", "fa_fp8_prepare_seeded", "fa_fp8_rotation_signs", "fa_fwd_fp8",
    "fa_sync_check",
    "fa_strerror",
    "fa_version", "fa_last_error_site", "fa_debug_set_wait_limit_ns", "fa_debug_set_fault",
    "STATUS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libfa.so")
_lib = None

STATUS = {
    0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_MISALIGNED",
    4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT", 6: "FA_ERR_WORKSPACE",
}


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = STATUS.get(status, str(status))
        if _lib is not None:
            msg += ": " + _lib.fa_strerror(status).decode()
        super().__init__(f"{where}: {msg}")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libfa.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_strerror.restype = ctypes.c_char_p
    lib.fa_strerror.argtypes = [i]
    lib.fa_version.restype = i
    lib.fa_version.argtypes = []
    lib.fa_fwd.restype = i
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, i, f, vp]
    lib.fa_fwd_strided.restype = i
    lib.fa_fwd_strided.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.fa_bwd_strided.restype = i
    lib.fa_bwd_strided.argtypes = [vp] * 17 + [vp, ctypes.c_size_t, i, i, i, i, i, f, i, vp]
    lib.fa_bwd_deterministic.restype = i
    lib.fa_bwd_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, i, f, vp]
    lib.fa_bwd_prep.restype = i
    lib.fa_bwd_prep.argtypes = [vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, vp]
    lib.fa_bwd_main.restype = i
    lib.fa_bwd_main.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, i, f, vp]
    lib.fa_bwd_dq.restype = i
    lib.fa_bwd_dq.argtypes = [vp, ctypes.c_size_t, vp, i, i, i, i, f, vp]
    lib.fa_fp8_workspace_size.restype = ctypes.c_size_t
    lib.fa_fp8_workspace_size.argtypes = [i, i, i, i]
    lib.fa_fp8_workspace_offsets.restype = i
    lib.fa_fp8_workspace_offsets.argtypes = [i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_fp8_prepare.restype = i
    lib.fa_fp8_prepare.argtypes = [vp, vp, vp, i, vp, vp, ctypes.c_size_t, i, i, i, i, vp]
    lib.fa_fp8_prepare_seeded.restype = i
    lib.fa_fp8_prepare_seeded.argtypes = [vp, vp, vp, i, ctypes.c_uint64, vp, ctypes.c_size_t, i, i, i, i, vp]
    lib.fa_fp8_prepare_strided.restype = i
    lib.fa_fp8_prepare_strided.argtypes = [vp, vp, vp, vp, vp, vp, i, vp, ctypes.c_uint64, vp, ctypes.c_size_t, i, i,
                                           i, i, vp]
    lib.fa_fp8_rotation_signs.restype = i
    lib.fa_fp8_rotation_signs.argtypes = [ctypes.c_uint64, i, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, ctypes.c_size_t, vp, vp, i, i, i, i, i, f, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_fp8_dequantize.argtypes = [vp, ctypes.c_size_t, vp, vp, vp, i, i, i, i, vp]
    lib.fa_fp8_dequantize.restype = i
    lib.fa_bwd_fp8_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_fp8_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_fp8.argtypes = [vp, ctypes.c_size_t, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, i, f,
                               i, i, vp]
    lib.fa_bwd_fp8.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.fa_bwd_noalloc_max_workspace.restype = ctypes.c_size_t
    lib.fa_bwd_noalloc_max_workspace.argtypes = []
    lib.fa_splitkv_workspace_size.restype = ctypes.c_size_t
    lib.fa_splitkv_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_splitkv_default_splits.restype = i
    lib.fa_splitkv_default_splits.argtypes = [i, i, i, i, i]
    lib.fa_fwd_splitkv_partial.restype = i
    lib.fa_fwd_splitkv_partial.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.fa_merge_partials.restype = i
    lib.fa_merge_partials.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, i, i, i, f, vp]
    lib.fa_fwd_splitkv_strided.restype = i
    lib.fa_fwd_splitkv_strided.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, i, i,
                                           i, f, vp]
    lib.fa_w4a16_workspace_size.restype = ctypes.c_size_t
    lib.fa_w4a16_workspace_size.argtypes = [i, i, i, i]
    lib.fa_w4a16_default_splits.restype = i
    lib.fa_w4a16_default_splits.argtypes = [i, i, i]
    lib.fa_w4a16_gemm.restype = i
    lib.fa_w4a16_gemm.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, vp]
    lib.fa_sync_check.restype = i
    lib.fa_sync_check.argtypes = [vp]
    lib.fa_last_error_site.restype = ctypes.c_uint
    lib.fa_last_error_site.argtypes = []
    lib.fa_debug_set_wait_limit_ns.restype = None
    lib.fa_debug_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.fa_debug_set_fault.restype = None
    lib.fa_debug_set_fault.argtypes = [i]
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != 0:
        raise FAError(status, where)


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _check_bhnd(name, t, shape, dtype):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous ([B, H, N, d] row-major)")


def _strides(t):
    """(row, head, batch) element strides of a [B, H, N, d] tensor with contiguous d, as int64[3]."""
    arr = (ctypes.c_int64 * 3)(t.stride(2), t.stride(1), t.stride(0))
    return ctypes.cast(arr, ctypes.c_void_p)  # the cast keeps the array alive


def _check_strided(name, t, shape, dtype):
    """Like _check_bhnd, but any layout whose last dimension is contiguous is accepted."""
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.stride(3) != 1:
        raise ValueError(f"{name} must have a contiguous last dimension")


def fa_fwd(q, k, v, o=None, lse=None, causal: bool = False, scale: float | None = None, stream=None):
    """bf16 attention forward: returns (o, lse).

    q, k, v: bf16 CUDA tensors indexed [B, H, N, d] with contiguous d: dense, or any
    strided view such as x.view(B, N, H, d).transpose(1, 2) (fa_fwd_strided).  ``o``
    (bf16 [B,H,N,d], allocated dense if not given, any such layout if given) and
    ``lse`` (fp32 [B,H,N], dense).  ``scale`` defaults to 1/sqrt(d).
    """
    import torch

    lib = load_library()
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_strided(name, t, (B, H, N, d), torch.bfloat16)
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_strided("o", o, (B, H, N, d), torch.bfloat16)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, H, N]")
    if scale is None:
        scale = d ** -0.5
    with torch.cuda.device(q.device):
        if all(t.is_contiguous() for t in (q, k, v, o)):
            st = lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, int(bool(causal)),
                            float(scale), _stream_handle(stream))
        else:
            st = lib.fa_fwd_strided(_ptr(q), _strides(q), _ptr(k), _strides(k), _ptr(v), _strides(v), _ptr(o),
                                    _strides(o), _ptr(lse), B, H, N, d, int(bool(causal)), float(scale),
                                    _stream_handle(stream))
    _check(st, "fa_fwd")
    return o, lse


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    """Bytes of device workspace fa_bwd needs (0 if unsupported)."""
    return int(load_library().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(q, k, v, o, do, lse, dq=None, dk=None, dv=None, workspace=None, causal: bool = False,
           scale: float | None = None, stream=None, deterministic: bool = False):
    """bf16 attention backward (d = 64 or 128): returns (dq, dk, dv).

    q, k, v, o, do: bf16 CUDA tensors [B, H, N, d]; lse: fp32 [B, H, N] from fa_fwd
    with the same causal/scale.  Outputs are allocated if not given; the
    workspace (uint8 CUDA tensor of fa_bwd_workspace_size bytes) too.
    ``deterministic=True`` calls fa_bwd_deterministic (dQ identical bits on every run).
    """
    import torch

    lib = load_library()
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check_strided(name, t, (B, H, N, d), torch.bfloat16)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, H, N]")
    dense = lambda: torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    dq = dense() if dq is None else dq
    dk = dense() if dk is None else dk
    dv = dense() if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_strided(name, t, (B, H, N, d), torch.bfloat16)
    need = int(lib.fa_bwd_workspace_size(B, H, N, d))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if scale is None:
        scale = d ** -0.5
    with torch.cuda.device(q.device):
        if all(t.is_contiguous() for t in (q, k, v, o, do, dq, dk, dv)):
            fn = lib.fa_bwd_deterministic if deterministic else lib.fa_bwd
            st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                    _ptr(workspace), workspace.numel() * workspace.element_size(), B, H, N, d,
                    int(bool(causal)), float(scale), _stream_handle(stream))
        else:
            st = lib.fa_bwd_strided(_ptr(q), _strides(q), _ptr(k), _strides(k), _ptr(v), _strides(v), _ptr(o),
                                    _strides(o), _ptr(do), _strides(do), _ptr(lse), _ptr(dq), _strides(dq), _ptr(dk),
                                    _strides(dk), _ptr(dv), _strides(dv), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), B, H, N, d, int(bool(causal)),
                                    float(scale), int(bool(deterministic)), _stream_handle(stream))
    _check(st, "fa_bwd_deterministic" if deterministic else "fa_bwd")
    return dq, dk, dv


def _ws_bytes(workspace):
    return workspace.numel() * workspace.element_size()


def fa_bwd_prep(o, do, lse, workspace, stream=None):
    """Backward stage 1: D = rowsum(dO * O), LSE * log2(e) and a zeroed dQ accumulator in `workspace`."""
    lib = load_library()
    B, H, N, d = o.shape
    with __import__("torch").cuda.device(o.device):
        st = lib.fa_bwd_prep(_ptr(o), _ptr(do), _ptr(lse), _ptr(workspace), _ws_bytes(workspace), B, H, N, d,
                             _stream_handle(stream))
    _check(st, "fa_bwd_prep")


def fa_bwd_main(q, k, v, do, dk, dv, workspace, causal: bool = False, scale: float | None = None, stream=None):
    """Backward stage 2: dK, dV and the fp32 dQ accumulator (needs fa_bwd_prep's workspace)."""
    lib = load_library()
    B, H, N, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    with __import__("torch").cuda.device(q.device):
        st = lib.fa_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dk), _ptr(dv), _ptr(workspace),
                             _ws_bytes(workspace), B, H, N, d, int(bool(causal)), float(scale),
                             _stream_handle(stream))
    _check(st, "fa_bwd_main")


def fa_bwd_dq(workspace, dq, scale: float | None = None, stream=None):
    """Backward stage 3: dq = bf16(scale * accumulator)."""
    lib = load_library()
    B, H, N, d = dq.shape
    scale = d ** -0.5 if scale is None else scale
    with __import__("torch").cuda.device(dq.device):
        st = lib.fa_bwd_dq(_ptr(workspace), _ws_bytes(workspace), _ptr(dq), B, H, N, d, float(scale),
                           _stream_handle(stream))
    _check(st, "fa_bwd_dq")


def fa_fp8_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa_fp8_workspace_size(B, H, N, d))


def fa_fp8_workspace_offsets(B: int, H: int, N: int, d: int) -> dict:
    """Byte offsets of the FP8 workspace regions (q8, k8, v8t, sq, sk, sv) plus npad and ntiles."""
    arr = (ctypes.c_size_t * 8)()
    _check(load_library().fa_fp8_workspace_offsets(B, H, N, d, arr), "fa_fp8_workspace_offsets")
    keys = ("q8", "k8", "v8t", "sq", "sk", "sv", "npad", "ntiles")
    return {kk: int(arr[i]) for i, kk in enumerate(keys)}


def _fp8_prepare_call(q, k, v, signs, seed, workspace, stream, name):
    import torch

    lib = load_library()
    B, H, N, d = q.shape
    dt = q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise TypeError("q, k, v must be float32 or bfloat16")
    for nm, t in (("q", q), ("k", k), ("v", v)):
        _check_strided(nm, t, (B, H, N, d), dt)
    if signs is not None and (signs.dtype != torch.int8 or tuple(signs.shape) != (d,) or not signs.is_cuda):
        raise ValueError("signs must be an int8 CUDA tensor of shape [d]")
    if workspace is None:
        workspace = torch.empty(max(fa_fp8_workspace_size(B, H, N, d), 1), dtype=torch.uint8, device=q.device)
    in_dtype = 1 if dt == torch.bfloat16 else 0
    seed64 = ctypes.c_uint64(seed & (2 ** 64 - 1))
    with torch.cuda.device(q.device):
        if not all(t.is_contiguous() for t in (q, k, v)):
            st = lib.fa_fp8_prepare_strided(_ptr(q), _strides(q), _ptr(k), _strides(k), _ptr(v), _strides(v),
                                            in_dtype, _ptr(signs) if signs is not None else None, seed64,
                                            _ptr(workspace), _ws_bytes(workspace), B, H, N, d, _stream_handle(stream))
        elif signs is not None:
            st = lib.fa_fp8_prepare(_ptr(q), _ptr(k), _ptr(v), in_dtype, _ptr(signs), _ptr(workspace),
                                    _ws_bytes(workspace), B, H, N, d, _stream_handle(stream))
        else:
            st = lib.fa_fp8_prepare_seeded(_ptr(q), _ptr(k), _ptr(v), in_dtype, seed64, _ptr(workspace),
                                           _ws_bytes(workspace), B, H, N, d, _stream_handle(stream))
    _check(st, name)
    return workspace


def fa_fp8_prepare(q, k, v, signs, workspace=None, stream=None):
    """Rotate Q, K and block-quantise Q, K, V to e4m3 into `workspace` (allocated if None); returns it.

    q, k, v: fp32 or bf16 CUDA tensors [B, H, N, d] with contiguous d: dense, or any
    strided view (fa_fp8_prepare_strided); signs: int8 CUDA tensor [d] (+-1).
    """
    if signs is None:
        raise ValueError("signs must be given (fa_fp8_prepare_seeded draws them from a seed)")
    return _fp8_prepare_call(q, k, v, signs, 0, workspace, stream, "fa_fp8_prepare")


def fa_fp8_prepare_seeded(q, k, v, seed: int, workspace=None, stream=None):
    """fa_fp8_prepare with the rotation signs drawn from a 64-bit seed on the device; returns the workspace."""
    return _fp8_prepare_call(q, k, v, None, seed, workspace, stream, "fa_fp8_prepare_seeded")


def fa_fp8_rotation_signs(seed: int, d: int):
    """The +-1 signs (int8 CPU tensor [d]) fa_fp8_prepare_seeded uses for ``seed``."""
    import torch

    out = torch.empty(d, dtype=torch.int8)
    _check(load_library().fa_fp8_rotation_signs(ctypes.c_uint64(seed & (2 ** 64 - 1)), d,
                                                 ctypes.c_void_p(out.data_ptr())), "fa_fp8_rotation_signs")
    return out


def fa_fwd_fp8(workspace, shape, o=None, lse=None, causal: bool = False, scale: float | None = None, stream=None):
    """FP8 forward from a prepared workspace; shape = (B, H, N, d).  Returns (o bf16, lse fp32)."""
    import torch

    lib = load_library()
    B, H, N, d = shape
    dev = workspace.device
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    _check_bhnd("o", o, (B, H, N, d), torch.bfloat16)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, H, N]")
    if scale is None:
        scale = d ** -0.5
    with torch.cuda.device(dev):
        st = lib.fa_fwd_fp8(_ptr(workspace), _ws_bytes(workspace), _ptr(o), _ptr(lse), B, H, N, d,
                            int(bool(causal)), float(scale), _stream_handle(stream))
    _check(st, "fa_fwd_fp8")
    return o, lse


def fa_fp8_dequantize(workspace, shape, stream=None):
    """The FP8 backward's bf16 operands (Q', K', V') from a prepared workspace; shape = (B, H, N, d)."""
    import torch

    lib = load_library()
    B, H, N, d = shape
    out = [torch.empty((B, H, N, d), dtype=torch.bfloat16, device=workspace.device) for _ in range(3)]
    with torch.cuda.device(workspace.device):
        st = lib.fa_fp8_dequantize(_ptr(workspace), _ws_bytes(workspace), _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                                   B, H, N, d, _stream_handle(stream))
    _check(st, "fa_fp8_dequantize")
    return tuple(out)


def fa_bwd_fp8_workspace_size(B: int, H: int, N: int, d: int) -> int:
    """Bytes of device workspace fa_bwd_fp8 needs (0 if unsupported)."""
    return int(load_library().fa_bwd_fp8_workspace_size(B, H, N, d))


def fa_bwd_fp8(fp8_workspace, signs, o, do, lse, dq=None, dk=None, dv=None, workspace=None, causal: bool = False,
               scale: float | None = None, deterministic: bool = False, recompute_forward: bool = False,
               stream=None):
    """Straight-through backward of the FP8 attention (d = 64 or 128): returns (dq, dk, dv), bf16.

    fp8_workspace: filled by fa_fp8_prepare; signs: the int8 [d] signs given to it;
    o, lse: the forward's outputs (bf16 [B, H, N, d], fp32 [B, H, N]), ignored and
    may be None when ``recompute_forward`` (O and LSE recomputed in bf16 from the
    FP8 operands, so that D uses the unrounded probabilities); do: bf16
    [B, H, N, d]; scale: the softmax scale given to fa_fwd_fp8.
    """
    import torch

    lib = load_library()
    B, H, N, d = do.shape
    _check_bhnd("do", do, (B, H, N, d), torch.bfloat16)
    if not recompute_forward:
        _check_bhnd("o", o, (B, H, N, d), torch.bfloat16)
        if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
            raise ValueError("lse must be a contiguous float32 tensor [B, H, N]")
    if signs.dtype != torch.int8 or tuple(signs.shape) != (d,) or not signs.is_cuda:
        raise ValueError("signs must be an int8 CUDA tensor of shape [d]")
    dense = lambda: torch.empty((B, H, N, d), dtype=torch.bfloat16, device=do.device)
    dq = dense() if dq is None else dq
    dk = dense() if dk is None else dk
    dv = dense() if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, (B, H, N, d), torch.bfloat16)
    if workspace is None:
        workspace = torch.empty(max(fa_bwd_fp8_workspace_size(B, H, N, d), 1), dtype=torch.uint8, device=do.device)
    if scale is None:
        scale = d ** -0.5
    with torch.cuda.device(do.device):
        st = lib.fa_bwd_fp8(_ptr(fp8_workspace), _ws_bytes(fp8_workspace), _ptr(signs),
                            None if recompute_forward else _ptr(o), _ptr(do),
                            None if recompute_forward else _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                            _ws_bytes(workspace), B, H, N, d, int(bool(causal)), float(scale),
                            int(bool(deterministic)), int(bool(recompute_forward)), _stream_handle(stream))
    _check(st, "fa_bwd_fp8")
    return dq, dk, dv


def fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, causal: bool = False, scale: float | None = None,
                   stream=None):
    """fa_bwd for callers that cannot allocate device memory: no workspace argument.

    The library supplies the scratch from a fixed per-device buffer of
    fa_bwd_noalloc_max_workspace() bytes (larger problems raise FAError with
    FA_ERR_WORKSPACE).  The caller passes every input and output tensor; this
    function allocates nothing.  Calls that overlap on the GPU share that buffer
    and must be serialised.
    """
    import torch

    lib = load_library()
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, (B, H, N, d), torch.bfloat16)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, H, N]")
    if scale is None:
        scale = d ** -0.5
    with torch.cuda.device(q.device):
        st = lib.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                                _ptr(dv), B, H, N, d, int(bool(causal)), float(scale), _stream_handle(stream))
    _check(st, "fa_bwd_noalloc")
    return dq, dk, dv


def fa_bwd_noalloc_max_workspace() -> int:
    return int(load_library().fa_bwd_noalloc_max_workspace())


def fa_splitkv_workspace_size(B: int, H: int, Nq: int, d: int, n_split: int) -> int:
    return int(load_library().fa_splitkv_workspace_size(B, H, Nq, d, n_split))


def fa_splitkv_default_splits(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(load_library().fa_splitkv_default_splits(B, H, Nq, Nk, d))


def _check_kv(q, k, v):
    import torch

    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    _check_bhnd("q", q, (B, H, Nq, d), torch.bfloat16)
    _check_bhnd("k", k, (B, H, Nk, d), torch.bfloat16)
    _check_bhnd("v", v, (B, H, Nk, d), torch.bfloat16)
    return B, H, Nq, Nk, d


def fa_fwd_splitkv_partial(q, k, v, n_split: int, o_part=None, lse_part=None, causal: bool = False,
                           scale: float | None = None, stream=None):
    """Split-KV partials: returns (o_part fp32 [n, B, H, Nq, d], lse_part fp32 [n, B, H, Nq]).

    q: bf16 [B, H, Nq, d]; k, v: bf16 [B, H, Nk, d].  Causal queries are the last Nq
    positions (query i sees key j iff j <= i + Nk - Nq).
    """
    import torch

    lib = load_library()
    B, H, Nq, Nk, d = _check_kv(q, k, v)
    if o_part is None:
        o_part = torch.empty((n_split, B, H, Nq, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((n_split, B, H, Nq), dtype=torch.float32, device=q.device)
    _check_bhnd("o_part", o_part.view(n_split * B, H, Nq, d), (n_split * B, H, Nq, d), torch.float32)
    _check_bhnd("lse_part", lse_part.view(n_split * B, H, Nq, 1), (n_split * B, H, Nq, 1), torch.float32)
    sc = float(scale) if scale is not None else d ** -0.5
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_splitkv_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(o_part), _ptr(lse_part), B, H, Nq, Nk, d,
                                        n_split, int(bool(causal)), sc, _stream_handle(stream))
    _check(st, "fa_fwd_splitkv_partial")
    return o_part, lse_part


def fa_merge_partials(o_part, lse_part, o=None, lse=None, stream=None):
    """Exact merge of split-KV partials: returns (o bf16 [B, H, Nq, d], lse fp32 [B, H, Nq])."""
    import torch

    lib = load_library()
    n_split, B, H, Nq, d = o_part.shape
    _check_bhnd("o_part", o_part.view(n_split * B, H, Nq, d), (n_split * B, H, Nq, d), torch.float32)
    _check_bhnd("lse_part", lse_part.view(n_split * B, H, Nq, 1), (n_split * B, H, Nq, 1), torch.float32)
    if o is None:
        o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=o_part.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=o_part.device)
    _check_bhnd("o", o, (B, H, Nq, d), torch.bfloat16)
    _check_bhnd("lse", lse.view(B, H, Nq, 1), (B, H, Nq, 1), torch.float32)
    with torch.cuda.device(o_part.device):
        st = lib.fa_merge_partials(_ptr(o_part), _ptr(lse_part), _ptr(o), _ptr(lse), n_split, B, H, Nq, d,
                                   _stream_handle(stream))
    _check(st, "fa_merge_partials")
    return o, lse


def fa_fwd_splitkv(q, k, v, o=None, lse=None, workspace=None, n_split: int = 0, causal: bool = False,
                   scale: float | None = None, stream=None):
    """Split-KV attention (partials + merge): returns (o bf16 [B, H, Nq, d], lse fp32 [B, H, Nq]).

    q, k, v, o: bf16 CUDA tensors with contiguous d, dense or any strided view
    (fa_fwd_splitkv_strided).  n_split <= 0 picks the library's default split count.
    """
    import torch

    lib = load_library()
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    _check_strided("q", q, (B, H, Nq, d), torch.bfloat16)
    _check_strided("k", k, (B, H, Nk, d), torch.bfloat16)
    _check_strided("v", v, (B, H, Nk, d), torch.bfloat16)
    n = n_split if n_split > 0 else max(1, fa_splitkv_default_splits(B, H, Nq, Nk, d))
    if o is None:
        o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _check_strided("o", o, (B, H, Nq, d), torch.bfloat16)
    _check_bhnd("lse", lse.view(B, H, Nq, 1), (B, H, Nq, 1), torch.float32)
    if workspace is None:
        workspace = torch.empty(max(fa_splitkv_workspace_size(B, H, Nq, d, n), 1), dtype=torch.uint8,
                                device=q.device)
    sc = float(scale) if scale is not None else d ** -0.5
    with torch.cuda.device(q.device):
        if all(t.is_contiguous() for t in (q, k, v, o)):
            st = lib.fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                    _ws_bytes(workspace), B, H, Nq, Nk, d, n, int(bool(causal)), sc,
                                    _stream_handle(stream))
        else:
            st = lib.fa_fwd_splitkv_strided(_ptr(q), _strides(q), _ptr(k), _strides(k), _ptr(v), _strides(v), _ptr(o),
                                            _strides(o), _ptr(lse), _ptr(workspace), _ws_bytes(workspace), B, H, Nq,
                                            Nk, d, n, int(bool(causal)), sc, _stream_handle(stream))
    _check(st, "fa_fwd_splitkv")
    return o, lse


def fa_w4a16_workspace_size(M: int, N: int, K: int, n_split: int) -> int:
    return int(load_library().fa_w4a16_workspace_size(M, N, K, n_split))


def fa_w4a16_default_splits(M: int, N: int, K: int) -> int:
    return int(load_library().fa_w4a16_default_splits(M, N, K))


def fa_w4a16_gemm(x, wq, scales, zeros, y=None, workspace=None, n_split: int = 0, stream=None):
    """Y = X W^T with W given as packed 4-bit codes (see fa_w4a16_gemm in include/fa.h).

    x: fp16 [M, K]; wq: int32 [N, K/8]; scales: fp16 [K/128, N]; zeros: uint8 [K/128, N];
    all CUDA, contiguous.  Returns y (fp16 [M, N]).
    """
    import torch

    lib = load_library()
    M, K = x.shape
    N = wq.shape[0]
    for name, t, shape, dt in (("x", x, (M, K), torch.float16), ("wq", wq, (N, K // 8), torch.int32),
                               ("scales", scales, (K // 128, N), torch.float16),
                               ("zeros", zeros, (K // 128, N), torch.uint8)):
        if t.dtype != dt or tuple(t.shape) != shape or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor of shape {shape}")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    n = n_split if n_split > 0 else max(1, int(lib.fa_w4a16_default_splits(M, N, K)))
    need = int(lib.fa_w4a16_workspace_size(M, N, K, n))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        st = lib.fa_w4a16_gemm(_ptr(x), _ptr(wq), _ptr(scales), _ptr(zeros), _ptr(y), _ptr(workspace),
                               0 if workspace is None else _ws_bytes(workspace), M, N, K, n, _stream_handle(stream))
    _check(st, "fa_w4a16_gemm")
    return y


def fa_sync_check(stream=None):
    """Synchronise the stream and raise FAError if a kernel reported an error."""
    lib = load_library()
    _check(lib.fa_sync_check(_stream_handle(stream)), "fa_sync_check")


def fa_strerror(status: int) -> str:
    return load_library().fa_strerror(status).decode()


def fa_version() -> int:
    return load_library().fa_version()


def fa_last_error_site() -> int:
    return load_library().fa_last_error_site()


def fa_debug_set_wait_limit_ns(ns: int):
    load_library().fa_debug_set_wait_limit_ns(int(ns))


def fa_debug_set_fault(fault: int):
    load_library().fa_debug_set_fault(int(fault))
