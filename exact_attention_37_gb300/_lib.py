"""ctypes binding of the C ABI in include/fa_attention.h -- argument marshalling only.

Every step of the computation runs in the CUDA kernels of ``libfa_attention.so``;
this module turns torch tensors into pointers, sizes and the current stream,
and turns status codes into exceptions.  There is no fallback: if the library
is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa_attention.so")

FA_OK = 0
STATUS = {
    0: "FA_OK",
    1: "FA_ERR_INVALID_ARG",
    2: "FA_ERR_UNSUPPORTED",
    3: "FA_ERR_MISALIGNED",
    4: "FA_ERR_WORKSPACE",
    5: "FA_ERR_CUDA",
    6: "FA_ERR_DEVICE_TIMEOUT",
    7: "FA_ERR_DEVICE_CHECK",
}
FA_FP16, FA_BF16 = 0, 1

# Every symbol the header declares, with (restype, argtypes).
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "fa_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "fa_bwd_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "fa_bwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _i, _f, _i, _i,
                       _vp]),
    "fa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "fa_host_scratch_size": (_sz, [_i, _i, _i, _i, _i]),
    "fa_host_chunk_plan": (_i, [_i, _i, _i, _i, ctypes.POINTER(ctypes.c_int), _i]),
    "fa_cta_head_group": (_i, [ctypes.c_longlong, _i, _sz, _i, _i]),
    "fa_fwd_host": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _f, _i, _i, _i, _vp]),
    "fa_fwd_bwd_host": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _f, _i, _i, _i,
                             _vp]),
    "fa_check_device_status": (_i, [_vp]),
    "fa_selftest_wait_timeout": (_i, [ctypes.c_uint32, _vp]),
    "fa_selftest_device_check": (_i, [_i, _vp]),
    "fa_last_device_error_bits": (ctypes.c_uint32, []),
    "fa_last_device_error_detail": (None, [_vp]),
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_profile_begin": (_i, [_i]),
    "fa_profile_end": (_i, [_vp, _vp, _i]),
    "fa_version": (ctypes.c_uint32, []),
}


class FaError(RuntimeError):
    def __init__(self, where: str, code: int, detail=None):
        extra = f" (device record {detail})" if detail else ""
        super().__init__(f"{where} failed: {STATUS.get(code, code)}{extra}")
        self.code = code
        self.detail = detail


_lib = None


def open_library(path: str):
    """Open a build of the library at ``path`` and declare its signatures (no caching)."""
    if not os.path.exists(path):
        raise FaError(f"loading {os.path.basename(path)} (not built; run exact_attention_37_gb300.build)", -1)
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str = LIB_PATH):
    """Load the shared library (once) and declare its signatures.  Raises if it is missing."""
    global _lib
    if _lib is None:
        _lib = open_library(path)
    return _lib


def _check(where: str, code: int):
    if code != FA_OK:
        raise FaError(where, code)


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float16:
        return FA_FP16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: fp16 or bf16 only")


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(int(x) for x in q.shape)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check_shapes(q, k, v):
    B, H, Nq, d = _shape(q)
    Bk, Hkv, Nk, dk = _shape(k)
    if tuple(v.shape) != tuple(k.shape) or Bk != B or dk != d:
        raise ValueError("k and v must be [B, H_kv, N_k, d] with q's B and d")
    if Hkv < 1 or H % Hkv:
        raise ValueError("the key/value head count must divide the query head count")
    return B, H, Hkv, Nq, Nk, d


def fa_fwd(q, k, v, o, lse, scale: float, causal: bool, stream=None):
    """O and L into caller-owned ``o`` [B,H,N_q,d] and ``lse`` [B,H,N_q] fp32 (all CUDA, contiguous).

    k, v: [B, H_kv, N_k, d] (H_kv divides H; N_k may differ from N_q)."""
    lib = load()
    B, H, Hkv, Nq, Nk, d = _check_shapes(q, k, v)
    for t in (q, k, v, o, lse):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    code = lib.fa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Nq, Nk, d, float(scale),
                         int(bool(causal)), _dtype_code(q), _stream(stream))
    _check("fa_fwd_ex", code)


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale: float, causal: bool, stream=None):
    """dQ, dK, dV into caller-owned tensors; ``workspace`` is a CUDA uint8 tensor of at least
    fa_bwd_workspace_size(B, H, N_q, d) bytes."""
    lib = load()
    B, H, Hkv, Nq, Nk, d = _check_shapes(q, k, v)
    for t in (q, k, v, o, dout, lse, dq, dk, dv):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    code = lib.fa_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                         _ptr(workspace), ws_bytes, B, H, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                         _dtype_code(q), _stream(stream))
    _check("fa_bwd_ex", code)


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, scale: float, causal: bool, stream=None):
    """fa_bwd with the library's fixed device scratch instead of a caller workspace (no allocation)."""
    lib = load()
    B, H, N, d = _shape(q)
    for t in (q, k, v, o, dout, lse, dq, dk, dv):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    code = lib.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                              _ptr(dv), B, H, N, d, float(scale), int(bool(causal)), _dtype_code(q), _stream(stream))
    _check("fa_bwd_noalloc", code)


def fa_host_scratch_size(B: int, H: int, N: int, d: int, backward: bool = True) -> int:
    return int(load().fa_host_scratch_size(B, H, N, d, int(bool(backward))))


def fa_host_chunk_plan(B: int, H: int, N: int, chunks: int = 0) -> list:
    """Heads per chunk of the host-buffer pipeline for these sizes (host query)."""
    plan = (ctypes.c_int * 64)()
    n = load().fa_host_chunk_plan(B, H, N, chunks, plan, 64)
    if n < 0:
        raise FaError("fa_host_chunk_plan", 1)
    return list(plan[:n])


def fa_cta_head_group(nheads: int, nblocks: int, bytes_per_head: int, causal: bool, num_sms: int) -> int:
    """Heads per group of the kernels' CTA order (host query)."""
    g = load().fa_cta_head_group(nheads, nblocks, bytes_per_head, int(bool(causal)), num_sms)
    if g < 0:
        raise FaError("fa_cta_head_group", 1)
    return int(g)


def _host_tensors(*ts):
    for t in ts:
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host entry points take contiguous CPU tensors (pinned for overlap)")


def fa_fwd_host(q, k, v, o, lse, scratch, scale: float, causal: bool, chunks: int = 0, stream=None):
    """Forward pass on host tensors (q, k, v, o [B,H,N,d]; lse [B,H,N] fp32) through a CUDA
    ``scratch`` (uint8) of at least fa_host_scratch_size(B, H, N, d, False) bytes."""
    lib = load()
    B, H, N, d = _shape(q)
    _host_tensors(q, k, v, o, lse)
    code = lib.fa_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(scratch),
                           scratch.numel() * scratch.element_size(), B, H, N, d, float(scale), int(bool(causal)),
                           _dtype_code(q), int(chunks), _stream(stream))
    _check("fa_fwd_host", code)


def fa_fwd_bwd_host(q, k, v, dout, o, lse, dq, dk, dv, scratch, scale: float, causal: bool, chunks: int = 0,
                    stream=None):
    """Forward and backward pass on host tensors through a CUDA ``scratch`` (uint8) of at
    least fa_host_scratch_size(B, H, N, d, True) bytes; outputs valid after ``stream`` syncs."""
    lib = load()
    B, H, N, d = _shape(q)
    _host_tensors(q, k, v, dout, o, lse, dq, dk, dv)
    code = lib.fa_fwd_bwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(o), _ptr(lse), _ptr(dq), _ptr(dk),
                               _ptr(dv), _ptr(scratch), scratch.numel() * scratch.element_size(), B, H, N, d,
                               float(scale), int(bool(causal)), _dtype_code(q), int(chunks), _stream(stream))
    _check("fa_fwd_bwd_host", code)


def fa_check_device_status(stream=None):
    """Synchronize and raise FaError(FA_ERR_DEVICE_TIMEOUT) if a kernel gave up on a wait."""
    lib = load()
    code = lib.fa_check_device_status(_stream(stream))
    if code != FA_OK:
        rec = (ctypes.c_uint32 * 4)()
        lib.fa_last_device_error_detail(rec)
        raise FaError("fa_check_device_status", code, [int(x) for x in rec])


def fa_selftest_wait_timeout(limit_us: int, stream=None):
    """Launch the failure-detection self-test (a wait that gives up after ``limit_us``);
    the next fa_check_device_status reports it."""
    _check("fa_selftest_wait_timeout", load().fa_selftest_wait_timeout(int(limit_us), _stream(stream)))


PROFILE_KINDS = {0: "fwd", 1: "bwd_kv", 2: "bwd_q", 3: "bwd_fused"}


def fa_profile_begin(n: int):
    """Record the time of each of the next ``n`` main-kernel launches of fa_fwd / fa_bwd."""
    _check("fa_profile_begin", load().fa_profile_begin(int(n)))


def fa_profile_end(max_out: int = 65536):
    """Wait for the recorded events; returns [(kind, ms)] in launch order, kind one of
    PROFILE_KINDS' names."""
    ms = (ctypes.c_float * max_out)()
    kind = (ctypes.c_int * max_out)()
    n = load().fa_profile_end(ms, kind, max_out)
    if n < 0:
        raise FaError("fa_profile_end", 5)
    return [(PROFILE_KINDS.get(kind[i], str(kind[i])), float(ms[i])) for i in range(n)]


def fa_status_string(code: int) -> str:
    return load().fa_status_string(int(code)).decode()


def fa_version() -> int:
    return int(load().fa_version())
