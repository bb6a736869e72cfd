"""Channelwise gated delta rule for GB300 (sm_103a): Python binding of libcgdr.

This module only marshals arguments: it turns torch tensors into the
``cgdr_args`` block of ``include/cgdr.h`` (device pointers and element
strides) and calls the C ABI on the current CUDA stream.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback.  If ``libcgdr.so`` is missing, calls raise ``RuntimeError``; build
it with ``gated_delta_rule_channelwise_gb300.build.build()``.

Public calls (same names as the C ABI without the ``cgdr_`` prefix):

* :func:`decode` -- one T = 1 step for every (batch, v-head).
* :func:`prefill` -- chunked prefill over T tokens.
* :func:`prefill_noalloc` -- prefill with the library's static scratch instead of a workspace.
* :func:`prefill_workspace_size`, :func:`workspace_status`, :func:`validate`, :func:`status_string`.
* :func:`prefill_path_for` -- which prefill kernel a call runs.

The prefill kernel is chosen per call (``path=``, one of the ``PREFILL_*``
codes; ``PREFILL_AUTO`` by default): the choice travels in the argument
block, so concurrent calls never affect each other.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcgdr.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS, ERR_RANGE = range(9)
F32, BF16 = 0, 1
GATE_CHANNEL, GATE_GDN = 0, 1
PREFILL_AUTO, PREFILL_PER_HEAD, PREFILL_CLUSTER, PREFILL_SIMT, PREFILL_RECURRENT, PREFILL_COOP = range(6)


class CgdrArgs(ctypes.Structure):
    """Mirror of ``struct cgdr_args`` in include/cgdr.h."""
    _i64 = ctypes.c_int64
    _fields_ = [
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("Hk", ctypes.c_int32), ("Hv", ctypes.c_int32),
        ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("gate", ctypes.c_int32), ("l2norm_qk", ctypes.c_int32),
        ("chunk", ctypes.c_int32), ("o_dtype", ctypes.c_int32),
        ("prefill_path", ctypes.c_int32), ("wait_polls", ctypes.c_int32),
        ("q_scale", ctypes.c_float), ("eps", ctypes.c_float),
        ("q", ctypes.c_void_p), ("q_sb", _i64), ("q_st", _i64), ("q_sh", _i64),
        ("k", ctypes.c_void_p), ("k_sb", _i64), ("k_st", _i64), ("k_sh", _i64),
        ("v", ctypes.c_void_p), ("v_sb", _i64), ("v_st", _i64), ("v_sh", _i64),
        ("g", ctypes.c_void_p), ("g_sb", _i64), ("g_st", _i64), ("g_sh", _i64),
        ("beta", ctypes.c_void_p), ("beta_sb", _i64), ("beta_st", _i64), ("beta_sh", _i64),
        ("a", ctypes.c_void_p), ("a_sb", _i64), ("a_st", _i64), ("a_sh", _i64),
        ("b", ctypes.c_void_p), ("b_sb", _i64), ("b_st", _i64), ("b_sh", _i64),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("state", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("o_sb", _i64), ("o_st", _i64), ("o_sh", _i64),
        ("status", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None

# (name, restype, argtypes) of every symbol include/cgdr.h declares.
_SIGNATURES = [
    ("cgdr_abi_version", ctypes.c_int, []),
    ("cgdr_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("cgdr_validate", ctypes.c_int, [ctypes.POINTER(CgdrArgs), ctypes.c_int]),
    ("cgdr_decode", ctypes.c_int, [ctypes.POINTER(CgdrArgs), ctypes.c_void_p]),
    ("cgdr_prefill_workspace_size", ctypes.c_size_t, [ctypes.POINTER(CgdrArgs)]),
    ("cgdr_prefill", ctypes.c_int, [ctypes.POINTER(CgdrArgs), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    ("cgdr_workspace_status", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    ("cgdr_prefill_noalloc", ctypes.c_int, [ctypes.POINTER(CgdrArgs), ctypes.c_void_p]),
    ("cgdr_prefill_path_for", ctypes.c_int, [ctypes.POINTER(CgdrArgs)]),
]


def lib():
    """The loaded libcgdr (ctypes.CDLL).  Raises if the library was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libcgdr.so is not built (%s); run gated_delta_rule_channelwise_gb300.build.build()"
                                   % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            for name, res, args in _SIGNATURES:
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


class CgdrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


def status_string(status: int) -> str:
    return lib().cgdr_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise CgdrError(status, where)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % t.dtype)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check_status(status):
    import torch
    if status is not None and (not status.is_cuda or status.dtype != torch.int32 or status.numel() < 1):
        raise TypeError("status must be an int32 CUDA tensor")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("every tensor must live on a CUDA device (the library has no CPU path)")


def _ptr_strides(t, name):
    """(data pointer, batch, token, head strides) of a 4-d view with a contiguous last dimension."""
    st = t.stride()
    if st[3] != 1:
        raise ValueError("%s: innermost dimension must be contiguous" % name)
    return (t.data_ptr(), st[0], st[1], st[2])


_NONE4 = (None, 0, 0, 0)


def make_args(q, k, v, state, o, *, T, g=None, beta=None, a=None, b=None, A_log=None, dt_bias=None,
              l2norm=True, q_scale=None, eps=None, chunk=0, path=PREFILL_AUTO, wait_polls=0,
              status=None) -> CgdrArgs:
    """Fill a ``cgdr_args`` block from 4-d views ``[B, T, H, d]`` (token dim included).

    Gate tensors are ``g [B,T,Hv,dk]`` and ``beta [B,T,Hv]`` (channel gate) or
    ``a, b [B,T,Hv]`` with ``A_log, dt_bias [Hv]`` (GatedDeltaNet gate).  ``path`` is the
    prefill kernel of the call, ``wait_polls`` the polls of a bounded device wait (0: the
    library's default; small values are for failure-path tests) and ``status`` an optional
    int32 device tensor that receives ``ERR_TIMEOUT`` if a wait gives up, or ``ERR_RANGE`` if a
    tensor-core prefill met a value beyond the fp16 range in one of its fp16 operands.
    The block is built in one constructor call (field order of ``struct cgdr_args``).
    """
    B, _, Hk, dk = q.shape
    _, _, Hv, dv = v.shape
    if not state.is_contiguous():
        raise ValueError("state must be a dense [B, Hv, dk, dv] fp32 tensor")
    if g is not None:
        gate = GATE_CHANNEL
        gg = _ptr_strides(g, "g")
        bs = beta.stride()
        bb = (beta.data_ptr(), bs[0], bs[1], bs[2])
        aa = ab = _NONE4
        alog = dtb = None
    else:
        gate = GATE_GDN
        gg = bb = _NONE4
        sa, sb = a.stride(), b.stride()
        aa = (a.data_ptr(), sa[0], sa[1], sa[2])
        ab = (b.data_ptr(), sb[0], sb[1], sb[2])
        alog, dtb = A_log.data_ptr(), dt_bias.data_ptr()
    return CgdrArgs(B, T, Hk, Hv, dk, dv, _dtype_code(q), gate, 1 if l2norm else 0, int(chunk), _dtype_code(o),
                    int(path), int(wait_polls),
                    float(q_scale) if q_scale is not None else 0.0, float(eps) if eps is not None else -1.0,
                    *_ptr_strides(q, "q"), *_ptr_strides(k, "k"), *_ptr_strides(v, "v"), *gg, *bb, *aa, *ab,
                    alog, dtb, state.data_ptr(), *_ptr_strides(o, "o"),
                    status.data_ptr() if status is not None else None)


def _check_types(q, k, v, state, o, g, beta, a, b, A_log, dt_bias):
    import torch
    _need_cuda(q, k, v, state, o, g, beta, a, b, A_log, dt_bias)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if o.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("o must be float32 or bfloat16")
    if state.dtype != torch.float32:
        raise TypeError("state must be float32")
    for name, t in (("g", g), ("beta", beta), ("A_log", A_log), ("dt_bias", dt_bias)):
        if t is not None and t.dtype != torch.float32:
            raise TypeError("%s must be float32" % name)
    for name, t in (("a", a), ("b", b)):
        if t is not None and t.dtype != q.dtype:
            raise TypeError("%s must have the dtype of q" % name)


def decode(q, k, v, state, o=None, *, g=None, beta=None, a=None, b=None, A_log=None, dt_bias=None,
           l2norm=True, q_scale=None, eps=None, status=None, wait_polls=0, stream=None):
    """One decode step.  q, k ``[B,Hk,dk]``; v ``[B,Hv,dv]``; state ``[B,Hv,dk,dv]`` fp32
    (updated in place); gate ``g [B,Hv,dk]`` + ``beta [B,Hv]`` or ``a, b [B,Hv]`` +
    ``A_log, dt_bias [Hv]``.  Returns o ``[B,Hv,dv]``: the given ``o`` (fp32 or bf16) or a
    new fp32 tensor (allocated through torch's caching allocator).  ``status``: optional
    int32 device tensor that receives ``ERR_TIMEOUT`` if a bounded wait gives up."""
    import torch
    if o is None:
        o = torch.empty(v.shape, dtype=torch.float32, device=v.device)
    _check_types(q, k, v, state, o, g, beta, a, b, A_log, dt_bias)
    _check_status(status)
    u = lambda t: None if t is None else t.unsqueeze(1)
    A = make_args(u(q), u(k), u(v), state, u(o), T=1, g=u(g), beta=u(beta), a=u(a), b=u(b),
                  A_log=A_log, dt_bias=dt_bias, l2norm=l2norm, q_scale=q_scale, eps=eps,
                  wait_polls=wait_polls, status=status)
    _check(lib().cgdr_decode(ctypes.byref(A), _stream_handle(stream)), "cgdr_decode")
    return o


def prefill_workspace_size(q, k, v, state, o, **kw) -> int:
    A = make_args(q, k, v, state, o, T=q.shape[1], **kw)
    return int(lib().cgdr_prefill_workspace_size(ctypes.byref(A)))


def prefill(q, k, v, state, o=None, *, g=None, beta=None, a=None, b=None, A_log=None, dt_bias=None,
            l2norm=True, q_scale=None, eps=None, chunk=64, path=PREFILL_AUTO, workspace=None, status=None,
            wait_polls=0, stream=None):
    """Chunked prefill.  q, k ``[B,T,Hk,dk]``; v ``[B,T,Hv,dv]``; state ``[B,Hv,dk,dv]``
    fp32 (updated in place); gate ``g [B,T,Hv,dk]`` + ``beta [B,T,Hv]`` or
    ``a, b [B,T,Hv]`` + ``A_log, dt_bias [Hv]``.  ``path`` forces a kernel for this call.
    Returns o ``[B,T,Hv,dv]``: the given ``o`` (fp32 or bf16) or a new fp32 tensor.

    The library itself allocates nothing.  This binding is a convenience: when ``o`` is not
    given, or ``workspace`` is missing or smaller than :func:`prefill_workspace_size`, it
    allocates them through torch's caching allocator (a ``cudaMalloc`` the first time a size
    is seen).  Pass both to keep the call free of allocations."""
    import torch
    if o is None:
        o = torch.empty(v.shape, dtype=torch.float32, device=v.device)
    _check_types(q, k, v, state, o, g, beta, a, b, A_log, dt_bias)
    _check_status(status)
    A = make_args(q, k, v, state, o, T=q.shape[1], g=g, beta=beta, a=a, b=b, A_log=A_log, dt_bias=dt_bias,
                  l2norm=l2norm, q_scale=q_scale, eps=eps, chunk=chunk, path=path, wait_polls=wait_polls,
                  status=status)
    L = lib()
    need = int(L.cgdr_prefill_workspace_size(ctypes.byref(A)))
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if (workspace is not None and need > 0) else 0
    ws_bytes = workspace.numel() * workspace.element_size() if (workspace is not None and need > 0) else 0
    _check(L.cgdr_prefill(ctypes.byref(A), ctypes.c_void_p(ws_ptr), ctypes.c_size_t(ws_bytes),
                          _stream_handle(stream)), "cgdr_prefill")
    return o


def prefill_noalloc(q, k, v, state, o=None, *, g=None, beta=None, a=None, b=None, A_log=None, dt_bias=None,
                    l2norm=True, q_scale=None, eps=None, chunk=64, path=PREFILL_AUTO, status=None, stream=None):
    """`prefill` with the library's static scratch instead of a workspace (allocates nothing
    on the device when ``o`` is given).  Calls that overlap on the GPU race on that scratch."""
    import torch
    if o is None:
        o = torch.empty(v.shape, dtype=torch.float32, device=v.device)
    _check_types(q, k, v, state, o, g, beta, a, b, A_log, dt_bias)
    _check_status(status)
    A = make_args(q, k, v, state, o, T=q.shape[1], g=g, beta=beta, a=a, b=b, A_log=A_log, dt_bias=dt_bias,
                  l2norm=l2norm, q_scale=q_scale, eps=eps, chunk=chunk, path=path, status=status)
    _check(lib().cgdr_prefill_noalloc(ctypes.byref(A), _stream_handle(stream)), "cgdr_prefill_noalloc")
    return o


def prefill_path_for(q, k, v, state, o, **kw) -> int:
    """The kernel (PREFILL_PER_HEAD, PREFILL_CLUSTER, PREFILL_SIMT or PREFILL_RECURRENT) a prefill with these
    arguments (``path=`` included) runs; PREFILL_AUTO if the arguments are invalid or there is no work."""
    A = make_args(q, k, v, state, o, T=q.shape[1], **kw)
    return int(lib().cgdr_prefill_path_for(ctypes.byref(A)))


def workspace_status(workspace, stream=None) -> int:
    """Device-side status word a prefill left in its workspace (synchronises the stream)."""
    return int(lib().cgdr_workspace_status(ctypes.c_void_p(workspace.data_ptr()), _stream_handle(stream)))


def validate(A: CgdrArgs, for_prefill: bool) -> int:
    return int(lib().cgdr_validate(ctypes.byref(A), 1 if for_prefill else 0))


__all__ = ["decode", "prefill", "prefill_noalloc", "prefill_workspace_size", "workspace_status", "validate",
           "status_string", "make_args", "prefill_path_for",
           "CgdrArgs", "CgdrError", "lib", "LIB_PATH"]
