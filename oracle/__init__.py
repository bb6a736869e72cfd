"""fp64 CPU oracle for the channelwise gated delta rule.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package.  The product path
(the CUDA library and its Python binding) never imports, links or calls it,
and the two share no code.

Two routines:

* :func:`recurrence` -- the plain token-by-token definition in fp64 C
  (``cgdr_oracle.c``), four traversals of the state per token (decay,
  prediction, rank-one correction, readout), following the summary of
  "Two-pass optimization for channelwise gated delta rule kernel"
  (executorch PR #21020) and the gating of "Add fused GatedDeltaNet decode
  Triton kernel" (executorch PR #18865).
* :func:`chunkwise` (in :mod:`oracle.chunkwise`) -- a naive fp64 numpy
  restatement of the chunked WY/UT form described in "Add parallel chunked
  prefill for channelwise gated delta rule" (executorch PR #21061), Summary.
  It exists to check that derivation against the recurrence on tiny inputs.

Both are pinned by ``tests/test_oracle_pins.py`` against closed forms,
invariants and brute force (see that file).  One convention is not fixed by
the pages and is therefore **parity unpinned**: which k-head a v-head reads
when Hv > Hk (this oracle uses repeat-interleave, v-head h -> k-head
h // (Hv/Hk)); any consistent choice passes parity.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cgdr_oracle.c")
_LIB = os.path.join(_HERE, "libcgdr_oracle.so")
_lock = threading.Lock()
_lib = None

DEFAULT_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Args(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("Hk", ctypes.c_int), ("Hv", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("gate_mode", ctypes.c_int), ("l2norm", ctypes.c_int),
        ("q_scale", ctypes.c_double), ("eps", ctypes.c_double),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("a", ctypes.c_void_p), ("b", ctypes.c_void_p),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("S0", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("S", ctypes.c_void_p),
        ("n_threads", ctypes.c_int),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.cgdr_oracle_recurrence.argtypes = [ctypes.POINTER(_Args)]
            lib.cgdr_oracle_recurrence.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    """Exact upcast to a contiguous fp64 numpy array (bf16 and fp32 embed exactly)."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def recurrence(q, k, v, *, g=None, beta=None, a=None, b=None, A_log=None, dt_bias=None,
               S0=None, l2norm=True, q_scale=None, eps=DEFAULT_EPS, threads=None):
    """Token-by-token fp64 recurrence.

    Shapes: q, k ``[B,T,Hk,dk]``; v ``[B,T,Hv,dv]``; channel gate ``g [B,T,Hv,dk]``
    and ``beta [B,T,Hv]``; or the GatedDeltaNet gate ``a, b [B,T,Hv]`` with
    ``A_log, dt_bias [Hv]``.  ``S0 [B,Hv,dk,dv]`` or None for zero.
    Returns ``(o [B,T,Hv,dv], S [B,Hv,dk,dv])`` as fp64 numpy arrays.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, T, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    assert k.shape == q.shape and v.shape[:2] == (B, T) and Hv % Hk == 0
    gate_mode = 0 if g is not None else 1
    keep = []
    args = _Args()
    args.B, args.T, args.Hk, args.Hv, args.dk, args.dv = B, T, Hk, Hv, dk, dv
    args.gate_mode = gate_mode
    args.l2norm = 1 if l2norm else 0
    args.q_scale = float(q_scale) if q_scale is not None else 0.0
    args.eps = float(eps)

    def ptr(x, shape=None):
        if x is None:
            return None
        x = _f64(x)
        if shape is not None:
            assert x.shape == tuple(shape), (x.shape, shape)
        keep.append(x)
        return x.ctypes.data

    args.q, args.k, args.v = ptr(q), ptr(k), ptr(v)
    if gate_mode == 0:
        assert beta is not None
        args.g = ptr(g, (B, T, Hv, dk))
        args.beta = ptr(beta, (B, T, Hv))
    else:
        assert a is not None and b is not None and A_log is not None and dt_bias is not None
        args.a, args.b = ptr(a, (B, T, Hv)), ptr(b, (B, T, Hv))
        args.A_log, args.dt_bias = ptr(A_log, (Hv,)), ptr(dt_bias, (Hv,))
    args.S0 = ptr(S0, (B, Hv, dk, dv)) if S0 is not None else None
    o = np.zeros((B, T, Hv, dv), dtype=np.float64)
    S = np.zeros((B, Hv, dk, dv), dtype=np.float64)
    args.o, args.S = o.ctypes.data, S.ctypes.data
    args.n_threads = int(threads) if threads else default_threads()
    rc = _load().cgdr_oracle_recurrence(ctypes.byref(args))
    if rc != 0:
        raise RuntimeError("cgdr_oracle_recurrence failed with code %d" % rc)
    return o, S


from .chunkwise import chunkwise  # noqa: E402  (numpy only)

__all__ = ["recurrence", "chunkwise", "build", "default_threads", "DEFAULT_EPS"]
