"""CPU oracle for kernelized linear attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports it and shares no code with it.

Two independent formulations live here:

* ``causal`` / ``noncausal``: the fp64 C recurrence in
  ``linattn_oracle.c`` (token by token, exactly as the pages write it), run
  through ctypes.
* ``oracle.bruteforce``: the O(T^2) pairwise-weight form in numpy, written
  from the kernel-trick view (weights phi(q_i).phi(k_j), j <= i).

Page citations (title, section):
  "[Feature] LinearAttention layer for Keras" -- Mathematical definition,
  Feature maps, Streaming State;
  "Causal Linear Attention" -- running sums and the read-out;
  ONNX-light "LinearAttention" -- layouts, GQA, update rules, scale.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "linattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblinattn_oracle.so")

FMAP = {"none": 0, "elu_plus_one": 1, "relu": 2}
RULE = {"linear": 0, "gated": 1, "delta": 2, "gated_delta": 3}


class _Params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("T", ctypes.c_int64),
        ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("Dk", ctypes.c_int32), ("Dv", ctypes.c_int32),
        ("feature_map", ctypes.c_int32), ("use_normalizer", ctypes.c_int32),
        ("eps", ctypes.c_double), ("scale", ctypes.c_double),
        ("rule", ctypes.c_int32), ("decay_per_dim", ctypes.c_int32),
        ("beta_per_head", ctypes.c_int32), ("nthreads", ctypes.c_int32),
    ]


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the C oracle with gcc (portable C11, no SIMD intrinsics)."""
    cmd = ["gcc", "-std=c11", "-O2", "-shared", "-fPIC", "-pthread", *extra_flags,
           "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


_lib_cache: dict = {}
_lock = threading.Lock()


def load(path: str = _LIB_PATH):
    """Load (building first if missing or stale) the oracle shared library."""
    with _lock:
        if path in _lib_cache:
            return _lib_cache[path]
        if path == _LIB_PATH and (not os.path.exists(path)
                                  or os.path.getmtime(path) < os.path.getmtime(_SRC)):
            build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.orc_causal.argtypes = [ctypes.POINTER(_Params)] + [dp] * 10
        lib.orc_causal.restype = ctypes.c_int
        lib.orc_noncausal.argtypes = [ctypes.POINTER(_Params)] + [dp] * 4
        lib.orc_noncausal.restype = ctypes.c_int
        bp = ctypes.c_void_p
        lib.orc_causal_masked.argtypes = [ctypes.POINTER(_Params)] + [dp] * 5 + [bp] + [dp] * 5
        lib.orc_causal_masked.restype = ctypes.c_int
        lib.orc_noncausal_masked.argtypes = [ctypes.POINTER(_Params)] + [dp] * 3 + [bp, dp]
        lib.orc_noncausal_masked.restype = ctypes.c_int
        _lib_cache[path] = lib
        return lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # a torch tensor: widen exactly on the CPU
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _mask(mask, B, T):
    """(B, T) validity mask as a contiguous uint8 array (nonzero = valid), or None."""
    if mask is None:
        return None
    if hasattr(mask, "detach"):
        mask = mask.detach().cpu().numpy()
    m = np.ascontiguousarray(np.asarray(mask).reshape(B, T) != 0, dtype=np.uint8)
    return m


def _mptr(m):
    return None if m is None else ctypes.c_void_p(m.ctypes.data)


def resolve_scale(scale: float, dk: int) -> float:
    """ONNX 'scale' attribute: 0.0 means 1/sqrt(d_k)."""
    return 1.0 / np.sqrt(dk) if scale == 0.0 else float(scale)


def _params(q, k, v, q_heads, kv_heads, feature_map, use_normalizer, eps, scale,
            rule, decay, beta, nthreads):
    B, T = q.shape[0], q.shape[1]
    Dk = q.shape[-1] // q_heads if q.ndim == 3 else q.shape[-1]
    Dv = v.shape[-1] // kv_heads if v.ndim == 3 else v.shape[-1]
    decay_per_dim = 0
    if decay is not None:
        last = decay.shape[-1] if decay.ndim == 3 else decay.shape[-1] * decay.shape[-2]
        if decay.ndim == 4 or (last == kv_heads * Dk and last != kv_heads):
            decay_per_dim = 1
    beta_per_head = 1
    if beta is not None and beta.shape[-1] == 1 and kv_heads != 1:
        beta_per_head = 0
    p = _Params(B, T, q_heads, kv_heads, Dk, Dv, FMAP[feature_map], int(bool(use_normalizer)),
                float(eps), resolve_scale(scale, Dk), RULE[rule], decay_per_dim, beta_per_head,
                int(nthreads or os.cpu_count() or 1))
    return p, B, T, Dk, Dv


def causal(q, k, v, *, q_heads, kv_heads, feature_map="elu_plus_one", use_normalizer=True,
           eps=1e-6, scale=1.0, rule="linear", decay=None, beta=None, S0=None, Z0=None,
           mask=None, nthreads=None, lib=None):
    """Causal pass.  q (B,T,Hq*Dk) or (B,T,Hq,Dk); k (B,T,Hkv[*]Dk); v (B,T,Hkv[*]Dv).

    Returns (y (B,T,Hq,Dv), S (B,Hkv,Dk,Dv), Z (B,Hkv,Dk)) in float64.
    ``scale`` follows the ONNX attribute: 0.0 means 1/sqrt(d_k).  ``mask``
    (B,T) is the Keras sequence-validity mask: an invalid step keeps the
    state and outputs zero."""
    q, k, v, decay, beta, S0, Z0 = map(_f64, (q, k, v, decay, beta, S0, Z0))
    p, B, T, Dk, Dv = _params(q, k, v, q_heads, kv_heads, feature_map, use_normalizer, eps,
                              scale, rule, decay, beta, nthreads)
    y = np.zeros((B, T, q_heads, Dv))
    S = np.zeros((B, kv_heads, Dk, Dv))
    Z = np.zeros((B, kv_heads, Dk))
    m = _mask(mask, B, T)
    rc = (lib or load()).orc_causal_masked(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(decay),
                                           _ptr(beta), _mptr(m), _ptr(S0), _ptr(Z0), _ptr(y), _ptr(S),
                                           _ptr(Z))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return y, S, Z


def noncausal(q, k, v, *, q_heads, kv_heads, feature_map="elu_plus_one", use_normalizer=True,
              eps=1e-6, scale=1.0, mask=None, nthreads=None, lib=None):
    """Non-causal pass with the global state.  Returns y (B,T,Hq,Dv) in float64.
    ``mask`` (B,T): invalid keys/values leave the sums, invalid queries give 0."""
    q, k, v = map(_f64, (q, k, v))
    p, B, T, Dk, Dv = _params(q, k, v, q_heads, kv_heads, feature_map, use_normalizer, eps,
                              scale, "linear", None, None, nthreads)
    y = np.zeros((B, T, q_heads, Dv))
    m = _mask(mask, B, T)
    rc = (lib or load()).orc_noncausal_masked(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _mptr(m),
                                              _ptr(y))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return y
