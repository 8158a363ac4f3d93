"""GB300 (sm_103a) kernelized linear attention: thin Python binding.

The compute lives in ``liblinattn.so`` (CUDA kernels behind the C ABI of
``include/linattn.h``).  This module only marshals arguments: it checks
tensor shapes and dtypes, allocates outputs and the workspace through
PyTorch (device memory and streams are PyTorch's job here) and calls the C
entry points of the same names on the current CUDA stream.  There is no CPU
or PyTorch fallback: if the library is missing every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblinattn.so")

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_WORKSPACE, LA_ERR_CUDA, LA_ERR_TIMEOUT = range(6)
LA_F32, LA_BF16 = 0, 1
LA_NOALLOC_SCRATCH_BYTES = 16 << 20  # built-in scratch of la_forward_causal_noalloc
FEATURE_MAPS = {"none": 0, "elu_plus_one": 1, "relu": 2}
UPDATE_RULES = {"linear": 0, "gated": 1, "delta": 2, "gated_delta": 3}
_DTYPES = {torch.float32: LA_F32, torch.bfloat16: LA_BF16}


class LinearAttentionError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[status {status}] {message}")
        self.status = status


class la_params(ctypes.Structure):
    """Mirror of ``struct la_params`` (include/linattn.h)."""
    _fields_ = [
        ("batch", ctypes.c_int64), ("seq_len", ctypes.c_int64),
        ("q_heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
        ("key_dim", ctypes.c_int32), ("value_dim", ctypes.c_int32),
        ("io_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
        ("feature_map", ctypes.c_int32), ("use_normalizer", ctypes.c_int32),
        ("epsilon", ctypes.c_float), ("scale", ctypes.c_float),
        ("update_rule", ctypes.c_int32), ("decay_per_key_dim", ctypes.c_int32),
    ]


_vp = ctypes.c_void_p
_SIGNATURES = {
    "la_get_initial_state": (ctypes.c_int, [ctypes.POINTER(la_params), _vp, _vp, _vp]),
    "la_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(la_params), ctypes.c_int]),
    "la_forward_causal": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 10 + [ctypes.c_size_t, _vp]),
    "la_forward_causal_noalloc": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 10),
    "la_forward_noncausal": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 5 + [ctypes.c_size_t, _vp]),
    "la_decode_step": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 8),
    "la_forward_causal_masked": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 11 + [ctypes.c_size_t, _vp]),
    "la_forward_noncausal_masked": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 6 + [ctypes.c_size_t, _vp]),
    "la_decode_step_masked": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 9),
    "la_forward_causal_delta": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 5 + [ctypes.c_int]
                                + [_vp] * 4 + [_vp]),
    "la_decode_step_delta": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 5 + [ctypes.c_int] + [_vp] * 4),
    "la_delta_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(la_params)]),
    "la_forward_causal_delta_ws": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 5 + [ctypes.c_int]
                                   + [_vp] * 4 + [_vp, ctypes.c_size_t, _vp]),
    "la_backward_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(la_params)]),
    "la_backward_causal": (ctypes.c_int, [ctypes.POINTER(la_params)] + [_vp] * 12 + [ctypes.c_size_t, _vp]),
    "la_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "la_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "la_device_status": (ctypes.c_int, [ctypes.c_int]),
    "la_last_error": (ctypes.c_char_p, []),
    "la_abi_version": (ctypes.c_int, []),
    "la_launch_count": (ctypes.c_uint64, []),
    "la_device_error": (ctypes.c_uint, [ctypes.c_int]),
    "la_check_bounded_wait": (ctypes.c_int, [ctypes.c_uint32, _vp]),
}

_lib = None


def lib():
    """The loaded C library (ctypes); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _check(status: int):
    if status != LA_OK:
        raise LinearAttentionError(status, lib().la_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_params(*, batch, seq_len, q_heads, kv_heads, key_dim, value_dim, io_dtype=torch.bfloat16,
                out_dtype=None, feature_map="elu_plus_one", use_normalizer=True, epsilon=1e-6,
                scale=1.0, update_rule="linear", decay_per_key_dim=False) -> la_params:
    out_dtype = io_dtype if out_dtype is None else out_dtype
    return la_params(batch, seq_len, q_heads, kv_heads, key_dim, value_dim, _DTYPES[io_dtype],
                     _DTYPES[out_dtype], FEATURE_MAPS[feature_map], int(bool(use_normalizer)),
                     float(epsilon), float(scale), UPDATE_RULES[update_rule], int(bool(decay_per_key_dim)))


def _as_bthd(x, heads, name):
    if x.dim() == 3:  # ONNX packed (B, T, H*D)
        if x.shape[2] % heads:
            raise ValueError(f"{name}: last dim {x.shape[2]} not divisible by {heads} heads")
        x = x.view(x.shape[0], x.shape[1], heads, x.shape[2] // heads)
    if x.dim() != 4 or x.shape[2] != heads:
        raise ValueError(f"{name}: expected (B,T,{heads},D) or (B,T,{heads}*D), got {tuple(x.shape)}")
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError(f"{name}: must be a contiguous CUDA tensor")
    return x


def _prep(q, k, v, q_heads, kv_heads, decay=None, **kw):
    q = _as_bthd(q, q_heads, "q")
    k = _as_bthd(k, kv_heads, "k")
    v = _as_bthd(v, kv_heads, "v")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPES:
        raise ValueError("q, k, v must share one dtype, float32 or bfloat16")
    B, T, _, Dk = q.shape
    if k.shape[:2] != (B, T) or v.shape[:2] != (B, T) or k.shape[3] != Dk:
        raise ValueError("q, k, v shapes disagree")
    per_dim = False
    if decay is not None:
        # ONNX decay layouts: (B, T, H_kv) per head, (B, T, H_kv*d_k) per key dimension
        if decay.numel() == B * T * kv_heads * Dk and Dk > 1:
            per_dim = True
        elif decay.numel() != B * T * kv_heads:
            raise ValueError(f"decay must have B*T*Hkv or B*T*Hkv*Dk elements, got {tuple(decay.shape)}")
    p = make_params(batch=B, seq_len=T, q_heads=q_heads, kv_heads=kv_heads, key_dim=Dk,
                    value_dim=v.shape[3], io_dtype=q.dtype, decay_per_key_dim=per_dim, **kw)
    return q, k, v, p


def _mask(mask, B, T):
    """Sequence-validity mask (B, T) as a contiguous one-byte CUDA tensor
    (bool or uint8, nonzero = valid), or None."""
    if mask is None:
        return None
    if mask.dtype not in (torch.bool, torch.uint8) or not mask.is_cuda:
        raise ValueError("mask must be a CUDA tensor of dtype bool or uint8")
    if mask.numel() != B * T:
        raise ValueError(f"mask must have B*T = {B * T} elements ({B}, {T}), got {tuple(mask.shape)}")
    return mask.contiguous()


DELTA_RULES = ("delta", "gated_delta")


def _beta(beta, B, T, kv_heads):
    """ONNX beta layouts: (B, T, H_kv) -> 1 (per head), (B, T, 1) -> 0."""
    if beta is None:
        raise ValueError("the delta rules need beta")
    if not beta.is_cuda or not beta.is_contiguous():
        raise ValueError("beta must be a contiguous CUDA tensor")
    if beta.numel() == B * T * kv_heads:
        return 1
    if beta.numel() == B * T:
        return 0
    raise ValueError(f"beta must have B*T*Hkv or B*T elements, got {tuple(beta.shape)}")


def la_workspace_bytes(params: la_params, causal: bool) -> int:
    return int(lib().la_workspace_bytes(ctypes.byref(params), int(bool(causal))))


def _workspace(params, causal, device, workspace):
    need = la_workspace_bytes(params, causal)
    if need == 0:
        return None, 0
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def la_get_initial_state(batch, kv_heads, key_dim, value_dim, use_normalizer=True, device="cuda",
                         stream=None):
    """Zero (S, Z) state (Keras get_initial_state); Z is None without the normalizer."""
    p = make_params(batch=batch, seq_len=0, q_heads=kv_heads, kv_heads=kv_heads, key_dim=key_dim,
                    value_dim=value_dim, use_normalizer=use_normalizer)
    S = torch.empty(batch, kv_heads, key_dim, value_dim, dtype=torch.float32, device=device)
    Z = torch.empty(batch, kv_heads, key_dim, dtype=torch.float32, device=device) if use_normalizer else None
    _check(lib().la_get_initial_state(ctypes.byref(p), _ptr(S), _ptr(Z), _stream(stream)))
    return S, Z


def la_forward_causal(q, k, v, *, q_heads, kv_heads, feature_map="elu_plus_one", use_normalizer=True,
                      epsilon=1e-6, scale=1.0, update_rule="linear", decay=None, initial_state=None,
                      return_state=False, out_dtype=None, out=None, state_out=None, workspace=None,
                      mask=None, beta=None, stream=None):
    """Causal pass.  q (B,T,Hq,Dk) / (B,T,Hq*Dk), k and v likewise with Hkv heads.

    initial_state: (S0, Z0) or None (zeros).  Returns y, or (y, (S, Z)) with
    return_state.  ``state_out`` may be the initial_state tensors themselves
    (in-place streaming).  ``mask`` (B,T) bool/uint8: invalid steps keep the
    state and output zero (la_forward_causal_masked).  update_rule "delta" /
    "gated_delta" take ``beta`` (B,T,Hkv) or (B,T,1) (la_forward_causal_delta);
    they keep no Z."""
    q, k, v, p = _prep(q, k, v, q_heads, kv_heads, out_dtype=out_dtype, feature_map=feature_map,
                       use_normalizer=use_normalizer, epsilon=epsilon, scale=scale,
                       update_rule=update_rule, decay=decay)
    B, T, _, Dk = q.shape
    Dv = v.shape[3]
    ydt = q.dtype if out_dtype is None else out_dtype
    y = out if out is not None else torch.empty(B, T, q_heads, Dv, dtype=ydt, device=q.device)
    S0, Z0 = initial_state if initial_state is not None else (None, None)
    S, Z = None, None
    if return_state:
        if state_out is not None:
            S, Z = state_out
        else:
            S = torch.empty(B, kv_heads, Dk, Dv, dtype=torch.float32, device=q.device)
            Z = torch.empty(B, kv_heads, Dk, dtype=torch.float32, device=q.device) if use_normalizer else None
    if decay is not None and (not decay.is_cuda or not decay.is_contiguous() or decay.dtype != q.dtype):
        raise ValueError("decay must be a contiguous CUDA tensor of the io dtype")
    if update_rule in DELTA_RULES:
        bph = _beta(beta, B, T, kv_heads)
        m = _mask(mask, B, T) if mask is not None else None
        need = int(lib().la_delta_workspace_bytes(ctypes.byref(p)))
        if need > 0:  # the chunk-parallel tensor-core form
            if workspace is None or workspace.numel() * workspace.element_size() < need:
                workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            _check(lib().la_forward_causal_delta_ws(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(beta),
                                                    bph, _ptr(m), _ptr(S0), _ptr(y), _ptr(S), _ptr(workspace),
                                                    workspace.numel() * workspace.element_size(), _stream(stream)))
        else:
            _check(lib().la_forward_causal_delta(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(beta),
                                                 bph, _ptr(m), _ptr(S0), _ptr(y), _ptr(S), _stream(stream)))
        return (y, (S, None)) if return_state else y
    ws, ws_bytes = _workspace(p, True, q.device, workspace)
    if mask is not None:
        m = _mask(mask, B, T)
        _check(lib().la_forward_causal_masked(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(m),
                                              _ptr(S0), _ptr(Z0), _ptr(y), _ptr(S), _ptr(Z), _ptr(ws), ws_bytes,
                                              _stream(stream)))
    else:
        _check(lib().la_forward_causal(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(S0),
                                       _ptr(Z0), _ptr(y), _ptr(S), _ptr(Z), _ptr(ws), ws_bytes,
                                       _stream(stream)))
    return (y, (S, Z)) if return_state else y


def la_forward_causal_noalloc(q, k, v, *, q_heads, kv_heads, feature_map="elu_plus_one",
                              use_normalizer=True, epsilon=1e-6, scale=1.0, update_rule="linear", decay=None,
                              initial_state=None, out, state_out=None, stream=None):
    """la_forward_causal on the library's built-in scratch: the caller passes
    every output buffer (``out`` and, to get the final state, ``state_out``),
    so neither this wrapper nor the library allocates device memory.  Calls
    that may overlap on one device race on the shared scratch."""
    q, k, v, p = _prep(q, k, v, q_heads, kv_heads, out_dtype=out.dtype, feature_map=feature_map,
                       use_normalizer=use_normalizer, epsilon=epsilon, scale=scale,
                       update_rule=update_rule, decay=decay)
    if decay is not None and (not decay.is_cuda or not decay.is_contiguous() or decay.dtype != q.dtype):
        raise ValueError("decay must be a contiguous CUDA tensor of the io dtype")
    S0, Z0 = initial_state if initial_state is not None else (None, None)
    S, Z = state_out if state_out is not None else (None, None)
    _check(lib().la_forward_causal_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(S0),
                                           _ptr(Z0), _ptr(out), _ptr(S), _ptr(Z), _stream(stream)))
    return out


def la_forward_noncausal(q, k, v, *, q_heads, kv_heads, feature_map="elu_plus_one", use_normalizer=True,
                         epsilon=1e-6, scale=1.0, out_dtype=None, out=None, workspace=None, mask=None,
                         stream=None):
    """Non-causal pass with the global state; returns y (B,T,Hq,Dv).  ``mask``
    (B,T): invalid keys/values leave the sums, invalid queries output zero."""
    q, k, v, p = _prep(q, k, v, q_heads, kv_heads, out_dtype=out_dtype, feature_map=feature_map,
                       use_normalizer=use_normalizer, epsilon=epsilon, scale=scale)
    B, T, _, _ = q.shape
    ydt = q.dtype if out_dtype is None else out_dtype
    y = out if out is not None else torch.empty(B, T, q_heads, v.shape[3], dtype=ydt, device=q.device)
    ws, ws_bytes = _workspace(p, False, q.device, workspace)
    if mask is not None:
        m = _mask(mask, B, T)
        _check(lib().la_forward_noncausal_masked(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(m), _ptr(y),
                                                 _ptr(ws), ws_bytes, _stream(stream)))
    else:
        _check(lib().la_forward_noncausal(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(ws),
                                          ws_bytes, _stream(stream)))
    return y


def la_decode_step(q, k, v, S, Z=None, *, q_heads, kv_heads, feature_map="elu_plus_one",
                   use_normalizer=True, epsilon=1e-6, scale=1.0, update_rule="linear", decay=None,
                   out_dtype=None, out=None, mask=None, beta=None, stream=None):
    """One token per sequence; S (and Z) are updated in place.  Returns y (B,1,Hq,Dv).
    ``mask`` (B,) or (B,1): a sequence whose step is invalid keeps S, Z and outputs zero."""
    q, k, v, p = _prep(q, k, v, q_heads, kv_heads, out_dtype=out_dtype, feature_map=feature_map,
                       use_normalizer=use_normalizer, epsilon=epsilon, scale=scale,
                       update_rule=update_rule, decay=decay)
    ydt = q.dtype if out_dtype is None else out_dtype
    y = out if out is not None else torch.empty(q.shape[0], 1, q_heads, v.shape[3], dtype=ydt,
                                                device=q.device)
    if update_rule in DELTA_RULES:
        bph = _beta(beta, q.shape[0], 1, kv_heads)
        m = _mask(mask, q.shape[0], 1) if mask is not None else None
        _check(lib().la_decode_step_delta(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(beta), bph,
                                          _ptr(m), _ptr(S), _ptr(y), _stream(stream)))
        return y
    if mask is not None:
        m = _mask(mask, q.shape[0], 1)
        _check(lib().la_decode_step_masked(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(m),
                                           _ptr(S), _ptr(Z), _ptr(y), _stream(stream)))
    else:
        _check(lib().la_decode_step(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(S),
                                    _ptr(Z), _ptr(y), _stream(stream)))
    return y


def la_backward_workspace_bytes(params: la_params) -> int:
    return int(lib().la_backward_workspace_bytes(ctypes.byref(params)))


def la_backward_causal(q, k, v, dy, *, q_heads, kv_heads, feature_map="elu_plus_one", use_normalizer=True,
                       epsilon=1e-6, scale=1.0, initial_state=None, grad_dtype=torch.float32,
                       return_state_grad=False, workspace=None, stream=None):
    """Gradients of la_forward_causal (linear rule) given dy (the shape of y,
    io dtype): returns (dq, dk, dv) in ``grad_dtype``, and (dS0, dZ0) as well
    with ``return_state_grad``."""
    q, k, v, p = _prep(q, k, v, q_heads, kv_heads, out_dtype=grad_dtype, feature_map=feature_map,
                       use_normalizer=use_normalizer, epsilon=epsilon, scale=scale)
    dy = _as_bthd(dy, q_heads, "dy")
    if dy.dtype != q.dtype or dy.shape[:2] != q.shape[:2] or dy.shape[3] != v.shape[3]:
        raise ValueError("dy must have the shape of y and the dtype of q")
    B, T, _, Dk = q.shape
    Dv = v.shape[3]
    dq = torch.empty(q.shape, dtype=grad_dtype, device=q.device)
    dk = torch.empty(k.shape, dtype=grad_dtype, device=q.device)
    dv = torch.empty(v.shape, dtype=grad_dtype, device=q.device)
    S0, Z0 = initial_state if initial_state is not None else (None, None)
    dS0 = dZ0 = None
    if return_state_grad:
        dS0 = torch.empty(B, kv_heads, Dk, Dv, dtype=torch.float32, device=q.device)
        dZ0 = torch.empty(B, kv_heads, Dk, dtype=torch.float32, device=q.device) if use_normalizer else None
    need = la_backward_workspace_bytes(p)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(1, need), dtype=torch.uint8, device=q.device)
    _check(lib().la_backward_causal(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(S0), _ptr(Z0), _ptr(dy), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(dS0), _ptr(dZ0), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)))
    return (dq, dk, dv, dS0, dZ0) if return_state_grad else (dq, dk, dv)


def la_launch_count() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(lib().la_launch_count())


def la_device_error(reset: bool = True) -> int:
    """Error word of the bounded pipeline waits on the current device (0 = none)."""
    return int(lib().la_device_error(int(bool(reset))))


LA_SELFTEST_WARP_WAIT = 1 << 30
LA_SELFTEST_THREAD_WAIT = 1 << 31


def la_check_bounded_wait(limit_us: int = 1000, stream=None) -> None:
    """Enqueue the bounded-wait self-test: both wait forms give up after
    ``limit_us`` on a barrier nothing completes and set their bits in the
    device error word (read it with ``la_device_error``)."""
    _check(lib().la_check_bounded_wait(int(limit_us), _stream(stream)))


def la_device_status(reset: bool = True) -> int:
    """Synchronise the device and return LA_OK, or LA_ERR_TIMEOUT when a
    kernel gave up on a bounded wait (LA_ERR_CUDA on a device error)."""
    return int(lib().la_device_status(int(bool(reset))))


def la_delta_workspace_bytes(params: la_params) -> int:
    """Workspace of la_forward_causal_delta_ws (0: the shape runs the recurrence)."""
    return int(lib().la_delta_workspace_bytes(ctypes.byref(params)))
