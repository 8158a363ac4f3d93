"""Gradients of causal kernelized linear attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite imports this module.  It writes the causal recurrence of
"[Feature] LinearAttention layer for Keras" (Mathematical definition /
Causal: S_t = S_{t-1} + phi(K_t)^T V_t, Z_t = Z_{t-1} + phi(K_t),
Y_t = phi(Q_t) S_t / (phi(Q_t) Z_t + eps), the current token included) token by
token in plain float64 PyTorch CPU ops, and takes its gradients with
autograd.  The same request asks for "Float64 numerical-gradient checks where
supported" (Test Plan, Stability); the pins in tests/oracle_pins.py hold this
module to the C oracle's forward values and to finite differences.

Grouped heads follow the ONNX-light "LinearAttention" operator: query head h
reads kv head h // (Hq / Hkv).
"""
from __future__ import annotations

import torch


def phi(x, feature_map: str, eps: float):
    """Feature maps of the Keras request, section "Feature maps"."""
    if feature_map == "elu_plus_one":
        return torch.where(x > 0, x + 1.0, torch.exp(torch.clamp(x, max=0.0)))
    if feature_map == "relu":
        return torch.clamp(x, min=0.0) + eps
    if feature_map == "none":
        return x
    raise ValueError(feature_map)


def causal_forward(q, k, v, *, q_heads, kv_heads, feature_map="elu_plus_one", use_normalizer=True, eps=1e-6,
                   scale=1.0, S0=None, Z0=None):
    """y (B,T,Hq,Dv) from q (B,T,Hq,Dk), k (B,T,Hkv,Dk), v (B,T,Hkv,Dv), all float64
    CPU tensors; S0 (B,Hkv,Dk,Dv) and Z0 (B,Hkv,Dk) optional.  Differentiable."""
    B, T = q.shape[:2]
    Dk, Dv = q.shape[-1], v.shape[-1]
    G = q_heads // kv_heads
    S = S0.clone() if S0 is not None else torch.zeros(B, kv_heads, Dk, Dv, dtype=q.dtype)
    Z = Z0.clone() if Z0 is not None else torch.zeros(B, kv_heads, Dk, dtype=q.dtype)
    fq, fk = phi(q, feature_map, eps), phi(k, feature_map, eps)
    ys = []
    for t in range(T):
        S = S + fk[:, t, :, :, None] * v[:, t, :, None, :]          # (B,Hkv,Dk,Dv)
        Z = Z + fk[:, t]                                             # (B,Hkv,Dk)
        Sg = S.repeat_interleave(G, dim=1)                           # query head h -> kv head h // G
        Zg = Z.repeat_interleave(G, dim=1)
        num = torch.einsum("bhi,bhij->bhj", fq[:, t], Sg)            # (B,Hq,Dv)
        if use_normalizer:
            den = torch.einsum("bhi,bhi->bh", fq[:, t], Zg) + eps
            num = num / den[..., None]
        ys.append(scale * num)
    return torch.stack(ys, dim=1)


def causal_backward(q, k, v, dy, *, q_heads, kv_heads, feature_map="elu_plus_one", use_normalizer=True, eps=1e-6,
                    scale=1.0, S0=None, Z0=None):
    """(dq, dk, dv, dS0, dZ0) of sum(y * dy) in float64 (dS0/dZ0 None without S0/Z0)."""
    to = lambda x: None if x is None else (x.detach().to("cpu", torch.float64).clone().requires_grad_(True))
    q, k, v, S0, Z0 = map(to, (q, k, v, S0, Z0))
    dy = dy.detach().to("cpu", torch.float64)
    y = causal_forward(q, k, v, q_heads=q_heads, kv_heads=kv_heads, feature_map=feature_map,
                       use_normalizer=use_normalizer, eps=eps, scale=scale, S0=S0, Z0=Z0)
    ins = [x for x in (q, k, v, S0, Z0) if x is not None]
    grads = torch.autograd.grad(y, ins, grad_outputs=dy, allow_unused=True)
    out = list(grads[:3])
    rest = list(grads[3:])
    out.append(rest.pop(0) if S0 is not None else None)
    out.append(rest.pop(0) if Z0 is not None else None)
    return tuple(out)
