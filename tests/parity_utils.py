"""Helpers for the GPU parity tests: tolerances and sampled-slice oracle runs."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances (norm-wise relative error ||gpu - ref|| / ||ref||):
#  - float32 inputs: 1e-5;
#  - bf16 inputs with a float32 output: 2e-3 (fp32 state, bf16 tensor-core products);
#  - bf16 inputs with a bf16 output: 2e-3 plus the output rounding itself, which
#    is at most 2^-8 of every element (round-to-nearest into 8 significant bits),
#    so by the triangle inequality the bound is 2e-3 + 2^-8.
TOL_F32 = 1e-5
TOL_BF16 = 2e-3
TOL_BF16_OUT = 2e-3 + 2.0 ** -8


def tol_for(io_dtype, out_dtype):
    if io_dtype == torch.float32:
        return TOL_F32 if out_dtype == torch.float32 else TOL_F32 + 2.0 ** -8
    return TOL_BF16 if out_dtype == torch.float32 else TOL_BF16_OUT


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def to64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def assert_close(got, ref, tol, what=""):
    e = rel_err(got, ref)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite values"
    assert e <= tol, f"{what}: rel err {e:.3e} > {tol:.3e}"
    return e


def oracle_slices(q, k, v, samples, G, *, decay=None, S0=None, Z0=None, **kw):
    """Run the oracle on sampled (b, kv-head) streams only.

    samples: list of (b, hk).  Returns y (n, T, G, Dv), S (n, 1, Dk, Dv), Z (n, 1, Dk)."""
    qs = torch.stack([q[b, :, hk * G:(hk + 1) * G] for b, hk in samples]).cpu()
    ks = torch.stack([k[b, :, hk:hk + 1] for b, hk in samples]).cpu()
    vs = torch.stack([v[b, :, hk:hk + 1] for b, hk in samples]).cpu()
    ds = None if decay is None else torch.stack([decay[b, :, hk:hk + 1] for b, hk in samples]).cpu()
    S0s = None if S0 is None else torch.stack([S0[b, hk:hk + 1] for b, hk in samples]).cpu()
    Z0s = None if Z0 is None else torch.stack([Z0[b, hk:hk + 1] for b, hk in samples]).cpu()
    return oracle.causal(qs, ks, vs, q_heads=G, kv_heads=1, decay=ds, S0=S0s, Z0=Z0s, **kw)


def gpu_slices(y, samples, G):
    return torch.stack([y[b, :, hk * G:(hk + 1) * G] for b, hk in samples])
