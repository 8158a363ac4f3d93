"""Helpers for the GPU parity tests: tolerances, the comparison, and
sampled-slice oracle runs.

The comparison (``assert_close``) applies two bars with the same tolerance:

- norm-wise over the whole tensor, ||gpu - ref||_2 / ||ref||_2 <= tol;
- row by row: every row along the last axis (an output row (b, t, head) of
  Dv values, a state row (b, kv head, i) of Dv values, a key-sum row of Dk
  values, a gradient row) must satisfy
      ||gpu_r - ref_r||_2 <= tol * max(||ref_r||_2, ROW_FLOOR * rms_row)
  where rms_row is the root-mean-square row norm of the reference tensor.
  The floor only matters for rows whose reference is near zero relative to
  the tensor (cancellation); a zero reference row (a masked step) still
  needs an output within tol * ROW_FLOOR * rms_row of zero.  An error
  confined to one region (a ragged tail, one segment, one head) fails the
  row bar even when the norm over the whole tensor would hide it.

Every comparison also records the norm-wise error, the largest row error
and the largest absolute difference; with LA_PARITY_REPORT=<path> set, the
test session writes them to that file (one JSON object per comparison).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle

# Tolerances (relative errors as defined above):
#  - float32 inputs: 1e-5;
#  - bf16 inputs with a float32 output: 2e-3 (fp32 state, bf16 tensor-core products);
#  - bf16 inputs with a bf16 output: 2e-3 plus the output rounding itself, which
#    is at most 2^-8 of every element (round-to-nearest into 8 significant bits),
#    so by the triangle inequality the bound is 2e-3 + 2^-8 (row by row as well).
TOL_F32 = 1e-5
TOL_BF16 = 2e-3
TOL_BF16_OUT = 2e-3 + 2.0 ** -8
# rows whose reference norm is below this fraction of the tensor's rms row norm
# are held to an absolute bar of tol * ROW_FLOOR * rms_row
ROW_FLOOR = 1e-2

RECORDS: list = []


def tol_for(io_dtype, out_dtype):
    if io_dtype == torch.float32:
        return TOL_F32 if out_dtype == torch.float32 else TOL_F32 + 2.0 ** -8
    return TOL_BF16 if out_dtype == torch.float32 else TOL_BF16_OUT


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def row_errors(got, ref):
    """Per-row relative errors ||d_r|| / max(||ref_r||, ROW_FLOOR * rms_row)
    along the last axis, flattened over the leading axes."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    n = ref.shape[-1] if ref.ndim else 1
    g2 = got.reshape(-1, n)
    r2 = ref.reshape(-1, n)
    rn = np.linalg.norm(r2, axis=1)
    rms = float(np.sqrt(np.mean(rn ** 2))) if rn.size else 0.0
    den = np.maximum(rn, ROW_FLOOR * rms)
    dn = np.linalg.norm(g2 - r2, axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        e = np.where(den > 0, dn / np.where(den > 0, den, 1.0), np.where(dn > 0, np.inf, 0.0))
    return e


def to64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def assert_close(got, ref, tol, what=""):
    """Norm-wise and row-by-row comparison (module docstring); returns the
    norm-wise relative error."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.shape != ref.shape:
        assert got.size == ref.size, f"{what}: shape {got.shape} != {ref.shape}"
        got = got.reshape(ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    e = rel_err(got, ref)
    rows = row_errors(got, ref)
    worst = int(np.argmax(rows)) if rows.size else 0
    row_max = float(rows[worst]) if rows.size else 0.0
    abs_max = float(np.max(np.abs(got - ref))) if got.size else 0.0
    rec = {"what": what, "tol": tol, "norm_rel": e, "row_rel_max": row_max, "abs_max": abs_max,
           "rows": int(rows.size), "shape": list(ref.shape)}
    if rows.size:
        r2 = ref.reshape(-1, ref.shape[-1])
        rn = np.linalg.norm(r2, axis=1)
        rms = float(np.sqrt(np.mean(rn ** 2)))
        rec["worst_row"] = worst
        rec["worst_row_ref_over_rms"] = float(rn[worst] / rms) if rms > 0 else 0.0
        rec["rows_over_tol"] = int(np.sum(rows > tol))
    RECORDS.append(rec)
    assert e <= tol, f"{what}: rel err {e:.3e} > {tol:.3e} (max abs diff {abs_max:.3e})"
    if rows.size:
        idx = np.unravel_index(worst, ref.shape[:-1]) if ref.ndim > 1 else (worst,)
        assert row_max <= tol, (f"{what}: row {tuple(int(i) for i in idx)} rel err {row_max:.3e} > {tol:.3e} "
                                f"(norm-wise {e:.3e}, max abs diff {abs_max:.3e})")
    return e


def write_report(path=None):
    path = path or os.environ.get("LA_PARITY_REPORT")
    if not path or not RECORDS:
        return
    with open(path, "a") as f:
        for r in RECORDS:
            f.write(json.dumps(r) + "\n")
    RECORDS.clear()


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
