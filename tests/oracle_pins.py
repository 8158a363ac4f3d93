"""Pins that tie the CPU oracle to what the pages and the mathematics fix.

Each ``pin_*`` function raises AssertionError when the oracle (the compiled C
library ``lib``; None = the committed one) disagrees.  They are run by
``test_oracle.py`` and, against deliberately broken copies of the oracle, by
``test_oracle_mutants.py``.  None of them re-types the oracle's formula: each
compares it with a printed value, a second formulation (the O(T^2) brute
force), a closed form or an invariant.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
from oracle import bruteforce as bf
from linattn_inputs import tiny_paper_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


ONNX = _load("onnx_linear_attention_examples.json")["examples"]
P2 = _load("causal_vs_noncausal_mean_abs_diff.json")


def pin_onnx_example(name, lib=None):
    """ONNX-light 'LinearAttention', Examples: output and present_state as printed."""
    e = ONNX[name]
    dt = np.float16 if e.get("dtype") == "float16" else np.float32
    f = lambda key: None if key not in e else np.array(e[key], dtype=dt).astype(np.float64)
    y, S, _ = oracle.causal(f("query"), f("key"), f("value"), q_heads=e["q_num_heads"],
                            kv_heads=e["kv_num_heads"], feature_map="none", use_normalizer=False,
                            scale=e.get("scale", 0.0), rule=e["update_rule"], decay=f("decay"),
                            beta=f("beta"), S0=f("past_state"), lib=lib)
    y_ref = np.array(e["output"], dtype=np.float64).reshape(y.shape)
    S_ref = np.array(e["present_state"], dtype=np.float64)
    # printed float32 values carry ~8 significant digits; the fp16 example was
    # computed in fp16 arithmetic, so it is held to two fp16 ulps at |x|~2
    atol = 4e-3 if dt == np.float16 else 5e-7
    rtol = 2e-3 if dt == np.float16 else 1e-6
    np.testing.assert_allclose(y, y_ref, rtol=rtol, atol=atol, err_msg=name + " output")
    np.testing.assert_allclose(S, S_ref, rtol=rtol, atol=atol, err_msg=name + " state")


def pin_paper_mean_abs_diff(lib=None):
    """'Causal Linear Attention', Out[23]: mean |causal - non-causal| = 0.2188."""
    Q, K, V = tiny_paper_inputs(P2["seed"], P2["n"], P2["d"])
    yc, _, _ = oracle.causal(Q[None], K[None], V[None], q_heads=1, kv_heads=1,
                             feature_map="elu_plus_one", eps=P2["eps"], lib=lib)
    yn = oracle.noncausal(Q[None], K[None], V[None], q_heads=1, kv_heads=1,
                          feature_map="elu_plus_one", eps=P2["eps"], lib=lib)
    diff = float(np.mean(np.abs(yc - yn)))
    assert round(diff, P2["printed_decimals"]) == P2["printed_mean_abs_diff"], diff


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def pin_recurrence_vs_bruteforce(lib=None, seed=0):
    """The token-by-token recurrence equals the O(T^2) pairwise form, for every
    feature map, with and without the normalizer, with GQA, a carried state,
    and the gated rule with scalar and per-key-dimension decay."""
    rng = np.random.default_rng(seed)
    B, T, Hq, Hkv, Dk, Dv = 2, 23, 4, 2, 5, 3
    cases = []
    for fmap in ("elu_plus_one", "relu", "none"):
        for norm in (True, False):
            if fmap == "none" and norm:
                continue  # identity map can make the denominator vanish
            cases.append(dict(feature_map=fmap, use_normalizer=norm, rule="linear"))
    cases.append(dict(feature_map="none", use_normalizer=False, rule="gated", decay="head"))
    cases.append(dict(feature_map="none", use_normalizer=False, rule="gated", decay="dim"))
    cases.append(dict(feature_map="elu_plus_one", use_normalizer=False, rule="gated", decay="head"))
    for c in cases:
        q = _rand(rng, B, T, Hq, Dk, std=0.7)
        k = _rand(rng, B, T, Hkv, Dk, std=0.7)
        v = _rand(rng, B, T, Hkv, Dv)
        S0 = _rand(rng, B, Hkv, Dk, Dv)
        Z0 = np.abs(_rand(rng, B, Hkv, Dk)) + 0.5 if c["use_normalizer"] else None
        decay = None
        if c.get("decay") == "head":
            decay = np.log(1 / (1 + np.exp(-_rand(rng, B, T, Hkv) - 2.0)))
        elif c.get("decay") == "dim":
            decay = np.log(1 / (1 + np.exp(-_rand(rng, B, T, Hkv * Dk) - 2.0)))
        kw = dict(feature_map=c["feature_map"], use_normalizer=c["use_normalizer"], eps=1e-3,
                  scale=0.75)
        y, _, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, rule=c["rule"], decay=decay,
                                S0=S0, Z0=Z0, lib=lib, **kw)
        yb = bf.attention_bthd(q, k, v, q_heads=Hq, kv_heads=Hkv, causal=True, decay=decay,
                               S0=S0, Z0=Z0, **kw)
        np.testing.assert_allclose(y, yb, rtol=1e-10, atol=1e-10, err_msg=str(c))


def pin_noncausal_vs_bruteforce(lib=None, seed=1):
    rng = np.random.default_rng(seed)
    B, T, Hq, Hkv, Dk, Dv = 2, 17, 6, 3, 4, 6
    for fmap in ("elu_plus_one", "relu"):
        for norm in (True, False):
            q = _rand(rng, B, T, Hq, Dk)
            k = _rand(rng, B, T, Hkv, Dk)
            v = _rand(rng, B, T, Hkv, Dv)
            kw = dict(feature_map=fmap, use_normalizer=norm, eps=1e-3, scale=1.25)
            y = oracle.noncausal(q, k, v, q_heads=Hq, kv_heads=Hkv, lib=lib, **kw)
            yb = bf.attention_bthd(q, k, v, q_heads=Hq, kv_heads=Hkv, causal=False, **kw)
            np.testing.assert_allclose(y, yb, rtol=1e-10, atol=1e-10)


def pin_last_row_equals_noncausal(lib=None, seed=2):
    """At the last position the causal prefix state is the global state."""
    rng = np.random.default_rng(seed)
    for fmap in ("elu_plus_one", "relu"):
        q = _rand(rng, 3, 40, 2, 8)
        k = _rand(rng, 3, 40, 2, 8)
        v = _rand(rng, 3, 40, 2, 8)
        yc, _, _ = oracle.causal(q, k, v, q_heads=2, kv_heads=2, feature_map=fmap, lib=lib)
        yn = oracle.noncausal(q, k, v, q_heads=2, kv_heads=2, feature_map=fmap, lib=lib)
        np.testing.assert_allclose(yc[:, -1], yn[:, -1], rtol=1e-12, atol=1e-12)
        assert np.abs(yc[:, 0] - yn[:, 0]).max() > 1e-3  # and not elsewhere


def pin_chunked_equals_full(lib=None, seed=3):
    """Chunked execution with the carried (S, Z) equals one full call (Keras
    request, Streaming State); checked on uneven chunk boundaries too."""
    rng = np.random.default_rng(seed)
    B, T, H, D = 2, 64, 2, 16
    q = _rand(rng, B, T, H, D, std=0.5)
    k = _rand(rng, B, T, H, D, std=0.5)
    v = _rand(rng, B, T, H, D)
    for norm in (True, False):
        y, S, Z = oracle.causal(q, k, v, q_heads=H, kv_heads=H, use_normalizer=norm, lib=lib)
        for cuts in ([0, 16, 32, 48, 64], [0, 1, 7, 40, 64]):
            Sc = Zc = None
            ys = []
            for a, b in zip(cuts[:-1], cuts[1:]):
                yi, Sc, Zc = oracle.causal(q[:, a:b], k[:, a:b], v[:, a:b], q_heads=H, kv_heads=H,
                                           use_normalizer=norm, S0=Sc, Z0=Zc, lib=lib)
                ys.append(yi)
            np.testing.assert_allclose(np.concatenate(ys, axis=1), y, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(Sc, S, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(Zc, Z, rtol=1e-12, atol=1e-12)


def pin_state_closed_form(lib=None, seed=4):
    """Returned state: S_T = sum_t phi(k_t)^T v_t (outer product k-index by
    v-index), Z_T = sum_t phi(k_t), written out with einsum on phi."""
    rng = np.random.default_rng(seed)
    q = _rand(rng, 1, 9, 1, 3)
    k = _rand(rng, 1, 9, 1, 3)
    v = _rand(rng, 1, 9, 1, 5)
    for fmap in ("elu_plus_one", "relu", "none"):
        _, S, Z = oracle.causal(q, k, v, q_heads=1, kv_heads=1, feature_map=fmap,
                                use_normalizer=False, eps=1e-2, lib=lib)
        fk = bf.phi(k[0, :, 0], fmap, 1e-2)
        np.testing.assert_allclose(S[0, 0], fk.T @ v[0, :, 0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(Z[0, 0], fk.sum(0), rtol=1e-12, atol=1e-12)


def pin_first_token(lib=None):
    """From a zero state, y_0 = v_0 * w / (w + eps) with w = phi(q_0).phi(k_0)
    (the current token is included in its own context)."""
    q = np.array([[[[0.3, -1.2, 0.8]]]])
    k = np.array([[[[-0.4, 0.9, 0.1]]]])
    v = np.array([[[[2.0, -3.0]]]])
    eps = 0.25
    y, _, _ = oracle.causal(q, k, v, q_heads=1, kv_heads=1, feature_map="elu_plus_one",
                            eps=eps, lib=lib)
    w = (1.3 * math.exp(-0.4)) + (math.exp(-1.2) * 1.9) + (1.8 * 1.1)
    np.testing.assert_allclose(y[0, 0, 0], np.array([2.0, -3.0]) * w / (w + eps), rtol=1e-12)


def pin_feature_map_values(lib=None):
    """elu(x)+1 = x+1 (x>0), exp(x) (x<=0); relu(x)+eps (Keras request, Feature
    maps).  With Dk = Dv = 1, q = 0 under elu+1 (phi = 1), v = 1 and no
    normalizer, the first output is phi(k)."""
    xs = np.array([-3.0, -0.5, 0.0, 0.25, 2.0])
    want = {"elu_plus_one": np.array([math.exp(-3.0), math.exp(-0.5), 1.0, 1.25, 3.0]),
            "relu": np.array([0.0, 0.0, 0.0, 0.25, 2.0]) + 0.125}
    for fmap, ref in want.items():
        for x, r in zip(xs, ref):
            qv = 0.0 if fmap == "elu_plus_one" else 1.0
            q = np.array([[[[qv]]]])
            k = np.array([[[[x]]]])
            v = np.ones((1, 1, 1, 1))
            y, _, _ = oracle.causal(q, k, v, q_heads=1, kv_heads=1, feature_map=fmap,
                                    use_normalizer=False, eps=0.125, lib=lib)
            phi_q = 1.0 if fmap == "elu_plus_one" else 1.125
            np.testing.assert_allclose(y[0, 0, 0, 0], phi_q * r, rtol=1e-14, err_msg=fmap)


def pin_constant_value(lib=None, seed=5):
    """V = c everywhere gives y_i = c * D_i / (D_i + eps), D_i = phi(q_i).Z_i."""
    rng = np.random.default_rng(seed)
    q = _rand(rng, 1, 30, 1, 4)
    k = _rand(rng, 1, 30, 1, 4)
    v = np.full((1, 30, 1, 3), -1.75)
    y, _, _ = oracle.causal(q, k, v, q_heads=1, kv_heads=1, eps=1e-9, lib=lib)
    np.testing.assert_allclose(y, -1.75, rtol=1e-7)


def pin_gated_reductions(lib=None, seed=6):
    """g = 0 turns 'gated' into 'linear'; a decay of -inf at step t forgets
    every earlier token, so output t equals a fresh start at t."""
    rng = np.random.default_rng(seed)
    q = _rand(rng, 1, 12, 2, 4)
    k = _rand(rng, 1, 12, 2, 4)
    v = _rand(rng, 1, 12, 2, 4)
    kw = dict(q_heads=2, kv_heads=2, feature_map="none", use_normalizer=False, scale=1.0)
    yl, Sl, _ = oracle.causal(q, k, v, rule="linear", lib=lib, **kw)
    yg, Sg, _ = oracle.causal(q, k, v, rule="gated", decay=np.zeros((1, 12, 2)), lib=lib, **kw)
    np.testing.assert_allclose(yg, yl, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(Sg, Sl, rtol=1e-13, atol=1e-13)
    g = np.zeros((1, 12, 2))
    g[0, 5, :] = -800.0  # exp(-800) == 0 in double
    yg, _, _ = oracle.causal(q, k, v, rule="gated", decay=g, lib=lib, **kw)
    ys, _, _ = oracle.causal(q[:, 5:], k[:, 5:], v[:, 5:], rule="linear", lib=lib, **kw)
    np.testing.assert_allclose(yg[:, 5:], ys, rtol=1e-12, atol=1e-12)


def pin_gqa_equals_repeated_mha(lib=None, seed=7):
    """GQA equals multi-head attention on K/V repeated per query head, with
    query head h reading kv head h // (Hq/Hkv)."""
    rng = np.random.default_rng(seed)
    B, T, Hq, Hkv, D = 2, 11, 6, 2, 4
    q = _rand(rng, B, T, Hq, D)
    k = _rand(rng, B, T, Hkv, D)
    v = _rand(rng, B, T, Hkv, D)
    for fmap, norm in (("elu_plus_one", True), ("none", False)):
        yg, _, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap,
                                 use_normalizer=norm, lib=lib)
        kr = np.repeat(k, Hq // Hkv, axis=2)
        vr = np.repeat(v, Hq // Hkv, axis=2)
        ym, _, _ = oracle.causal(q, kr, vr, q_heads=Hq, kv_heads=Hq, feature_map=fmap,
                                 use_normalizer=norm, lib=lib)
        np.testing.assert_allclose(yg, ym, rtol=1e-13, atol=1e-13)


def pin_scale(lib=None, seed=8):
    """Output scale enters linearly; scale 0 means 1/sqrt(d_k) (ONNX attribute)."""
    rng = np.random.default_rng(seed)
    q = _rand(rng, 1, 7, 2, 9)
    k = _rand(rng, 1, 7, 2, 9)
    v = _rand(rng, 1, 7, 2, 4)
    kw = dict(q_heads=2, kv_heads=2, feature_map="none", use_normalizer=False, lib=lib)
    y1, _, _ = oracle.causal(q, k, v, scale=1.0, **kw)
    y3, _, _ = oracle.causal(q, k, v, scale=3.0, **kw)
    y0, _, _ = oracle.causal(q, k, v, scale=0.0, **kw)
    np.testing.assert_allclose(y3, 3.0 * y1, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(y0, y1 / 3.0, rtol=1e-13, atol=1e-13)


def _masks(rng, B, T):
    """Validity masks of the shapes the Keras request's tests name (Mask and
    state behavior): right padding, left padding, interior gaps, all false,
    all true, and random validity."""
    out = []
    m = np.ones((B, T), bool); m[0, T - 5:] = False; m[1, T // 2:] = False; out.append(m)
    m = np.ones((B, T), bool); m[0, :3] = False; m[1, :T - 4] = False; out.append(m)
    m = np.ones((B, T), bool); m[0, 4:9] = False; m[1, 1::3] = False; out.append(m)
    out.append(np.zeros((B, T), bool))
    out.append(np.ones((B, T), bool))
    out.append(rng.random((B, T)) < 0.6)
    return out


def pin_mask_causal(lib=None, seed=9):
    """Keras request, Masking (causal): an invalid step leaves (S, Z) as they
    were and outputs zero.  So the outputs at the valid steps equal the O(T^2)
    brute force run on the valid tokens alone (with their decays, for the
    gated rule), invalid outputs are exactly 0, and the returned state is the
    closed form S0 + sum over valid t of phi(k_t)^T v_t (linear) with Z
    likewise; for the gated rule the state equals an unmasked pass over the
    valid tokens alone."""
    rng = np.random.default_rng(seed)
    B, T, Hq, Hkv, Dk, Dv = 2, 19, 4, 2, 5, 3
    cases = [dict(feature_map="elu_plus_one", use_normalizer=True, rule="linear"),
             dict(feature_map="relu", use_normalizer=False, rule="linear"),
             dict(feature_map="none", use_normalizer=False, rule="gated")]
    for c in cases:
        for mask in _masks(rng, B, T):
            q = _rand(rng, B, T, Hq, Dk, std=0.7)
            k = _rand(rng, B, T, Hkv, Dk, std=0.7)
            v = _rand(rng, B, T, Hkv, Dv)
            S0 = _rand(rng, B, Hkv, Dk, Dv)
            Z0 = np.abs(_rand(rng, B, Hkv, Dk)) + 0.5 if c["use_normalizer"] else None
            decay = np.log(1 / (1 + np.exp(-_rand(rng, B, T, Hkv) - 2.0))) if c["rule"] == "gated" else None
            kw = dict(feature_map=c["feature_map"], use_normalizer=c["use_normalizer"], eps=1e-3, scale=0.75)
            y, S, Z = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, rule=c["rule"], decay=decay, S0=S0,
                                    Z0=Z0, mask=mask, lib=lib, **kw)
            for b in range(B):
                idx = np.nonzero(mask[b])[0]
                assert np.all(y[b, ~mask[b]] == 0.0), str(c)
                if idx.size:
                    sl = lambda x: None if x is None else x[b:b + 1, idx]
                    yb = bf.attention_bthd(sl(q), sl(k), sl(v), q_heads=Hq, kv_heads=Hkv, causal=True,
                                           decay=sl(decay), S0=S0[b:b + 1],
                                           Z0=None if Z0 is None else Z0[b:b + 1], **kw)
                    np.testing.assert_allclose(y[b, idx], yb[0], rtol=1e-10, atol=1e-10, err_msg=str(c))
                fk = bf.phi(k[b, idx], c["feature_map"], 1e-3)  # (n, Hkv, Dk)
                if c["rule"] == "linear":
                    S_ref = S0[b] + np.einsum("thi,thj->hij", fk, v[b, idx])
                    np.testing.assert_allclose(S[b], S_ref, rtol=1e-11, atol=1e-11, err_msg=str(c))
                    if c["use_normalizer"]:
                        np.testing.assert_allclose(Z[b], Z0[b] + fk.sum(axis=0), rtol=1e-11, atol=1e-11)
                else:
                    _, Sc, _ = oracle.causal(q[b:b + 1, idx], k[b:b + 1, idx], v[b:b + 1, idx], q_heads=Hq,
                                             kv_heads=Hkv, rule="gated", decay=decay[b:b + 1, idx],
                                             S0=S0[b:b + 1], lib=lib, **kw)
                    np.testing.assert_allclose(S[b], Sc[0], rtol=1e-11, atol=1e-11, err_msg=str(c))


def pin_mask_noncausal(lib=None, seed=10):
    """Keras request, Masking (non-causal): invalid keys and values add nothing
    to the global sums and invalid query positions output zero, so the valid
    outputs equal the brute force over the valid positions alone."""
    rng = np.random.default_rng(seed)
    B, T, Hq, Hkv, Dk, Dv = 2, 17, 4, 2, 4, 6
    for fmap, norm in (("elu_plus_one", True), ("relu", False)):
        for mask in _masks(rng, B, T):
            q = _rand(rng, B, T, Hq, Dk)
            k = _rand(rng, B, T, Hkv, Dk)
            v = _rand(rng, B, T, Hkv, Dv)
            kw = dict(feature_map=fmap, use_normalizer=norm, eps=1e-3, scale=1.25)
            y = oracle.noncausal(q, k, v, q_heads=Hq, kv_heads=Hkv, mask=mask, lib=lib, **kw)
            for b in range(B):
                idx = np.nonzero(mask[b])[0]
                assert np.all(y[b, ~mask[b]] == 0.0)
                if idx.size:
                    yb = bf.attention_bthd(q[b:b + 1, idx], k[b:b + 1, idx], v[b:b + 1, idx], q_heads=Hq,
                                           kv_heads=Hkv, causal=False, **kw)
                    np.testing.assert_allclose(y[b, idx], yb[0], rtol=1e-10, atol=1e-10)


def pin_grad_forward_matches_recurrence(lib=None, seed=11):
    """The differentiable float64 recurrence used for gradients computes the
    same outputs as the C oracle (GQA, carried state, every feature map)."""
    import torch
    from oracle import grad as og
    rng = np.random.default_rng(seed)
    B, T, Hq, Hkv, Dk, Dv = 2, 9, 4, 2, 3, 5
    for fmap, norm in (("elu_plus_one", True), ("relu", True), ("none", False), ("elu_plus_one", False)):
        q, k = _rand(rng, B, T, Hq, Dk, std=0.7), _rand(rng, B, T, Hkv, Dk, std=0.7)
        v = _rand(rng, B, T, Hkv, Dv)
        S0 = _rand(rng, B, Hkv, Dk, Dv)
        Z0 = np.abs(_rand(rng, B, Hkv, Dk)) + 0.5 if norm else None
        kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm, eps=1e-3, scale=0.75)
        y, _, _ = oracle.causal(q, k, v, S0=S0, Z0=Z0, lib=lib, **kw)
        t = lambda x: None if x is None else torch.tensor(x, dtype=torch.float64)
        yg = og.causal_forward(t(q), t(k), t(v), S0=t(S0), Z0=t(Z0), **kw).numpy()
        np.testing.assert_allclose(yg, y, rtol=1e-11, atol=1e-11, err_msg=fmap)


def pin_grad_finite_differences(lib=None, seed=12):
    """Keras request, Test Plan (Stability): float64 numerical-gradient checks.
    The autograd gradients of the recurrence match central finite
    differences for q, k, v and the carried state, with and without the
    normalizer, with grouped heads."""
    import torch
    from oracle import grad as og
    g = torch.Generator().manual_seed(seed)
    B, T, Hq, Hkv, Dk, Dv = 1, 5, 2, 1, 3, 2
    for fmap, norm in (("elu_plus_one", True), ("relu", False)):
        q = (torch.randn(B, T, Hq, Dk, generator=g, dtype=torch.float64) * 0.7).requires_grad_(True)
        k = (torch.randn(B, T, Hkv, Dk, generator=g, dtype=torch.float64) * 0.7).requires_grad_(True)
        v = torch.randn(B, T, Hkv, Dv, generator=g, dtype=torch.float64).requires_grad_(True)
        S0 = torch.randn(B, Hkv, Dk, Dv, generator=g, dtype=torch.float64).requires_grad_(True)
        Z0 = (torch.rand(B, Hkv, Dk, generator=g, dtype=torch.float64) + 0.5).requires_grad_(True)
        f = lambda q, k, v, S0, Z0: og.causal_forward(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap,
                                                      use_normalizer=norm, eps=1e-3, scale=1.3, S0=S0,
                                                      Z0=Z0 if norm else None)
        # keep away from the kinks of elu / relu at 0, where one-sided differences disagree
        for x in (q, k):
            with torch.no_grad():
                x.add_(torch.sign(x) * 0.05)
        assert torch.autograd.gradcheck(f, (q, k, v, S0, Z0), eps=1e-6, atol=1e-7, rtol=1e-5)


def pin_delta_overwrite(lib=None, seed=13):
    """ONNX-light "LinearAttention", update rule delta: with beta = 1 and a
    unit key, S_t = S_{t-1} + k (v - S_{t-1}^T k)^T stores v at k exactly
    (S_t^T k = v), overwriting what the key held.  With orthonormal keys
    (basis vectors, some repeated) and the query equal to the key, every
    output is scale * v_t, and the final state maps each key to the last
    value written at it."""
    rng = np.random.default_rng(seed)
    Dk, Dv, T = 4, 3, 7
    order = [0, 1, 2, 1, 3, 0, 2]  # keys e_0, e_1, e_2, e_1 again, ...
    k = np.zeros((1, T, 1, Dk))
    for t, i in enumerate(order):
        k[0, t, 0, i] = 1.0
    v = rng.standard_normal((1, T, 1, Dv))
    beta = np.ones((1, T, 1))
    S0 = rng.standard_normal((1, 1, Dk, Dv))
    y, S, _ = oracle.causal(k.copy(), k, v, q_heads=1, kv_heads=1, feature_map="none", use_normalizer=False,
                            scale=0.5, rule="delta", beta=beta, S0=S0, lib=lib)
    np.testing.assert_allclose(y[0, :, 0], 0.5 * v[0, :, 0], rtol=1e-13, atol=1e-13)
    last = {}
    for t, i in enumerate(order):
        last[i] = v[0, t, 0]
    for i in range(Dk):
        np.testing.assert_allclose(S[0, 0, i], last[i], rtol=1e-13, atol=1e-13)


def pin_gated_delta_without_decay_is_delta(lib=None, seed=14):
    """gated_delta with g = 0 (no decay) equals delta; a decay of -inf before
    step t forgets the earlier state, so step t starts from S = 0."""
    rng = np.random.default_rng(seed)
    B, T, Hq, Hkv, D = 1, 9, 2, 1, 4
    q = rng.standard_normal((B, T, Hq, D))
    k = rng.standard_normal((B, T, Hkv, D))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hkv, D))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, T, Hkv))))
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, beta=beta, lib=lib)
    yd, Sd, _ = oracle.causal(q, k, v, rule="delta", **kw)
    yg, Sg, _ = oracle.causal(q, k, v, rule="gated_delta", decay=np.zeros((B, T, Hkv)), **kw)
    np.testing.assert_allclose(yg, yd, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(Sg, Sd, rtol=1e-13, atol=1e-13)
    g = np.zeros((B, T, Hkv))
    g[0, 4] = -800.0
    yg, _, _ = oracle.causal(q, k, v, rule="gated_delta", decay=g, **kw)
    kw2 = dict(kw, beta=beta[:, 4:])
    ys, _, _ = oracle.causal(q[:, 4:], k[:, 4:], v[:, 4:], rule="delta", **kw2)
    np.testing.assert_allclose(yg[:, 4:], ys, rtol=1e-12, atol=1e-12)


ALL_PINS = [pin_paper_mean_abs_diff, pin_recurrence_vs_bruteforce, pin_noncausal_vs_bruteforce,
            pin_last_row_equals_noncausal, pin_chunked_equals_full, pin_state_closed_form,
            pin_first_token, pin_feature_map_values, pin_constant_value, pin_gated_reductions,
            pin_gqa_equals_repeated_mha, pin_scale, pin_mask_causal, pin_mask_noncausal,
            pin_grad_forward_matches_recurrence, pin_grad_finite_differences, pin_delta_overwrite,
            pin_gated_delta_without_decay_is_delta]


def run_all(lib=None):
    """Run every pin; return the names of those that failed."""
    failed = []
    for name in ONNX:
        try:
            pin_onnx_example(name, lib)
        except (AssertionError, ValueError):
            failed.append(name)
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    return failed
