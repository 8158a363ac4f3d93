"""CPU-only: property-based checks of the oracle against the O(T^2) brute
force over randomly drawn shapes (batch, length, head grouping, head sizes),
feature maps, the normalizer, the gated rule and validity masks.  Skipped
where hypothesis is not installed."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st

import oracle
from oracle import bruteforce as bf


@st.composite
def problems(draw):
    B = draw(st.integers(1, 2))
    T = draw(st.integers(1, 24))
    Hkv = draw(st.integers(1, 2))
    G = draw(st.integers(1, 3))
    Dk = draw(st.integers(1, 6))
    Dv = draw(st.integers(1, 6))
    rule = draw(st.sampled_from(["linear", "gated"]))
    if rule == "gated":
        fmap, norm = "none", False
    else:
        fmap = draw(st.sampled_from(["elu_plus_one", "relu", "none"]))
        norm = fmap != "none" and draw(st.booleans())
    masked = draw(st.booleans())
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return B, T, Hkv * G, Hkv, Dk, Dv, rule, fmap, norm, masked, seed


@settings(max_examples=40, deadline=None)
@given(problems())
def test_recurrence_equals_bruteforce(pr):
    B, T, Hq, Hkv, Dk, Dv, rule, fmap, norm, masked, seed = pr
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, Dk)) * 0.7
    k = rng.standard_normal((B, T, Hkv, Dk)) * 0.7
    v = rng.standard_normal((B, T, Hkv, Dv))
    S0 = rng.standard_normal((B, Hkv, Dk, Dv))
    Z0 = np.abs(rng.standard_normal((B, Hkv, Dk))) + 0.5 if norm else None
    decay = np.log(1 / (1 + np.exp(-rng.standard_normal((B, T, Hkv)) - 2.0))) if rule == "gated" else None
    mask = rng.random((B, T)) < 0.7 if masked else np.ones((B, T), bool)
    kw = dict(feature_map=fmap, use_normalizer=norm, eps=1e-3, scale=0.9)
    y, S, Z = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, rule=rule, decay=decay, S0=S0, Z0=Z0,
                            mask=mask if masked else None, **kw)
    for b in range(B):
        idx = np.nonzero(mask[b])[0]
        assert np.all(y[b, ~mask[b]] == 0.0)
        if idx.size == 0:
            np.testing.assert_array_equal(S[b], S0[b])
            continue
        sl = lambda x: None if x is None else x[b:b + 1, idx]
        yb = bf.attention_bthd(sl(q), sl(k), sl(v), q_heads=Hq, kv_heads=Hkv, causal=True, decay=sl(decay),
                               S0=S0[b:b + 1], Z0=None if Z0 is None else Z0[b:b + 1], **kw)
        np.testing.assert_allclose(y[b, idx], yb[0], rtol=1e-9, atol=1e-9)
