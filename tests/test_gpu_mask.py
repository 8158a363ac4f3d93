"""GPU parity of the sequence-validity mask ("[Feature] LinearAttention layer
for Keras", Masking): the CUDA library through its masked C entry points
against the CPU oracle with the same mask.

Causal: an invalid step leaves (S, Z) unchanged -- no update and, for the
gated rule, no decay -- and outputs zero.  Non-causal: invalid keys/values
leave the global sums and invalid queries output zero.  Every mask layout the
request's tests name is covered (right and left padding, interior gaps, all
false, all true) plus random validity; outputs at invalid steps must be
exactly zero, everything else within the tolerances of tests/parity_utils.py.
"""
import numpy as np
import pytest
import torch

import kernelized_linear_attention_02_gb300 as la
import linattn_inputs as inputs
from parity_utils import assert_close, to64, tol_for
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from kernelized_linear_attention_02_gb300 import build
    build.build()
    la.lib()
    la.la_device_error(reset=True)
    yield
    assert la.la_device_error(reset=True) == 0, "a tensor-core kernel gave up on a bounded wait"


def rand(shape, seed, dtype, std=1.0):
    g = inputs.generator(seed, DEV)
    return inputs.normal(shape, g, std, dtype=dtype, device=DEV)


def assert_zero_where_invalid(y, mask, what):
    """y (B, T, H, D): every output of an invalid step is exactly 0."""
    bad = y[~mask.to(y.device)]
    assert bad.numel() == 0 or torch.count_nonzero(bad).item() == 0, f"{what}: nonzero output at an invalid step"


def masked_case(B, T, Hq, Hkv, Dk, Dv, dtype, kind, fmap, norm, rule="linear", seed=0, S0=True,
                out_dtype=torch.float32, scale=1.0, decay_mean=3.0):
    std = 0.5 if fmap == "elu_plus_one" else 1.0
    q = rand((B, T, Hq, Dk), seed, dtype, std)
    k = rand((B, T, Hkv, Dk), seed + 1, dtype, std)
    v = rand((B, T, Hkv, Dv), seed + 2, dtype)
    decay = None
    if rule == "gated":
        decay = torch.nn.functional.logsigmoid(rand((B, T, Hkv), seed + 3, torch.float32) + decay_mean).to(dtype)
    mask = inputs.validity_mask(kind, B, T, seed, DEV)
    init = None
    if S0:
        init = (rand((B, Hkv, Dk, Dv), seed + 4, torch.float32),
                rand((B, Hkv, Dk), seed + 5, torch.float32).abs() + 1.0 if norm else None)
    y, (S, Z) = la.la_forward_causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm,
                                     scale=scale, update_rule=rule, decay=decay, initial_state=init,
                                     return_state=True, out_dtype=out_dtype, mask=mask)
    torch.cuda.synchronize()
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm,
                               scale=scale, rule=rule, decay=decay, mask=mask,
                               S0=None if init is None else init[0], Z0=None if init is None else init[1])
    assert_zero_where_invalid(y, mask, "y")
    assert_close(to64(y), yr, tol_for(dtype, out_dtype), "y")
    assert_close(to64(S), Sr, tol_for(dtype, torch.float32), "S")
    if norm:
        assert_close(to64(Z), Zr, 1e-5, "Z")
    return mask, y, S, Z


SHAPES = [  # B, T, Hq, Hkv, Dk, Dv
    (2, 37, 2, 2, 16, 16),
    (2, 300, 4, 4, 64, 64),
    (1, 257, 8, 2, 128, 128),
    (2, 200, 6, 2, 64, 64),
    (2, 130, 3, 1, 32, 64),
]
MODES = [("elu_plus_one", True), ("relu", True), ("none", False)]
ids = lambda s: "x".join(map(str, s))


@pytest.mark.parametrize("shape", SHAPES, ids=ids)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("kind", inputs.MASK_KINDS)
@pytest.mark.parametrize("mode", MODES, ids=lambda m: f"{m[0]}-{'norm' if m[1] else 'raw'}")
def test_causal_masked(shape, dtype, kind, mode):
    masked_case(*shape, dtype, kind, *mode, seed=shape[1] + shape[4])


@pytest.mark.parametrize("shape", SHAPES, ids=ids)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("kind", ["right", "gaps", "random"])
def test_gated_masked(shape, dtype, kind):
    """Gated rule: an invalid step takes no decay either (S_t = S_{t-1})."""
    masked_case(*shape, dtype, kind, "none", False, rule="gated", seed=5, scale=0.0)


@pytest.mark.parametrize("kind", ["right", "left", "gaps", "random"])
def test_causal_masked_bf16_output(kind):
    masked_case(2, 300, 4, 4, 64, 64, torch.bfloat16, kind, "elu_plus_one", True, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("shape", [(1, 3001, 2, 2, 64, 64), (1, 2500, 2, 2, 128, 128), (2, 1500, 4, 1, 64, 64)],
                         ids=ids)
@pytest.mark.parametrize("rule", ["linear", "gated"])
def test_masked_sequence_segments(shape, rule):
    """Few (batch, kv head) streams: the sequence is split into segments whose
    state increments are folded; invalid runs cross segment boundaries."""
    fmap, norm = ("elu_plus_one", True) if rule == "linear" else ("none", False)
    for kind in ("gaps", "random", "left"):
        masked_case(*shape, torch.bfloat16, kind, fmap, norm, rule=rule, seed=17)



@pytest.mark.parametrize("kind", ["right", "left", "gaps", "random"])
def test_masked_state_pass_sub_segments(kind):
    """The masked state pass on half-length sub-segments (head size 64, 16
    streams of 64 chunks): invalid runs cross sub-segment boundaries."""
    masked_case(2, 64 * 63 + 37, 16, 8, 64, 64, torch.bfloat16, kind, "elu_plus_one", True, seed=23)


def test_masked_one_stream_longest_fold():
    """The masked state pass with one stream of 601 chunks (300 sub-segments
    folded by the last segment), interior gaps crossing their boundaries."""
    masked_case(1, 64 * 600 + 17, 2, 1, 64, 64, torch.bfloat16, "gaps", "elu_plus_one", True, seed=29)


@pytest.mark.parametrize("shape", SHAPES, ids=ids)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("kind", inputs.MASK_KINDS)
@pytest.mark.parametrize("mode", MODES[:2] + [("relu", False)], ids=lambda m: f"{m[0]}-{'norm' if m[1] else 'raw'}")
def test_noncausal_masked(shape, dtype, kind, mode):
    B, T, Hq, Hkv, Dk, Dv = shape
    fmap, norm = mode
    q = rand((B, T, Hq, Dk), 11, dtype, 0.5)
    k = rand((B, T, Hkv, Dk), 12, dtype, 0.5)
    v = rand((B, T, Hkv, Dv), 13, dtype)
    mask = inputs.validity_mask(kind, B, T, 3, DEV)
    y = la.la_forward_noncausal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm,
                                out_dtype=torch.float32, mask=mask)
    torch.cuda.synchronize()
    yr = oracle.noncausal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm, mask=mask)
    assert_zero_where_invalid(y, mask, "non-causal y")
    assert_close(to64(y), yr, tol_for(dtype, torch.float32), "non-causal")


def test_masked_non_finite_padding_is_never_read():
    """Invalid steps contribute nothing even when their q, k, v hold NaN or
    inf (padding that was never initialised)."""
    B, T, H, D = 2, 300, 4, 64
    kind_mask = inputs.validity_mask("gaps", B, T, 9, DEV)
    q = rand((B, T, H, D), 1, torch.bfloat16, 0.5)
    k = rand((B, T, H, D), 2, torch.bfloat16, 0.5)
    v = rand((B, T, H, D), 3, torch.bfloat16)
    for x, val in ((q, float("nan")), (k, float("inf")), (v, float("nan"))):
        x[~kind_mask] = val
    y, (S, Z) = la.la_forward_causal(q, k, v, q_heads=H, kv_heads=H, return_state=True, out_dtype=torch.float32,
                                     mask=kind_mask)
    torch.cuda.synchronize()
    clean = lambda x: torch.where(kind_mask[:, :, None, None], x, torch.zeros_like(x))
    yr, Sr, Zr = oracle.causal(clean(q), clean(k), clean(v), q_heads=H, kv_heads=H, mask=kind_mask)
    assert_zero_where_invalid(y, kind_mask, "y")
    assert_close(to64(y), yr, tol_for(torch.bfloat16, torch.float32), "y")
    assert_close(to64(S), Sr, tol_for(torch.bfloat16, torch.float32), "S")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("rule", ["linear", "gated"])
def test_masked_decode_steps(dtype, rule):
    """A masked prefill, then steps with a per-sequence mask, equal one masked
    causal pass; a sequence whose step is invalid keeps S and Z bit for bit."""
    B, T0, steps, Hq, Hkv, D = 4, 40, 8, 4, 2, 64
    fmap, norm = ("elu_plus_one", True) if rule == "linear" else ("none", False)
    T = T0 + steps
    q = rand((B, T, Hq, D), 51, dtype, 0.5)
    k = rand((B, T, Hkv, D), 52, dtype, 0.5)
    v = rand((B, T, Hkv, D), 53, dtype)
    decay = None
    if rule == "gated":
        decay = torch.nn.functional.logsigmoid(rand((B, T, Hkv), 54, torch.float32) + 3.0).to(dtype)
    mask = inputs.validity_mask("random", B, T, 55, DEV)
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm, update_rule=rule,
              out_dtype=torch.float32)
    sl = lambda x, a, b: None if x is None else x[:, a:b].contiguous()
    _, (S, Z) = la.la_forward_causal(sl(q, 0, T0), sl(k, 0, T0), sl(v, 0, T0), decay=sl(decay, 0, T0),
                                     return_state=True, mask=sl(mask, 0, T0), **kw)
    ys = []
    for t in range(T0, T):
        S_before = S.clone()
        Z_before = Z.clone() if Z is not None else None
        ys.append(la.la_decode_step(sl(q, t, t + 1), sl(k, t, t + 1), sl(v, t, t + 1), S, Z,
                                    decay=sl(decay, t, t + 1), mask=sl(mask, t, t + 1), **kw))
        torch.cuda.synchronize()
        off = ~mask[:, t]
        assert torch.equal(S[off], S_before[off]), "state of an invalid step changed"
        if Z is not None:
            assert torch.equal(Z[off], Z_before[off])
    torch.cuda.synchronize()
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm,
                               rule=rule, decay=decay, mask=mask)
    yd = torch.cat(ys, 1)
    assert_zero_where_invalid(yd, mask[:, T0:], "decode y")
    tol = tol_for(dtype, torch.float32)
    assert_close(to64(yd), yr[:, T0:], tol, "decode y")
    assert_close(to64(S), Sr, tol, "decode S")
    if norm:
        assert_close(to64(Z), Zr, 1e-5, "decode Z")


def test_masked_chunked_equals_full():
    """Masked calls with carried state equal one masked full call."""
    B, T, H, D = 2, 700, 4, 64
    q = rand((B, T, H, D), 61, torch.bfloat16, 0.5)
    k = rand((B, T, H, D), 62, torch.bfloat16, 0.5)
    v = rand((B, T, H, D), 63, torch.bfloat16)
    mask = inputs.validity_mask("gaps", B, T, 64, DEV)
    kw = dict(q_heads=H, kv_heads=H, out_dtype=torch.float32)
    S, Z = la.la_get_initial_state(B, H, D, D)
    ys = []
    for a, b in zip([0, 1, 129, 300, 555], [1, 129, 300, 555, 700]):
        c = lambda x: x[:, a:b].contiguous()
        ys.append(la.la_forward_causal(c(q), c(k), c(v), initial_state=(S, Z), return_state=True, state_out=(S, Z),
                                       mask=c(mask), **kw)[0])
    torch.cuda.synchronize()
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=H, kv_heads=H, mask=mask)
    assert_close(to64(torch.cat(ys, 1)), yr, 2e-3, "chunked masked")
    assert_close(to64(S), Sr, 2e-3, "chunked masked S")
    assert_close(to64(Z), Zr, 1e-5, "chunked masked Z")


def test_masked_workload_sampled_slices():
    """The right-padded 2k prefill at full size, in the launch configuration
    the benchmark times: sampled (batch, kv head) streams against the oracle
    with the same mask, and zeros at every padded step."""
    w = inputs.PREFILL_2K_RIGHTPAD
    q, k, v, _ = inputs.make_qkv(w, device=DEV)
    mask = inputs.validity_mask(w.mask, w.B, w.T, w.seed, DEV)
    kw = dict(q_heads=w.q_heads, kv_heads=w.kv_heads, feature_map=w.feature_map, use_normalizer=w.use_normalizer,
              epsilon=w.eps, scale=w.scale)
    y = la.la_forward_causal(q, k, v, mask=mask, **kw)
    torch.cuda.synchronize()
    assert_zero_where_invalid(y, mask, "y")
    G = w.q_heads // w.kv_heads
    for b, hk in [(0, 0), (1, 5), (2, 3), (3, 7)]:
        yr, _, _ = oracle.causal(q[b:b + 1, :, hk * G:(hk + 1) * G], k[b:b + 1, :, hk:hk + 1],
                                 v[b:b + 1, :, hk:hk + 1], q_heads=G, kv_heads=1, feature_map=w.feature_map,
                                 use_normalizer=w.use_normalizer, eps=w.eps, scale=w.scale, mask=mask[b:b + 1])
        assert_close(to64(y[b:b + 1, :, hk * G:(hk + 1) * G]), yr, tol_for(w.dtype, w.dtype), f"slice {b},{hk}")


def test_mask_argument_checks():
    q = torch.zeros(2, 8, 2, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        la.la_forward_causal(q, q, q, q_heads=2, kv_heads=2, mask=torch.ones(2, 7, dtype=torch.bool, device=DEV))
    with pytest.raises(ValueError):
        la.la_forward_causal(q, q, q, q_heads=2, kv_heads=2, mask=torch.ones(2, 8, dtype=torch.float32, device=DEV))


@pytest.mark.parametrize("shape", [(1, 3001, 2, 2, 64, 64), (2, 2600, 4, 2, 128, 128)], ids=ids)
@pytest.mark.parametrize("kind", ["gaps", "left"])
def test_noncausal_masked_segments(shape, kind):
    """Long non-causal calls with few streams: the global state is reduced over
    sequence segments, and invalid runs cross their boundaries."""
    B, T, Hq, Hkv, Dk, Dv = shape
    q = rand((B, T, Hq, Dk), 71, torch.bfloat16, 0.5)
    k = rand((B, T, Hkv, Dk), 72, torch.bfloat16, 0.5)
    v = rand((B, T, Hkv, Dv), 73, torch.bfloat16)
    mask = inputs.validity_mask(kind, B, T, 74, DEV)
    y = la.la_forward_noncausal(q, k, v, q_heads=Hq, kv_heads=Hkv, out_dtype=torch.float32, mask=mask)
    torch.cuda.synchronize()
    yr = oracle.noncausal(q, k, v, q_heads=Hq, kv_heads=Hkv, mask=mask)
    assert_zero_where_invalid(y, mask, "y")
    assert_close(to64(y), yr, tol_for(torch.bfloat16, torch.float32), "non-causal segments")
