"""GPU parity at the full sizes of the measured workloads, in the launch
configuration the benchmark uses, against the oracle on sampled (batch,
kv-head) streams that the oracle computes in full."""
import numpy as np
import pytest
import torch

import kernelized_linear_attention_02_gb300 as la
import linattn_inputs as inputs
import oracle
from parity_utils import assert_close, gpu_slices, oracle_slices, to64, tol_for

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


def samples(B, Hkv, n=4, seed=0):
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (B - 1, Hkv - 1)}
    while len(picks) < min(n, B * Hkv):
        picks.add((int(rng.integers(B)), int(rng.integers(Hkv))))
    return sorted(picks)


def kwargs(w):
    return dict(q_heads=w.q_heads, kv_heads=w.kv_heads, feature_map=w.feature_map,
                use_normalizer=w.use_normalizer, epsilon=w.eps, scale=w.scale, update_rule=w.rule)


def okw(w):
    return dict(feature_map=w.feature_map, use_normalizer=w.use_normalizer, eps=w.eps, scale=w.scale,
                rule=w.rule)


CAUSAL = [inputs.PREFILL_2K, inputs.LONG_8K, inputs.LONG_8K_UNNORM, inputs.ONNX_LINEAR, inputs.ONNX_GATED]


@pytest.mark.parametrize("w", CAUSAL, ids=lambda w: w.name)
def test_causal_workload_sampled(w):
    q, k, v, d = inputs.make_qkv(w, device=DEV)
    G = w.q_heads // w.kv_heads
    sm = samples(w.B, w.kv_heads, n=4 if w.T <= 8192 else 3)
    yr, Sr, Zr = oracle_slices(q, k, v, sm, G, decay=d, **okw(w))
    # float32 output: the compute itself at the 2e-3 bar
    y32, (S, Z) = la.la_forward_causal(q, k, v, decay=d, return_state=True, out_dtype=torch.float32,
                                       **kwargs(w))
    torch.cuda.synchronize()
    assert_close(to64(gpu_slices(y32, sm, G)), yr, tol_for(w.dtype, torch.float32), "y (fp32 out)")
    Ss = torch.stack([S[b, hk] for b, hk in sm])
    assert_close(to64(Ss), Sr[:, 0], 2e-3, "final S")
    if w.use_normalizer:
        Zs = torch.stack([Z[b, hk] for b, hk in sm])
        assert_close(to64(Zs), Zr[:, 0], 1e-5, "final Z")
    del y32
    # bf16 output, the benchmarked configuration
    y16 = la.la_forward_causal(q, k, v, decay=d, **kwargs(w))
    torch.cuda.synchronize()
    assert y16.dtype == w.dtype
    assert_close(to64(gpu_slices(y16, sm, G)), yr, tol_for(w.dtype, w.dtype), "y (bf16 out)")
    assert torch.isfinite(y16).all()


def test_prefill_2k_in_four_chunks_with_carried_state():
    """The 2k-token prefill run as 4 calls of 512 tokens with initial_state /
    return_state equals the full call (Keras request, Streaming State)."""
    w = inputs.PREFILL_2K
    q, k, v, _ = inputs.make_qkv(w, device=DEV)
    kw = kwargs(w)
    y_full, (S_full, Z_full) = la.la_forward_causal(q, k, v, return_state=True, out_dtype=torch.float32, **kw)
    S, Z = la.la_get_initial_state(w.B, w.kv_heads, w.Dk, w.Dv)
    ys = []
    for c in range(4):
        sl = slice(512 * c, 512 * (c + 1))
        ys.append(la.la_forward_causal(q[:, sl].contiguous(), k[:, sl].contiguous(), v[:, sl].contiguous(),
                                       initial_state=(S, Z), return_state=True, state_out=(S, Z),
                                       out_dtype=torch.float32, **kw)[0])
    torch.cuda.synchronize()
    y_chunked = torch.cat(ys, 1)
    # both equal the oracle, and each other to well within the bar
    sm = samples(w.B, w.kv_heads)
    yr, Sr, Zr = oracle_slices(q, k, v, sm, 1, **okw(w))
    assert_close(to64(gpu_slices(y_chunked, sm, 1)), yr, 2e-3, "chunked y")
    assert_close(to64(y_chunked), to64(y_full), 1e-3, "chunked vs full")
    assert_close(to64(S), to64(S_full), 1e-4, "chunked vs full S")
    assert_close(to64(Z), to64(Z_full), 1e-5, "chunked vs full Z")


@pytest.mark.parametrize("w", [inputs.LONG_8K, inputs.LONG_8K_UNNORM], ids=lambda w: w.name)
def test_noncausal_workload_sampled(w):
    q, k, v, _ = inputs.make_qkv(w, device=DEV)
    kw = kwargs(w)
    kw.pop("update_rule")
    y = la.la_forward_noncausal(q, k, v, out_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    sm = samples(w.B, w.kv_heads)
    qs = torch.stack([q[b, :, hk:hk + 1] for b, hk in sm]).cpu()
    ks = torch.stack([k[b, :, hk:hk + 1] for b, hk in sm]).cpu()
    vs = torch.stack([v[b, :, hk:hk + 1] for b, hk in sm]).cpu()
    yr = oracle.noncausal(qs, ks, vs, q_heads=1, kv_heads=1, feature_map=w.feature_map,
                          use_normalizer=w.use_normalizer, eps=w.eps, scale=w.scale)
    assert_close(to64(gpu_slices(y, sm, 1)), yr, 2e-3, "non-causal y")
    # the last causal row equals the non-causal row (global state == final prefix state)
    yc = la.la_forward_causal(q[:, -64:].contiguous(), k[:, -64:].contiguous(), v[:, -64:].contiguous(),
                              out_dtype=torch.float32, **kwargs(w))  # smoke of the short path
    assert torch.isfinite(yc).all()


def test_decode_workload_sampled():
    """State from a 4096-token prefill, then 1024 single-token steps; sampled
    streams against the oracle run over all 5120 tokens."""
    w = inputs.DECODE
    steps = inputs.DECODE_STEPS
    kw = kwargs(w)
    q, k, v, _ = inputs.make_qkv(w, device=DEV)
    _, (S, Z) = la.la_forward_causal(q, k, v, return_state=True, **kw)
    g = inputs.generator(1000, DEV)
    tq = inputs.normal((steps, w.B, 1, w.q_heads, w.Dk), g, dtype=w.dtype, device=DEV)
    tk = inputs.normal((steps, w.B, 1, w.kv_heads, w.Dk), g, dtype=w.dtype, device=DEV)
    tv = inputs.normal((steps, w.B, 1, w.kv_heads, w.Dv), g, dtype=w.dtype, device=DEV)
    ys = torch.empty(steps, w.B, 1, w.q_heads, w.Dv, dtype=torch.float32, device=DEV)
    for i in range(steps):
        la.la_decode_step(tq[i], tk[i], tv[i], S, Z, out=ys[i], out_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    sm = samples(w.B, w.kv_heads, n=6)
    qs = torch.stack([torch.cat([q[b, :, h], tq[:, b, 0, h]], 0) for b, h in sm])[:, :, None]
    ks = torch.stack([torch.cat([k[b, :, h], tk[:, b, 0, h]], 0) for b, h in sm])[:, :, None]
    vs = torch.stack([torch.cat([v[b, :, h], tv[:, b, 0, h]], 0) for b, h in sm])[:, :, None]
    yr, Sr, Zr = oracle.causal(qs.cpu(), ks.cpu(), vs.cpu(), q_heads=1, kv_heads=1, **okw(w))
    ydec = torch.stack([ys[:, b, 0, h] for b, h in sm])
    assert_close(to64(ydec), yr[:, w.T:, 0], 2e-3, "decode y")
    assert_close(to64(torch.stack([S[b, h] for b, h in sm])), Sr[:, 0], 2e-3, "decode S")
    assert_close(to64(torch.stack([Z[b, h] for b, h in sm])), Zr[:, 0], 1e-5, "decode Z")


@pytest.mark.parametrize("rule", ["linear", "gated"])
def test_many_segments_with_initial_state(rule):
    """Few streams, long sequence: the sequence splits into many segments
    (state pass, scan, output pass), with a carried initial state and a
    ragged tail."""
    B, T, Hq, Hkv, D = 1, 3001, 8, 2, 128
    g = inputs.generator(5, DEV)
    q = inputs.normal((B, T, Hq, D), g, dtype=torch.bfloat16, device=DEV)
    k = inputs.normal((B, T, Hkv, D), g, 0.3, dtype=torch.bfloat16, device=DEV)
    v = inputs.normal((B, T, Hkv, D), g, dtype=torch.bfloat16, device=DEV)
    S0 = inputs.normal((B, Hkv, D, D), g, device=DEV)
    d = None
    fmap, norm = ("elu_plus_one", True) if rule == "linear" else ("none", False)
    Z0 = inputs.normal((B, Hkv, D), g, device=DEV).abs() + 1.0 if norm else None
    if rule == "gated":
        d = torch.nn.functional.logsigmoid(inputs.normal((B, T, Hkv), g, device=DEV) + 4.0).to(torch.bfloat16)
    y, (S, Z) = la.la_forward_causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm,
                                     update_rule=rule, decay=d, initial_state=(S0, Z0), return_state=True,
                                     out_dtype=torch.float32, scale=0.0)
    torch.cuda.synchronize()
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm,
                               rule=rule, decay=d, S0=S0, Z0=Z0, scale=0.0)
    assert_close(to64(y), yr, 2e-3, "y")
    assert_close(to64(S), Sr, 2e-3, "S")
    if norm:
        assert_close(to64(Z), Zr, 1e-5, "Z")
