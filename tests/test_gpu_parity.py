"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Small cases are compared over the whole output, norm-wise and row by row
(every (token, head) output row and every state row against the same
tolerance, tests/parity_utils.py); they span several chunks of the
tensor-core kernels and end on ragged tails.  The workloads at full size are
compared the same way on sampled (batch, kv-head) streams the oracle computes
in full.
"""
import itertools

import numpy as np
import pytest
import torch

import kernelized_linear_attention_02_gb300 as la
import linattn_inputs as inputs
from parity_utils import (assert_close, gpu_slices, oracle_slices, rel_err, to64, tol_for, TOL_F32)
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


def run_case(B, T, Hq, Hkv, Dk, Dv, dtype, out_dtype, fmap, norm, rule="linear", S0=False, seed=0,
             scale=1.0, eps=1e-6, std=1.0, decay_mean=3.0):
    q = rand((B, T, Hq, Dk), seed, dtype, std)
    k = rand((B, T, Hkv, Dk), seed + 1, dtype, std)
    v = rand((B, T, Hkv, Dv), seed + 2, dtype)
    decay = None
    if rule == "gated":
        x = rand((B, T, Hkv), seed + 3, torch.float32) + decay_mean
        decay = torch.nn.functional.logsigmoid(x).to(dtype)
    init = None
    if S0:
        S0t = rand((B, Hkv, Dk, Dv), seed + 4, torch.float32)
        Z0t = rand((B, Hkv, Dk), seed + 5, torch.float32).abs() + 1.0 if norm else None
        init = (S0t, Z0t)
    y, (S, Z) = la.la_forward_causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap,
                                     use_normalizer=norm, epsilon=eps, scale=scale, update_rule=rule,
                                     decay=decay, initial_state=init, return_state=True,
                                     out_dtype=out_dtype)
    torch.cuda.synchronize()
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap,
                               use_normalizer=norm, eps=eps, scale=scale, rule=rule, decay=decay,
                               S0=None if init is None else init[0],
                               Z0=None if init is None else init[1])
    tol = tol_for(dtype, out_dtype)
    assert_close(to64(y), yr, tol, "y")
    assert_close(to64(S), Sr, tol_for(dtype, torch.float32), "S")
    if norm:
        assert_close(to64(Z), Zr, 1e-5, "Z")
    return y, S, Z


# ---------------------------------------------------------------------------
# near-zero denominators (Keras request, Test Plan / Stability: "near-zero
# denominators"; Mathematical definition: eps in the denominator).  Queries
# far below zero make phi(q).Z tiny: with relu+eps every query feature is eps
# itself, with elu+1 at q ~ -16 every feature is ~1e-7, so den = phi(q).Z + eps
# comes within a few eps of eps on the first tokens.


NEAR_ZERO = [  # fmap, query mean, query std
    ("relu", -3.0, 1.0),
    ("elu_plus_one", -16.0, 0.5),
]


@pytest.mark.parametrize("case", NEAR_ZERO, ids=lambda c: c[0])
@pytest.mark.parametrize("cfg", [(torch.bfloat16, 64, 2, 2), (torch.bfloat16, 128, 4, 2), (torch.float32, 64, 2, 2)],
                         ids=["bf16-d64", "bf16-d128-gqa", "f32-d64"])
@pytest.mark.parametrize("carried", [False, True], ids=["zero-state", "carried-state"])
def test_near_zero_denominator(case, cfg, carried):
    fmap, qmean, qstd = case
    dtype, D, Hq, Hkv = cfg
    B, T = 2, 200
    g = inputs.generator(77, DEV)
    q = (inputs.normal((B, T, Hq, D), g, qstd, dtype=torch.float32, device=DEV) + qmean).to(dtype)
    k = inputs.normal((B, T, Hkv, D), g, 0.5, dtype=dtype, device=DEV)
    v = inputs.normal((B, T, Hkv, D), g, 1.0, dtype=dtype, device=DEV)
    init = None
    if carried:  # a small carried key sum keeps den close to eps on the first tokens
        S0 = inputs.normal((B, Hkv, D, D), g, 1e-3, dtype=torch.float32, device=DEV)
        Z0 = inputs.normal((B, Hkv, D), g, 1e-3, dtype=torch.float32, device=DEV).abs()
        init = (S0, Z0)
    y, (S, Z) = la.la_forward_causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=True,
                                     epsilon=1e-6, initial_state=init, return_state=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=True, eps=1e-6,
                               S0=None if init is None else init[0], Z0=None if init is None else init[1])
    tol = tol_for(dtype, torch.float32)
    assert_close(to64(y), yr, tol, "y")
    assert_close(to64(S), Sr, tol, "S")
    assert_close(to64(Z), Zr, 1e-5, "Z")


# ---------------------------------------------------------------------------
# the tiny workload: causal, non-causal, and chunks of 16 with carried state


def test_tiny_workload_fp32():
    w = inputs.TINY
    q, k, v, _ = inputs.make_qkv(w, device=DEV)
    kw = dict(q_heads=w.q_heads, kv_heads=w.kv_heads, feature_map=w.feature_map,
              use_normalizer=w.use_normalizer, epsilon=w.eps, scale=w.scale)
    y, (S, Z) = la.la_forward_causal(q, k, v, return_state=True, **kw)
    yn = la.la_forward_noncausal(q, k, v, **{k_: v_ for k_, v_ in kw.items()})
    # four chunks of 16 tokens, the state carried in place
    Sc, Zc = la.la_get_initial_state(w.B, w.kv_heads, w.Dk, w.Dv)
    ys = []
    for c in range(4):
        sl = slice(16 * c, 16 * (c + 1))
        ys.append(la.la_forward_causal(q[:, sl].contiguous(), k[:, sl].contiguous(), v[:, sl].contiguous(),
                                       initial_state=(Sc, Zc), return_state=True, state_out=(Sc, Zc),
                                       **kw)[0])
    torch.cuda.synchronize()
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=2, kv_heads=2, feature_map=w.feature_map, eps=w.eps)
    ynr = oracle.noncausal(q, k, v, q_heads=2, kv_heads=2, feature_map=w.feature_map, eps=w.eps)
    assert_close(to64(y), yr, TOL_F32, "causal")
    assert_close(to64(yn), ynr, TOL_F32, "non-causal")
    assert_close(to64(torch.cat(ys, 1)), yr, TOL_F32, "chunked")
    assert_close(to64(Sc), Sr, TOL_F32, "chunked S")
    assert_close(to64(Zc), Zr, TOL_F32, "chunked Z")
    assert_close(to64(S), Sr, TOL_F32, "S")


# ---------------------------------------------------------------------------
# a grid of small shapes: several chunks plus a ragged tail, GQA, odd dims

SHAPES = [  # B, T, Hq, Hkv, Dk, Dv
    (1, 1, 2, 2, 64, 64),
    (2, 37, 2, 2, 16, 16),
    (2, 300, 4, 4, 64, 64),
    (1, 257, 8, 2, 128, 128),
    (2, 130, 3, 1, 32, 64),
    (1, 200, 2, 2, 128, 64),
    (1, 129, 4, 2, 64, 128),
    (2, 200, 6, 2, 64, 64),    # GQA, 3 query heads per kv head (two MMA issuers; gated output order)
    (1, 96, 8, 1, 64, 64),     # GQA, 8 query heads per kv head
    (3, 150, 1, 1, 64, 64),    # odd number of (batch, kv head) streams: the last CTA runs one of a pair
]
MODES = [("elu_plus_one", True), ("relu", True), ("elu_plus_one", False), ("none", False)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("mode", MODES, ids=lambda m: f"{m[0]}-{'norm' if m[1] else 'raw'}")
def test_causal_small(shape, dtype, mode):
    B, T, Hq, Hkv, Dk, Dv = shape
    fmap, norm = mode
    std = 0.5 if fmap == "elu_plus_one" else 1.0
    run_case(B, T, Hq, Hkv, Dk, Dv, dtype, torch.float32, fmap, norm, S0=(T % 2 == 0), std=std,
             seed=T + Dk)


@pytest.mark.parametrize("shape", SHAPES[1:5], ids=lambda s: "x".join(map(str, s)))
def test_causal_small_bf16_output(shape):
    B, T, Hq, Hkv, Dk, Dv = shape
    run_case(B, T, Hq, Hkv, Dk, Dv, torch.bfloat16, torch.bfloat16, "elu_plus_one", True, std=0.5)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_gated_small(shape, dtype):
    B, T, Hq, Hkv, Dk, Dv = shape
    run_case(B, T, Hq, Hkv, Dk, Dv, dtype, torch.float32, "none", False, rule="gated", S0=True,
             scale=0.0, seed=7)


@pytest.mark.parametrize("shape", SHAPES + [(1, 192, 32, 2, 64, 64), (2, 129, 16, 1, 128, 128)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gated_small_bf16_output(shape):
    """Gated rule with a bf16 output: the staged 16-byte output stores."""
    B, T, Hq, Hkv, Dk, Dv = shape
    run_case(B, T, Hq, Hkv, Dk, Dv, torch.bfloat16, torch.bfloat16, "none", False, rule="gated", S0=True,
             scale=0.0, seed=9)


@pytest.mark.parametrize("shape", [(2, 200, 4, 2, 64, 64), (1, 257, 8, 2, 128, 128)], ids=lambda s: "x".join(map(str, s)))
def test_gated_strong_decay(shape):
    """Log decay near -5 per token: a 64-token chunk spans several hundred in
    cumulative decay, so the score epilogue takes exp(G_i - G_j) per element
    instead of the factored weights."""
    B, T, Hq, Hkv, Dk, Dv = shape
    run_case(B, T, Hq, Hkv, Dk, Dv, torch.bfloat16, torch.float32, "none", False, rule="gated", S0=True,
             scale=0.0, seed=11, decay_mean=-5.0)


@pytest.mark.parametrize("shape", [(80, 200, 8, 2, 64, 64), (40, 300, 16, 4, 128, 128)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32out", "bf16out"])
def test_gated_grouped_heads_several_chunks_per_cta(shape, out_dtype):
    """At least one CTA per SM without sequence segments, so every CTA walks
    several chunks with four query heads per kv head: the state warps emit
    each chunk's outputs around the next chunk's state conversion."""
    B, T, Hq, Hkv, Dk, Dv = shape
    run_case(B, T, Hq, Hkv, Dk, Dv, torch.bfloat16, out_dtype, "none", False, rule="gated", S0=True, scale=0.0,
             seed=13)


@pytest.mark.parametrize("shape", [(2, 200, 4, 2, 64, 64), (1, 257, 8, 2, 128, 128), (2, 300, 2, 2, 64, 64)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_gated_infinite_decay(shape, dtype):
    """A log decay of -inf forgets everything before its step (ONNX gated:
    S_t = exp(g_t) S_{t-1} + k_t v_t^T with exp(-inf) = 0), inside a chunk,
    on the first and last step of a chunk, and in later sequence segments."""
    B, T, Hq, Hkv, Dk, Dv = shape
    q = rand((B, T, Hq, Dk), 31, dtype)
    k = rand((B, T, Hkv, Dk), 32, dtype)
    v = rand((B, T, Hkv, Dv), 33, dtype)
    x = rand((B, T, Hkv), 34, torch.float32) + 3.0
    g = torch.nn.functional.logsigmoid(x)
    for t, h in [(37, 0), (63, 1 % Hkv), (64, 0), (128, 1 % Hkv), (150, 0), (T - 1, 0)]:
        g[:, t, h] = -float("inf")
    g[1 % B, 100, :] = -float("inf")
    decay = g.to(dtype)
    S0 = rand((B, Hkv, Dk, Dv), 35, torch.float32)
    y, (S, _) = la.la_forward_causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                                     scale=0.0, update_rule="gated", decay=decay, initial_state=(S0, None),
                                     return_state=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    yr, Sr, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                              scale=0.0, rule="gated", decay=decay, S0=S0)
    assert np.isfinite(yr).all() and np.isfinite(Sr).all()
    tol = tol_for(dtype, torch.float32)
    assert_close(to64(y), yr, tol, "y")
    assert_close(to64(S), Sr, tol, "S")



@pytest.mark.parametrize("mode", [("elu_plus_one", True), ("relu", True), ("none", False)],
                         ids=lambda m: f"{m[0]}-{'norm' if m[1] else 'raw'}")
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32out", "bf16out"])
def test_causal_state_pass_sub_segments(mode, out_dtype):
    """Head size 64 with 16 (batch, kv head) streams of 64 chunks: 8 sequence
    segments of 8 chunks, whose state pass (two CTAs per SM) runs as 14
    half-length sub-segments, so that every segment folds two increments per
    earlier segment.  Ragged last chunk, grouped heads, carried initial state
    and the final state, against the oracle."""
    fmap, norm = mode
    run_case(2, 64 * 63 + 37, 16, 8, 64, 64, torch.bfloat16, out_dtype, fmap, norm, S0=True, seed=71,
             std=0.5 if fmap == "elu_plus_one" else 1.0)


def test_causal_one_stream_longest_fold():
    """One (batch, kv head) stream of 601 chunks at head size 64: 151 segments
    of 4 chunks (the last holds one ragged chunk), a state pass of 300
    sub-segments, and a last segment that folds all 300 increments onto the
    carried initial state."""
    run_case(1, 64 * 600 + 17, 2, 1, 64, 64, torch.bfloat16, torch.float32, "elu_plus_one", True, S0=True,
             seed=73, std=0.5)


@pytest.mark.parametrize("shape", SHAPES[1:], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("mode", MODES[:3], ids=lambda m: f"{m[0]}-{'norm' if m[1] else 'raw'}")
def test_noncausal_small(shape, dtype, mode):
    B, T, Hq, Hkv, Dk, Dv = shape
    fmap, norm = mode
    q = rand((B, T, Hq, Dk), 11, dtype, 0.5)
    k = rand((B, T, Hkv, Dk), 12, dtype, 0.5)
    v = rand((B, T, Hkv, Dv), 13, dtype)
    y = la.la_forward_noncausal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap,
                                use_normalizer=norm, out_dtype=torch.float32)
    torch.cuda.synchronize()
    yr = oracle.noncausal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm)
    assert_close(to64(y), yr, tol_for(dtype, torch.float32), "non-causal")


def test_empty_sequence_passes_state_through():
    B, H, D = 2, 2, 64
    q = torch.empty(B, 0, H, D, dtype=torch.bfloat16, device=DEV)
    S0 = rand((B, H, D, D), 1, torch.float32)
    Z0 = rand((B, H, D), 2, torch.float32)
    y, (S, Z) = la.la_forward_causal(q, q, q, q_heads=H, kv_heads=H, initial_state=(S0, Z0),
                                     return_state=True)
    torch.cuda.synchronize()
    assert y.shape == (B, 0, H, D)
    assert torch.equal(S, S0) and torch.equal(Z, Z0)


def test_chunked_equals_full_bf16():
    """Calls with carried state equal one full call (ragged chunk lengths)."""
    B, T, H, D = 2, 700, 4, 64
    q = rand((B, T, H, D), 21, torch.bfloat16, 0.5)
    k = rand((B, T, H, D), 22, torch.bfloat16, 0.5)
    v = rand((B, T, H, D), 23, torch.bfloat16)
    kw = dict(q_heads=H, kv_heads=H, out_dtype=torch.float32)
    y_full, (S_full, Z_full) = la.la_forward_causal(q, k, v, return_state=True, **kw)
    S, Z = la.la_get_initial_state(B, H, D, D)
    ys = []
    for a, b in zip([0, 1, 129, 300, 555], [1, 129, 300, 555, 700]):
        ys.append(la.la_forward_causal(q[:, a:b].contiguous(), k[:, a:b].contiguous(),
                                       v[:, a:b].contiguous(), initial_state=(S, Z), return_state=True,
                                       state_out=(S, Z), **kw)[0])
    torch.cuda.synchronize()
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=H, kv_heads=H)
    assert_close(to64(torch.cat(ys, 1)), yr, 2e-3, "chunked")
    assert_close(to64(y_full), yr, 2e-3, "full")
    assert_close(to64(S), Sr, 2e-3, "chunked S")
    assert_close(to64(Z), Zr, 1e-5, "chunked Z")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("rule", ["linear", "gated"])
def test_decode_steps_small(dtype, rule):
    """Prefill then token-by-token steps equal one causal pass over all tokens."""
    B, T0, steps, Hq, Hkv, D = 3, 40, 9, 4, 2, 64
    fmap, norm = ("elu_plus_one", True) if rule == "linear" else ("none", False)
    T = T0 + steps
    q = rand((B, T, Hq, D), 31, dtype, 0.5)
    k = rand((B, T, Hkv, D), 32, dtype, 0.5)
    v = rand((B, T, Hkv, D), 33, dtype)
    decay = None
    if rule == "gated":
        decay = torch.nn.functional.logsigmoid(rand((B, T, Hkv), 34, torch.float32) + 3.0).to(dtype)
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm, update_rule=rule,
              out_dtype=torch.float32)
    _, (S, Z) = la.la_forward_causal(q[:, :T0].contiguous(), k[:, :T0].contiguous(),
                                     v[:, :T0].contiguous(), return_state=True,
                                     decay=None if decay is None else decay[:, :T0].contiguous(), **kw)
    ys = []
    for t in range(T0, T):
        ys.append(la.la_decode_step(q[:, t:t + 1].contiguous(), k[:, t:t + 1].contiguous(),
                                    v[:, t:t + 1].contiguous(), S, Z,
                                    decay=None if decay is None else decay[:, t:t + 1].contiguous(), **kw))
    torch.cuda.synchronize()
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap,
                               use_normalizer=norm, rule=rule, decay=decay)
    tol = tol_for(dtype, torch.float32)
    assert_close(to64(torch.cat(ys, 1)), yr[:, T0:], tol, "decode y")
    assert_close(to64(S), Sr, tol_for(dtype, torch.float32), "decode S")
    if norm:
        assert_close(to64(Z), Zr, 1e-5, "decode Z")


DECODE_SHAPES = [  # B, Hq, Hkv, Dk, Dv
    (2, 4, 2, 64, 128),   # Dk != Dv
    (1, 8, 1, 128, 32),   # 8 query heads per kv head
    (2, 2, 2, 20, 20),    # rows not a multiple of 16 bytes (bf16): the register-resident kernel
    (3, 3, 3, 12, 12),    # small odd-width rows
]


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_decode_shapes(shape, dtype):
    """Token-by-token steps from a prefilled state equal one causal pass, for
    head sizes and groupings away from the benchmarked ones."""
    B, Hq, Hkv, Dk, Dv = shape
    T0, steps = 17, 5
    T = T0 + steps
    q = rand((B, T, Hq, Dk), 41, dtype, 0.5)
    k = rand((B, T, Hkv, Dk), 42, dtype, 0.5)
    v = rand((B, T, Hkv, Dv), 43, dtype)
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map="elu_plus_one", use_normalizer=True, out_dtype=torch.float32)
    _, (S, Z) = la.la_forward_causal(q[:, :T0].contiguous(), k[:, :T0].contiguous(), v[:, :T0].contiguous(),
                                     return_state=True, **kw)
    ys = [la.la_decode_step(q[:, t:t + 1].contiguous(), k[:, t:t + 1].contiguous(), v[:, t:t + 1].contiguous(),
                            S, Z, **kw) for t in range(T0, T)]
    torch.cuda.synchronize()
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="elu_plus_one", use_normalizer=True)
    tol = tol_for(dtype, torch.float32)
    assert_close(to64(torch.cat(ys, 1)), yr[:, T0:], tol, "decode y")
    assert_close(to64(S), Sr, tol, "decode S")
    assert_close(to64(Z), Zr, 1e-5, "decode Z")


EDGE_SHAPES = [  # B, T, Hq, Hkv, Dk, Dv
    (20, 130, 8, 8, 64, 64),     # 160 (batch, kv head) streams: more CTAs than SMs, no sequence split
    (12, 70, 16, 16, 128, 128),  # 192 streams at head size 128
    (1, 192, 32, 2, 64, 64),     # 16 query heads per kv head; T a multiple of the chunk
    (2, 129, 16, 1, 128, 128),   # 16 query heads on one kv head; one step past a chunk
]


@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("rule", ["linear", "gated"])
def test_edge_shapes(shape, rule):
    B, T, Hq, Hkv, Dk, Dv = shape
    if rule == "linear":
        run_case(B, T, Hq, Hkv, Dk, Dv, torch.bfloat16, torch.bfloat16, "elu_plus_one", True, S0=True, std=0.5,
                 seed=3)
    else:
        run_case(B, T, Hq, Hkv, Dk, Dv, torch.bfloat16, torch.float32, "none", False, rule="gated", S0=True,
                 scale=0.0, seed=4)


def test_invalid_call_raises_and_launches_nothing():
    q = torch.zeros(1, 4, 3, 16, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(1, 4, 2, 16, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(la.LinearAttentionError) as e:
        la.la_forward_causal(q, k, k, q_heads=3, kv_heads=2)
    assert e.value.status == la.LA_ERR_INVALID_ARG


def test_calls_replay_in_a_cuda_graph():
    """The library's calls can be captured into a CUDA graph (the causal pass
    is a programmatic dependent of the segment state pass, an edge the graph
    keeps) and replay bit-identically to eager calls on new inputs."""
    B, T, H, D = 2, 1500, 4, 64  # few streams: a segment state pass and a dependent causal pass
    mk = lambda seed: (rand((B, T, H, D), seed, torch.bfloat16, 0.5), rand((B, T, H, D), seed + 1, torch.bfloat16, 0.5),
                       rand((B, T, H, D), seed + 2, torch.bfloat16))
    q, k, v = mk(81)
    kw = dict(q_heads=H, kv_heads=H)
    p = la.make_params(batch=B, seq_len=T, q_heads=H, kv_heads=H, key_dim=D, value_dim=D)
    ws = torch.empty(max(1, la.la_workspace_bytes(p, True)), dtype=torch.uint8, device=DEV)
    y = torch.empty(B, T, H, D, dtype=torch.bfloat16, device=DEV)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        la.la_forward_causal(q, k, v, out=y, workspace=ws, stream=st, **kw)  # configures the kernels
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    n0 = la.la_launch_count()
    with torch.cuda.graph(g, stream=st, capture_error_mode="relaxed"):
        la.la_forward_causal(q, k, v, out=y, workspace=ws, stream=st, **kw)
    assert la.la_launch_count() - n0 == 2
    q2, k2, v2 = mk(91)
    q.copy_(q2), k.copy_(k2), v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    y_eager = la.la_forward_causal(q2, k2, v2, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert torch.equal(y, y_eager)
    yr, _, _ = oracle.causal(q2, k2, v2, q_heads=H, kv_heads=H)
    assert_close(to64(y), yr, tol_for(torch.bfloat16, torch.bfloat16), "graph replay")


def test_bounded_wait_gives_up_and_reports():
    """Failure path of the bounded waits (no GPU fault): both wait forms poll
    a barrier nothing completes, give up after 2 ms, set their bits in the
    device error word and return; the context stays usable afterwards."""
    assert la.la_device_error(reset=True) == 0
    la.la_check_bounded_wait(2000)
    assert la.la_device_status(reset=False) == la.LA_ERR_TIMEOUT
    word = la.la_device_error(reset=True)
    assert word == la.LA_SELFTEST_WARP_WAIT | la.LA_SELFTEST_THREAD_WAIT, hex(word)
    assert la.la_device_status(reset=False) == la.LA_OK
    # the context still runs the library's kernels correctly
    run_case(2, 130, 4, 2, 64, 64, torch.bfloat16, torch.float32, "elu_plus_one", True, std=0.5)
    assert la.la_device_error(reset=False) == 0


def test_noncausal_more_streams_than_a_grid_row():
    """More (batch, kv head) streams than gridDim.y allows (65535): every
    kernel of the non-causal path takes the stream index from gridDim.x."""
    B, T, H, D = 65540, 3, 1, 64
    q = rand((B, T, H, D), 41, torch.bfloat16, 0.5)
    k = rand((B, T, H, D), 42, torch.bfloat16, 0.5)
    v = rand((B, T, H, D), 43, torch.bfloat16)
    y = la.la_forward_noncausal(q, k, v, q_heads=H, kv_heads=H, out_dtype=torch.float32)
    torch.cuda.synchronize()
    yr = oracle.noncausal(q, k, v, q_heads=H, kv_heads=H)
    assert_close(to64(y), yr, tol_for(torch.bfloat16, torch.float32), "non-causal")
