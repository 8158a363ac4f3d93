"""GPU parity of the backward pass of the causal linear rule: the library's
dq, dk, dv (and the initial state's gradients) against float64 autograd of
the plain recurrence in oracle/grad.py (itself pinned to finite
differences, as the Keras request's Test Plan asks).

bf16 inputs with Dk = Dv in {64, 128} run the chunk-parallel tensor-core
form (five launches) and are held to the bf16-input bar, 2e-3; every other
shape and float32 inputs run the CUDA-core scans, held to 2e-5."""
import pytest
import torch

import kernelized_linear_attention_02_gb300 as la
import linattn_inputs as inputs
from parity_utils import TOL_BF16, assert_close, rel_err, to64
from oracle import grad as og

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
    assert la.la_device_error(reset=True) == 0


def rand(shape, seed, dtype, std=1.0):
    g = inputs.generator(seed, DEV)
    return inputs.normal(shape, g, std, dtype=dtype, device=DEV)


def tensor_core_form(dtype, Dk, Dv):
    return dtype == torch.bfloat16 and Dk == Dv and Dk in (64, 128)


def bwd_tol(dtype, Dk, Dv, grad_dtype=torch.float32):
    """2e-3 for the bf16 tensor-core form (bf16 products of hi + lo splits,
    fp32 accumulation), 2e-5 for the fp32 CUDA-core scans; plus the rounding
    of bf16 gradients themselves (2^-8 of every element)."""
    tol = TOL_BF16 if tensor_core_form(dtype, Dk, Dv) else 2e-5
    return tol + (2.0 ** -8 if grad_dtype == torch.bfloat16 else 0.0)


SHAPES = [  # B, T, Hq, Hkv, Dk, Dv
    (2, 37, 2, 2, 16, 16),
    (1, 70, 4, 2, 64, 64),
    (2, 45, 3, 1, 32, 48),
    (1, 33, 2, 2, 128, 128),
    (1, 20, 16, 1, 64, 32),
]
MODES = [("elu_plus_one", True), ("relu", True), ("none", False), ("elu_plus_one", False)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", MODES, ids=lambda m: f"{m[0]}-{'norm' if m[1] else 'raw'}")
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_backward_matches_autograd(shape, mode, dtype):
    B, T, Hq, Hkv, Dk, Dv = shape
    fmap, norm = mode
    std = 0.5 if fmap == "elu_plus_one" else 1.0
    q = rand((B, T, Hq, Dk), 1, dtype, std)
    k = rand((B, T, Hkv, Dk), 2, dtype, std)
    v = rand((B, T, Hkv, Dv), 3, dtype)
    dy = rand((B, T, Hq, Dv), 4, dtype)
    S0 = rand((B, Hkv, Dk, Dv), 5, torch.float32)
    Z0 = rand((B, Hkv, Dk), 6, torch.float32).abs() + 1.0 if norm else None
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm, scale=0.8)
    dq, dk, dv, dS0, dZ0 = la.la_backward_causal(q, k, v, dy, initial_state=(S0, Z0), return_state_grad=True,
                                                 epsilon=1e-3, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, rS0, rZ0 = og.causal_backward(q, k, v, dy, S0=S0, Z0=Z0, eps=1e-3, **kw)
    tol = bwd_tol(dtype, Dk, Dv)
    assert_close(to64(dq), rq.numpy(), tol, "dq")
    assert_close(to64(dk), rk.numpy(), tol, "dk")
    assert_close(to64(dv), rv.numpy(), tol, "dv")
    assert_close(to64(dS0), rS0.numpy(), tol, "dS0")
    if norm:
        assert_close(to64(dZ0), rZ0.numpy(), tol, "dZ0")


def test_backward_without_initial_state_bf16_grads():
    B, T, H, D = 2, 150, 4, 64
    q = rand((B, T, H, D), 11, torch.bfloat16, 0.5)
    k = rand((B, T, H, D), 12, torch.bfloat16, 0.5)
    v = rand((B, T, H, D), 13, torch.bfloat16)
    dy = rand((B, T, H, D), 14, torch.bfloat16)
    dq, dk, dv = la.la_backward_causal(q, k, v, dy, q_heads=H, kv_heads=H, grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    rq, rk, rv, _, _ = og.causal_backward(q, k, v, dy, q_heads=H, kv_heads=H)
    tol = bwd_tol(torch.bfloat16, D, D, torch.bfloat16)
    assert_close(to64(dq), rq.numpy(), tol, "dq")
    assert_close(to64(dk), rk.numpy(), tol, "dk")
    assert_close(to64(dv), rv.numpy(), tol, "dv")


def test_backward_rejects_other_rules():
    p = la.make_params(batch=1, seq_len=4, q_heads=2, kv_heads=2, key_dim=16, value_dim=16, feature_map="none",
                       use_normalizer=False, update_rule="gated")
    import ctypes
    d = ctypes.c_void_p(256)
    assert la.lib().la_backward_causal(ctypes.byref(p), d, d, d, None, None, d, d, d, d, None, None, d, 1 << 20,
                                       None) == la.LA_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape", [(1, 1500, 2, 2, 64, 64), (2, 1100, 4, 2, 32, 48), (1, 800, 3, 1, 128, 128)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", [("elu_plus_one", True), ("relu", False)], ids=["elu-norm", "relu-raw"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_backward_sequence_segments(shape, mode, dtype):
    """Long sequences with few streams: both scans run over sequence
    segments, folded from the other segments' increments."""
    B, T, Hq, Hkv, Dk, Dv = shape
    fmap, norm = mode
    std = 0.5 if fmap == "elu_plus_one" else 1.0
    q = rand((B, T, Hq, Dk), 21, dtype, std)
    k = rand((B, T, Hkv, Dk), 22, dtype, std)
    v = rand((B, T, Hkv, Dv), 23, dtype)
    dy = rand((B, T, Hq, Dv), 24, dtype)
    S0 = rand((B, Hkv, Dk, Dv), 25, torch.float32)
    Z0 = rand((B, Hkv, Dk), 26, torch.float32).abs() + 1.0 if norm else None
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm)
    dq, dk, dv, dS0, dZ0 = la.la_backward_causal(q, k, v, dy, initial_state=(S0, Z0), return_state_grad=True, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, rS0, rZ0 = og.causal_backward(q, k, v, dy, S0=S0, Z0=Z0, **kw)
    tol = bwd_tol(dtype, Dk, Dv)
    assert_close(to64(dq), rq.numpy(), tol, "dq")
    assert_close(to64(dk), rk.numpy(), tol, "dk")
    assert_close(to64(dv), rv.numpy(), tol, "dv")
    assert_close(to64(dS0), rS0.numpy(), tol, "dS0")
    if norm:
        assert_close(to64(dZ0), rZ0.numpy(), tol, "dZ0")


TC_SHAPES = [  # B, T, Hq, Hkv, D: several chunks, ragged tails, grouped heads
    (2, 200, 4, 2, 64),
    (1, 130, 8, 2, 128),
    (3, 64, 2, 2, 64),
    (1, 1, 2, 1, 128),
    (2, 333, 6, 3, 64),
    (1, 257, 3, 1, 128),
]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", MODES, ids=lambda m: f"{m[0]}-{'norm' if m[1] else 'raw'}")
def test_backward_tensor_core_form(shape, mode):
    """The chunk-parallel tensor-core backward (five launches) against float64
    autograd, with a carried initial state and an output scale."""
    B, T, Hq, Hkv, D = shape
    fmap, norm = mode
    std = 0.5 if fmap == "elu_plus_one" else 1.0
    dt = torch.bfloat16
    q = rand((B, T, Hq, D), 31, dt, std)
    k = rand((B, T, Hkv, D), 32, dt, std)
    v = rand((B, T, Hkv, D), 33, dt)
    dy = rand((B, T, Hq, D), 34, dt)
    S0 = rand((B, Hkv, D, D), 35, torch.float32)
    Z0 = rand((B, Hkv, D), 36, torch.float32).abs() + 1.0 if norm else None
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm, scale=0.7)
    n0 = la.la_launch_count()
    dq, dk, dv, dS0, dZ0 = la.la_backward_causal(q, k, v, dy, initial_state=(S0, Z0), return_state_grad=True, **kw)
    torch.cuda.synchronize()
    assert la.la_launch_count() - n0 == 5
    rq, rk, rv, rS0, rZ0 = og.causal_backward(q, k, v, dy, S0=S0, Z0=Z0, **kw)
    tol = bwd_tol(dt, D, D)
    assert_close(to64(dq), rq.numpy(), tol, "dq")
    assert_close(to64(dk), rk.numpy(), tol, "dk")
    assert_close(to64(dv), rv.numpy(), tol, "dv")
    assert_close(to64(dS0), rS0.numpy(), tol, "dS0")
    if norm:
        assert_close(to64(dZ0), rZ0.numpy(), tol, "dZ0")


NEAR_ZERO = [  # feature map, query mean, query std
    ("relu", -3.0, 1.0),       # phi(q) = eps in almost every dimension
    ("relu", -1.5, 1.0),
    ("elu_plus_one", -6.0, 0.5),  # phi(q) = e^q ~ 2.5e-3 everywhere
]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("case", NEAR_ZERO, ids=lambda c: f"{c[0]}{c[1]:+g}")
def test_backward_tensor_core_near_zero_denominator(D, case):
    """Queries drawn far below zero: phi(q) is small, the denominator sits near
    its eps floor and ds = dy / den is large (Keras request, Test Plan,
    Stability: near-zero denominators).

    With relu + eps at mean -3 most queries have one or two active feature
    dimensions; along such a dimension the output is a weighted mean that does
    not depend on the query's size, so d a there is a sum of large terms that
    cancel to O(eps).  That row-wise value is ill-conditioned for any float32
    evaluation (rounding the scores to float32 alone moves such rows by more
    than the bar), so in that case dq is held to the norm-wise bar and dk, dv
    to both bars; every other case is held to both bars throughout."""
    fmap, mu, sd = case
    B, T, H = 1, 150, 2
    dt = torch.bfloat16
    q = (rand((B, T, H, D), 41, torch.float32) * sd + mu).to(dt)
    k = rand((B, T, H, D), 42, dt, 0.5 if fmap == "elu_plus_one" else 1.0)
    v = rand((B, T, H, D), 43, dt)
    dy = rand((B, T, H, D), 44, dt)
    kw = dict(q_heads=H, kv_heads=H, feature_map=fmap, use_normalizer=True)
    dq, dk, dv = la.la_backward_causal(q, k, v, dy, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, _, _ = og.causal_backward(q, k, v, dy, **kw)
    tol = bwd_tol(dt, D, D)
    if fmap == "relu" and mu <= -3.0:
        assert rel_err(to64(dq), rq.numpy()) <= tol
    else:
        assert_close(to64(dq), rq.numpy(), tol, "dq")
    assert_close(to64(dk), rk.numpy(), tol, "dk")
    assert_close(to64(dv), rv.numpy(), tol, "dv")


def test_backward_tensor_core_bf16_grads_in_place_of_fp32():
    """bf16 gradients from the tensor-core form: the fp32 result rounded once."""
    B, T, Hq, Hkv, D = 2, 180, 4, 2, 128
    dt = torch.bfloat16
    q = rand((B, T, Hq, D), 51, dt, 0.5)
    k = rand((B, T, Hkv, D), 52, dt, 0.5)
    v = rand((B, T, Hkv, D), 53, dt)
    dy = rand((B, T, Hq, D), 54, dt)
    kw = dict(q_heads=Hq, kv_heads=Hkv)
    dq, dk, dv = la.la_backward_causal(q, k, v, dy, grad_dtype=torch.bfloat16, **kw)
    torch.cuda.synchronize()
    rq, rk, rv, _, _ = og.causal_backward(q, k, v, dy, **kw)
    tol = bwd_tol(dt, D, D, torch.bfloat16)
    assert_close(to64(dq), rq.numpy(), tol, "dq")
    assert_close(to64(dk), rk.numpy(), tol, "dk")
    assert_close(to64(dv), rv.numpy(), tol, "dv")


def test_backward_workload_sampled():
    """The 2k prefill workload (B=4, T=2048, 8 heads, D=64, elu + 1 with the
    normalizer) in the launch configuration the benchmark times; batch row 0,
    kv heads 0 and 1 (independent streams) against the oracle over all 2048
    steps."""
    w = inputs.PREFILL_2K
    q, k, v, _ = inputs.make_qkv(w, device=DEV, seed=w.seed)
    dy = inputs.normal((w.B, w.T, w.q_heads, w.Dv), inputs.generator(w.seed + 1, DEV), 1.0, dtype=w.dtype,
                       device=DEV)
    kw = dict(q_heads=w.q_heads, kv_heads=w.kv_heads, feature_map=w.feature_map, use_normalizer=w.use_normalizer,
              epsilon=w.eps, scale=w.scale)
    dq, dk, dv = la.la_backward_causal(q, k, v, dy, **kw)
    torch.cuda.synchronize()
    G = w.q_heads // w.kv_heads
    sq = slice(0, 2 * G)
    skv = slice(0, 2)
    rq, rk, rv, _, _ = og.causal_backward(q[:1, :, sq], k[:1, :, skv], v[:1, :, skv], dy[:1, :, sq], q_heads=2 * G,
                                          kv_heads=2, feature_map=w.feature_map, use_normalizer=w.use_normalizer,
                                          eps=w.eps, scale=w.scale)
    tol = bwd_tol(w.dtype, w.Dk, w.Dv)
    assert_close(to64(dq[:1, :, sq]), rq.numpy(), tol, "dq")
    assert_close(to64(dk[:1, :, skv]), rk.numpy(), tol, "dk")
    assert_close(to64(dv[:1, :, skv]), rv.numpy(), tol, "dv")
