"""GPU parity of the backward pass of the causal linear rule: the library's
dq, dk, dv (and the initial state's gradients) against float64 autograd of
the plain recurrence in oracle/grad.py (itself pinned to finite
differences, as the Keras request's Test Plan asks)."""
import pytest
import torch

import kernelized_linear_attention_02_gb300 as la
import linattn_inputs as inputs
from parity_utils import assert_close, to64
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
    tol = 2e-5
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
    tol = 2e-5 + 2.0 ** -8  # the bf16 rounding of the gradients themselves
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
    tol = 2e-5
    assert_close(to64(dq), rq.numpy(), tol, "dq")
    assert_close(to64(dk), rk.numpy(), tol, "dk")
    assert_close(to64(dv), rv.numpy(), tol, "dv")
    assert_close(to64(dS0), rS0.numpy(), tol, "dS0")
    if norm:
        assert_close(to64(dZ0), rZ0.numpy(), tol, "dZ0")
