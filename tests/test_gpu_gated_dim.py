"""GPU parity of the gated rule with one log decay per key dimension
(ONNX-light "LinearAttention", decay of shape (B, T, H_kv*d_k): row i of the
state is scaled by exp(g_t[i]) at step t).  The library runs it on the
CUDA-core recurrence and in the decode kernels; the oracle takes the same
decay layout."""
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
    assert la.la_device_error(reset=True) == 0


def rand(shape, seed, dtype, std=1.0, mean=0.0):
    g = inputs.generator(seed, DEV)
    return inputs.normal(shape, g, std, mean=mean, dtype=dtype, device=DEV)


def perdim_decay(B, T, Hkv, Dk, seed, dtype, mean=3.0):
    return torch.nn.functional.logsigmoid(rand((B, T, Hkv, Dk), seed, torch.float32, mean=mean)).to(dtype)


SHAPES = [  # B, T, Hq, Hkv, Dk, Dv
    (2, 37, 2, 2, 16, 16),
    (2, 300, 4, 4, 64, 64),
    (1, 257, 8, 2, 128, 128),
    (2, 130, 3, 1, 32, 64),
    (1, 129, 4, 2, 64, 128),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("mean", [3.0, -1.0], ids=["mild", "strong"])
def test_gated_per_key_dim(shape, dtype, mean):
    B, T, Hq, Hkv, Dk, Dv = shape
    q = rand((B, T, Hq, Dk), 1, dtype)
    k = rand((B, T, Hkv, Dk), 2, dtype)
    v = rand((B, T, Hkv, Dv), 3, dtype)
    d = perdim_decay(B, T, Hkv, Dk, 4, dtype, mean)
    S0 = rand((B, Hkv, Dk, Dv), 5, torch.float32)
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, scale=0.0, update_rule="gated")
    y, (S, _) = la.la_forward_causal(q, k, v, decay=d, initial_state=(S0, None), return_state=True,
                                     out_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    yr, Sr, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                              scale=0.0, rule="gated", decay=d.reshape(B, T, Hkv * Dk), S0=S0)
    tol = tol_for(dtype, torch.float32)
    assert_close(to64(y), yr, tol, "y")
    assert_close(to64(S), Sr, tol, "S")


def test_per_key_dim_equal_rows_is_the_per_head_rule():
    """A per-dimension decay that is equal across the key dimensions gives the
    per-head result (the tensor-core path) within the bf16 tolerance."""
    B, T, H, D = 2, 300, 4, 64
    q = rand((B, T, H, D), 11, torch.bfloat16)
    k = rand((B, T, H, D), 12, torch.bfloat16)
    v = rand((B, T, H, D), 13, torch.bfloat16)
    dh = torch.nn.functional.logsigmoid(rand((B, T, H), 14, torch.float32, mean=3.0)).to(torch.bfloat16)
    dd = dh[..., None].expand(B, T, H, D).contiguous()
    kw = dict(q_heads=H, kv_heads=H, feature_map="none", use_normalizer=False, update_rule="gated",
              out_dtype=torch.float32)
    yh = la.la_forward_causal(q, k, v, decay=dh, **kw)
    yd = la.la_forward_causal(q, k, v, decay=dd, **kw)
    torch.cuda.synchronize()
    yr, _, _ = oracle.causal(q, k, v, q_heads=H, kv_heads=H, feature_map="none", use_normalizer=False,
                             rule="gated", decay=dh)
    assert_close(to64(yh), yr, 2e-3, "per head")
    assert_close(to64(yd), yr, 2e-3, "per dim")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_per_key_dim_decode_steps(dtype):
    B, T0, steps, Hq, Hkv, D = 3, 30, 6, 4, 2, 64
    T = T0 + steps
    q = rand((B, T, Hq, D), 21, dtype)
    k = rand((B, T, Hkv, D), 22, dtype)
    v = rand((B, T, Hkv, D), 23, dtype)
    d = perdim_decay(B, T, Hkv, D, 24, dtype)
    mask = inputs.validity_mask("random", B, T, 25, DEV)
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, update_rule="gated",
              out_dtype=torch.float32)
    c = lambda x, a, b: x[:, a:b].contiguous()
    _, (S, _) = la.la_forward_causal(c(q, 0, T0), c(k, 0, T0), c(v, 0, T0), decay=c(d, 0, T0), return_state=True,
                                     mask=c(mask, 0, T0), **kw)
    ys = [la.la_decode_step(c(q, t, t + 1), c(k, t, t + 1), c(v, t, t + 1), S, None, decay=c(d, t, t + 1),
                            mask=c(mask, t, t + 1), **kw) for t in range(T0, T)]
    torch.cuda.synchronize()
    yr, Sr, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                              rule="gated", decay=d.reshape(B, T, Hkv * D), mask=mask)
    tol = tol_for(dtype, torch.float32)
    assert_close(to64(torch.cat(ys, 1)), yr[:, T0:], tol, "decode y")
    assert_close(to64(S), Sr, tol, "decode S")


def test_per_key_dim_workload_sampled_slices():
    """The measured per-dimension workload at full size: sampled (batch, kv
    head) streams against the oracle."""
    w = inputs.GATED_PERDIM
    q, k, v, d = inputs.make_qkv(w, device=DEV)
    kw = dict(q_heads=w.q_heads, kv_heads=w.kv_heads, feature_map=w.feature_map, use_normalizer=w.use_normalizer,
              epsilon=w.eps, scale=w.scale, update_rule=w.rule)
    y = la.la_forward_causal(q, k, v, decay=d, **kw)
    torch.cuda.synchronize()
    G = w.q_heads // w.kv_heads
    for b, hk in [(0, 0), (1, 5)]:
        yr, _, _ = oracle.causal(q[b:b + 1, :, hk * G:(hk + 1) * G], k[b:b + 1, :, hk:hk + 1], v[b:b + 1, :, hk:hk + 1],
                                 q_heads=G, kv_heads=1, feature_map=w.feature_map, use_normalizer=w.use_normalizer,
                                 scale=w.scale, rule="gated", decay=d[b:b + 1, :, hk:hk + 1].reshape(1, w.T, w.Dk))
        assert_close(to64(y[b:b + 1, :, hk * G:(hk + 1) * G]), yr, tol_for(w.dtype, w.dtype), f"slice {b},{hk}")


# ---------------------------------------------------------------------------
# the chunk-parallel tensor-core form (bf16, Dk = Dv = 128)

TC_SHAPES = [  # B, T, Hq, Hkv
    (2, 300, 4, 2),
    (1, 257, 3, 1),
    (3, 130, 1, 1),
    (1, 640, 8, 1),
]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mean", [3.0, -1.0, -4.0], ids=["mild", "strong", "very-strong"])
@pytest.mark.parametrize("masked", [False, True], ids=["nomask", "mask"])
def test_per_key_dim_tensor_core_form(shape, mean, masked):
    """Mild decays factor in every chunk; strong ones (cumulative decay below
    -80 inside a chunk) make those chunks compute their scores on CUDA cores."""
    B, T, Hq, Hkv = shape
    D = 128
    q = rand((B, T, Hq, D), 31, torch.bfloat16)
    k = rand((B, T, Hkv, D), 32, torch.bfloat16)
    v = rand((B, T, Hkv, D), 33, torch.bfloat16)
    d = perdim_decay(B, T, Hkv, D, 34, torch.bfloat16, mean)
    S0 = rand((B, Hkv, D, D), 35, torch.float32)
    mask = inputs.validity_mask("gaps", B, T, 36, DEV) if masked else None
    p = la.make_params(batch=B, seq_len=T, q_heads=Hq, kv_heads=Hkv, key_dim=D, value_dim=D, feature_map="none",
                       use_normalizer=False, update_rule="gated", decay_per_key_dim=True)
    assert la.la_workspace_bytes(p, True) > 0
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, scale=0.0, update_rule="gated")
    n0 = la.la_launch_count()
    y, (S, _) = la.la_forward_causal(q, k, v, decay=d, initial_state=(S0, None), return_state=True, mask=mask,
                                     out_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    assert la.la_launch_count() - n0 == 3  # prep, scan, out
    yr, Sr, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                              scale=0.0, rule="gated", decay=d.reshape(B, T, Hkv * D), S0=S0, mask=mask)
    tol = tol_for(torch.bfloat16, torch.float32)
    assert_close(to64(y), yr, tol, "y")
    assert_close(to64(S), Sr, tol, "S")
    if masked:
        assert torch.count_nonzero(y[~mask]).item() == 0


def test_per_key_dim_tensor_core_form_bf16_out_chunked_in_place():
    """bf16 output, and calls over consecutive pieces with the state carried
    in place equal one call."""
    B, T, Hq, Hkv, D = 2, 500, 4, 2, 128
    q = rand((B, T, Hq, D), 41, torch.bfloat16)
    k = rand((B, T, Hkv, D), 42, torch.bfloat16)
    v = rand((B, T, Hkv, D), 43, torch.bfloat16)
    d = perdim_decay(B, T, Hkv, D, 44, torch.bfloat16)
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, update_rule="gated",
              out_dtype=torch.bfloat16)
    S = torch.zeros(B, Hkv, D, D, device=DEV)
    ys = []
    for a0, a1 in [(0, 64), (64, 199), (199, 500)]:
        c = lambda x: x[:, a0:a1].contiguous()
        ys.append(la.la_forward_causal(c(q), c(k), c(v), decay=c(d), initial_state=(S, None), return_state=True,
                                       state_out=(S, None), **kw)[0])
    torch.cuda.synchronize()
    yr, Sr, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                              rule="gated", decay=d.reshape(B, T, Hkv * D))
    assert_close(to64(torch.cat(ys, 1)), yr, tol_for(torch.bfloat16, torch.bfloat16), "chunked y")
    assert_close(to64(S), Sr, tol_for(torch.bfloat16, torch.float32), "chunked S")
