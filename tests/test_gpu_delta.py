"""GPU parity of the delta rules of the ONNX-light "LinearAttention" operator
(update_rule "delta" and "gated_delta":
S_t = exp(g_t) S_{t-1} + beta_t k_t (x) (v_t - exp(g_t) S_{t-1}^T k_t)), and
every worked example of that page run through the CUDA library itself.

The page's printed outputs and present states are the reference for the
examples; random cases are compared with the CPU oracle.  Keys are
L2-normalised over d_k, as the page recommends for the delta rules."""
import json
import os

import numpy as np
import pytest
import torch

import kernelized_linear_attention_02_gb300 as la
import linattn_inputs as inputs
from parity_utils import assert_close, to64, tol_for
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "onnx_linear_attention_examples.json")


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


EXAMPLES = json.load(open(GOLDEN))["examples"]


@pytest.mark.parametrize("name", sorted(EXAMPLES))
def test_onnx_worked_example_on_gpu(name):
    """Every worked example of the ONNX page, all four update rules, through
    the library's entry points (float32; the float16 example's inputs widened
    exactly and held to the same fp16 bound as the oracle pin)."""
    e = EXAMPLES[name]
    dt = np.float16 if e.get("dtype") == "float16" else np.float32
    f = lambda key: None if key not in e else torch.tensor(np.array(e[key], dtype=dt).astype(np.float32),
                                                          device=DEV).contiguous()
    q, k, v = f("query"), f("key"), f("value")
    Hq, Hkv = e["q_num_heads"], e["kv_num_heads"]
    rule = e["update_rule"]
    S0 = f("past_state")
    y, (S, _) = la.la_forward_causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                                     scale=e.get("scale", 0.0), update_rule=rule, decay=f("decay"), beta=f("beta"),
                                     initial_state=None if S0 is None else (S0, None), return_state=True,
                                     out_dtype=torch.float32)
    torch.cuda.synchronize()
    fp16 = e.get("dtype") == "float16"
    atol, rtol = (4e-3, 2e-3) if fp16 else (1e-5, 1e-5)
    y_ref = np.array(e["output"], dtype=np.float64).reshape(y.shape)
    np.testing.assert_allclose(to64(y), y_ref, rtol=rtol, atol=atol, err_msg=name + " output")
    np.testing.assert_allclose(to64(S), np.array(e["present_state"], dtype=np.float64), rtol=rtol, atol=atol,
                               err_msg=name + " state")


def rand(shape, seed, dtype, std=1.0, mean=0.0):
    g = inputs.generator(seed, DEV)
    return inputs.normal(shape, g, std, mean=mean, dtype=dtype, device=DEV)


def delta_inputs(B, T, Hq, Hkv, Dk, Dv, dtype, rule, per_dim, beta_heads, seed):
    q = rand((B, T, Hq, Dk), seed, dtype)
    k32 = rand((B, T, Hkv, Dk), seed + 1, torch.float32)
    k = (k32 / k32.norm(dim=-1, keepdim=True)).to(dtype)
    v = rand((B, T, Hkv, Dv), seed + 2, dtype)
    beta = torch.sigmoid(rand((B, T, beta_heads), seed + 3, torch.float32)).to(dtype)
    decay = None
    if rule == "gated_delta":
        shape = (B, T, Hkv, Dk) if per_dim else (B, T, Hkv)
        decay = torch.nn.functional.logsigmoid(rand(shape, seed + 4, torch.float32, mean=3.0)).to(dtype)
    return q, k, v, beta, decay


CASES = [  # B, T, Hq, Hkv, Dk, Dv, rule, decay per key dim, beta heads (Hkv or 1)
    (2, 37, 2, 2, 16, 16, "delta", False, 2),
    (2, 300, 4, 2, 64, 64, "gated_delta", False, 2),
    (1, 257, 8, 2, 128, 128, "gated_delta", True, 2),
    (3, 130, 3, 1, 32, 64, "delta", False, 1),
    (2, 200, 4, 4, 64, 128, "gated_delta", False, 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + f"-{c[6]}{'-dim' if c[7] else ''}-b{c[8]}")
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("masked", [False, True], ids=["nomask", "mask"])
def test_delta_rules(case, dtype, masked):
    B, T, Hq, Hkv, Dk, Dv, rule, per_dim, bh = case
    q, k, v, beta, decay = delta_inputs(B, T, Hq, Hkv, Dk, Dv, dtype, rule, per_dim, bh, 11)
    S0 = rand((B, Hkv, Dk, Dv), 15, torch.float32)
    mask = inputs.validity_mask("gaps", B, T, 16, DEV) if masked else None
    y, (S, _) = la.la_forward_causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                                     scale=0.0, update_rule=rule, decay=decay, beta=beta, initial_state=(S0, None),
                                     return_state=True, out_dtype=torch.float32, mask=mask)
    torch.cuda.synchronize()
    d_or = None if decay is None else (decay.reshape(B, T, Hkv * Dk) if per_dim else decay)
    yr, Sr, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, scale=0.0,
                              rule=rule, decay=d_or, beta=beta, S0=S0, mask=mask)
    tol = tol_for(dtype, torch.float32)
    assert_close(to64(y), yr, tol, "y")
    assert_close(to64(S), Sr, tol, "S")
    if masked:
        assert torch.count_nonzero(y[~mask]).item() == 0


@pytest.mark.parametrize("rule", ["delta", "gated_delta"])
def test_delta_decode_steps_equal_one_pass(rule):
    B, T0, steps, Hq, Hkv, D = 3, 20, 6, 4, 2, 64
    T = T0 + steps
    q, k, v, beta, decay = delta_inputs(B, T, Hq, Hkv, D, D, torch.float32, rule, False, Hkv, 21)
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, update_rule=rule,
              out_dtype=torch.float32)
    c = lambda x, a, b: None if x is None else x[:, a:b].contiguous()
    _, (S, _) = la.la_forward_causal(c(q, 0, T0), c(k, 0, T0), c(v, 0, T0), decay=c(decay, 0, T0),
                                     beta=c(beta, 0, T0), return_state=True, **kw)
    ys = [la.la_decode_step(c(q, t, t + 1), c(k, t, t + 1), c(v, t, t + 1), S, None, decay=c(decay, t, t + 1),
                            beta=c(beta, t, t + 1), **kw) for t in range(T0, T)]
    torch.cuda.synchronize()
    yr, Sr, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, rule=rule,
                              decay=decay, beta=beta)
    assert_close(to64(torch.cat(ys, 1)), yr[:, T0:], 1e-5, "decode y")
    assert_close(to64(S), Sr, 1e-5, "decode S")


def test_delta_argument_checks():
    q = torch.zeros(1, 4, 2, 16, device=DEV)
    with pytest.raises(ValueError):  # beta missing
        la.la_forward_causal(q, q, q, q_heads=2, kv_heads=2, feature_map="none", use_normalizer=False,
                             update_rule="delta")
    with pytest.raises(la.LinearAttentionError):  # a feature map is not defined for the delta rules
        la.la_forward_causal(q, q, q, q_heads=2, kv_heads=2, feature_map="elu_plus_one", use_normalizer=False,
                             update_rule="delta", beta=torch.ones(1, 4, 2, device=DEV))
    with pytest.raises(la.LinearAttentionError):  # gated_delta without decay
        la.la_forward_causal(q, q, q, q_heads=2, kv_heads=2, feature_map="none", use_normalizer=False,
                             update_rule="gated_delta", beta=torch.ones(1, 4, 2, device=DEV))


def test_gated_delta_workload_sampled_slices():
    """The measured gated_delta workload at full size (the launch the
    benchmark times): sampled (batch, kv head) streams against the oracle."""
    w = inputs.GATED_DELTA
    q, k, v, d = inputs.make_qkv(w, device=DEV)
    beta = inputs.make_beta(w, DEV)
    y = la.la_forward_causal(q, k, v, q_heads=w.q_heads, kv_heads=w.kv_heads, feature_map=w.feature_map,
                             use_normalizer=w.use_normalizer, epsilon=w.eps, scale=w.scale, update_rule=w.rule,
                             decay=d, beta=beta)
    torch.cuda.synchronize()
    G = w.q_heads // w.kv_heads
    for b, hk in [(0, 3), (1, 6)]:
        yr, _, _ = oracle.causal(q[b:b + 1, :, hk * G:(hk + 1) * G], k[b:b + 1, :, hk:hk + 1], v[b:b + 1, :, hk:hk + 1],
                                 q_heads=G, kv_heads=1, feature_map=w.feature_map, use_normalizer=w.use_normalizer,
                                 scale=w.scale, rule=w.rule, decay=d[b:b + 1, :, hk:hk + 1],
                                 beta=beta[b:b + 1, :, hk:hk + 1])
        assert_close(to64(y[b:b + 1, :, hk * G:(hk + 1) * G]), yr, tol_for(w.dtype, w.dtype), f"slice {b},{hk}")


# ---------------------------------------------------------------------------
# the chunk-parallel (WY) tensor-core form: bf16, Dk = Dv = 128, decay per kv head

TC_CASES = [  # B, T, Hq, Hkv, rule, beta heads (Hkv or 1)
    (2, 300, 4, 2, "gated_delta", 2),
    (1, 257, 6, 2, "delta", 1),
    (3, 130, 3, 1, "gated_delta", 1),
    (1, 64, 1, 1, "delta", 1),
    (2, 1000, 8, 8, "gated_delta", 8),
    (1, 513, 2, 1, "gated_delta", 1),
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: "x".join(map(str, c[:4])) + f"-{c[4]}-b{c[5]}")
@pytest.mark.parametrize("masked", [False, True], ids=["nomask", "mask"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32out", "bf16out"])
def test_delta_tensor_core_form(case, masked, out_dtype):
    B, T, Hq, Hkv, rule, bh = case
    D = 128
    q, k, v, beta, decay = delta_inputs(B, T, Hq, Hkv, D, D, torch.bfloat16, rule, False, bh, 31)
    S0 = rand((B, Hkv, D, D), 35, torch.float32)
    mask = inputs.validity_mask("gaps", B, T, 36, DEV) if masked else None
    p = la.make_params(batch=B, seq_len=T, q_heads=Hq, kv_heads=Hkv, key_dim=D, value_dim=D, feature_map="none",
                       use_normalizer=False, update_rule=rule)
    assert la.la_delta_workspace_bytes(p) > 0  # this shape takes the tensor-core form
    n0 = la.la_launch_count()
    y, (S, _) = la.la_forward_causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                                     scale=0.0, update_rule=rule, decay=decay, beta=beta, initial_state=(S0, None),
                                     return_state=True, out_dtype=out_dtype, mask=mask)
    torch.cuda.synchronize()
    assert la.la_launch_count() - n0 == 3  # prep, scan, out
    yr, Sr, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, scale=0.0,
                              rule=rule, decay=decay, beta=beta, S0=S0, mask=mask)
    assert_close(to64(y), yr, tol_for(torch.bfloat16, out_dtype), "y")
    assert_close(to64(S), Sr, tol_for(torch.bfloat16, torch.float32), "S")
    if masked:
        assert torch.count_nonzero(y[~mask]).item() == 0


def test_delta_tensor_core_form_in_place_state_and_restarts():
    """The final state written over the initial one, and log decays of -inf
    (forget everything) inside and on the edges of chunks."""
    B, T, Hq, Hkv, D = 2, 400, 4, 2, 128
    q, k, v, beta, decay = delta_inputs(B, T, Hq, Hkv, D, D, torch.bfloat16, "gated_delta", False, Hkv, 41)
    d = decay.float()
    for t, h in [(10, 0), (63, 1), (64, 0), (200, 1), (399, 0)]:
        d[:, t, h] = -float("inf")
    decay = d.to(torch.bfloat16)
    S0 = rand((B, Hkv, D, D), 45, torch.float32)
    S = S0.clone()
    y, _ = la.la_forward_causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                                scale=0.0, update_rule="gated_delta", decay=decay, beta=beta, initial_state=(S, None),
                                return_state=True, state_out=(S, None), out_dtype=torch.float32)
    torch.cuda.synchronize()
    yr, Sr, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, scale=0.0,
                              rule="gated_delta", decay=decay, beta=beta, S0=S0)
    assert np.isfinite(yr).all()
    assert_close(to64(y), yr, tol_for(torch.bfloat16, torch.float32), "y")
    assert_close(to64(S), Sr, tol_for(torch.bfloat16, torch.float32), "S")


def test_delta_tensor_core_form_chunked_calls_equal_one_call():
    """Calls over consecutive pieces with the state carried equal one call."""
    B, T, Hq, Hkv, D = 1, 600, 4, 2, 128
    q, k, v, beta, decay = delta_inputs(B, T, Hq, Hkv, D, D, torch.bfloat16, "gated_delta", False, 1, 51)
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False, update_rule="gated_delta",
              out_dtype=torch.float32)
    S = torch.zeros(B, Hkv, D, D, device=DEV)
    ys = []
    for a0, a1 in [(0, 100), (100, 164), (164, 600)]:
        c = lambda x: x[:, a0:a1].contiguous()
        ys.append(la.la_forward_causal(c(q), c(k), c(v), decay=c(decay), beta=c(beta), initial_state=(S, None),
                                       return_state=True, state_out=(S, None), **kw)[0])
    torch.cuda.synchronize()
    yr, Sr, _ = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map="none", use_normalizer=False,
                              rule="gated_delta", decay=decay, beta=beta)
    assert_close(to64(torch.cat(ys, 1)), yr, tol_for(torch.bfloat16, torch.float32), "chunked y")
    assert_close(to64(S), Sr, tol_for(torch.bfloat16, torch.float32), "chunked S")
