"""GPU parity of the CUDA-core recurrence split into sequence segments (few
(batch, kv head) streams, long sequences): float32 inputs, the gated rule
with one decay per kv head or per key dimension, masks, a carried state and
in-place streaming, against the CPU oracle."""
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


CASES = [  # B, T, Hq, Hkv, Dk, Dv, dtype, rule, decay per key dim, mask kind
    (1, 2000, 2, 2, 64, 64, torch.float32, "linear", False, ""),
    (2, 1537, 4, 2, 32, 48, torch.float32, "linear", False, "gaps"),
    (1, 1800, 3, 1, 128, 128, torch.float32, "gated", False, ""),
    (1, 2100, 4, 2, 64, 64, torch.bfloat16, "gated", True, ""),
    (2, 1600, 2, 2, 128, 64, torch.float32, "gated", True, "random"),
    (1, 1500, 2, 2, 64, 64, torch.bfloat16, "gated", True, "left"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + f"-{c[7]}{'-dim' if c[8] else ''}{'-' + c[9] if c[9] else ''}")
@pytest.mark.parametrize("in_place", [False, True], ids=["state_out", "in_place"])
def test_segmented_recurrence(case, in_place):
    B, T, Hq, Hkv, Dk, Dv, dtype, rule, per_dim, kind = case
    fmap, norm = ("elu_plus_one", True) if rule == "linear" else ("none", False)
    q = rand((B, T, Hq, Dk), 1, dtype, 0.5)
    k = rand((B, T, Hkv, Dk), 2, dtype, 0.5)
    v = rand((B, T, Hkv, Dv), 3, dtype)
    decay = None
    if rule == "gated":
        shape = (B, T, Hkv, Dk) if per_dim else (B, T, Hkv)
        decay = torch.nn.functional.logsigmoid(rand(shape, 4, torch.float32, mean=4.0)).to(dtype)
    mask = inputs.validity_mask(kind, B, T, 5, DEV) if kind else None
    S0 = rand((B, Hkv, Dk, Dv), 6, torch.float32)
    Z0 = rand((B, Hkv, Dk), 7, torch.float32).abs() + 1.0 if norm else None
    S0_ref, Z0_ref = S0.clone(), None if Z0 is None else Z0.clone()
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm, update_rule=rule,
              out_dtype=torch.float32)
    state_out = (S0, Z0) if in_place else None
    y, (S, Z) = la.la_forward_causal(q, k, v, decay=decay, initial_state=(S0, Z0), return_state=True,
                                     state_out=state_out, mask=mask, **kw)
    torch.cuda.synchronize()
    d_or = None if decay is None else (decay.reshape(B, T, Hkv * Dk) if per_dim else decay)
    yr, Sr, Zr = oracle.causal(q, k, v, q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm, rule=rule,
                               decay=d_or, S0=S0_ref, Z0=Z0_ref, mask=mask)
    tol = tol_for(dtype, torch.float32)
    assert_close(to64(y), yr, tol, "y")
    assert_close(to64(S), Sr, tol, "S")
    if norm:
        assert_close(to64(Z), Zr, 1e-5, "Z")
