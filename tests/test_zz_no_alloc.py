"""la_forward_causal_noalloc: the causal pass on the library's built-in
scratch must give what la_forward_causal gives with a caller workspace.

Each case makes two calls in a row on different inputs, so the second one
runs on scratch the first has filled (nothing may depend on it starting at
zero).  Shapes are chosen so the sequence is split into several segments:
the scratch is then really used.  This file sorts last so that it also runs
after every other test in one session; it passes on its own as well.
"""
import re
import os

import pytest
import torch

import kernelized_linear_attention_02_gb300 as la
import linattn_inputs as inputs
from parity_utils import rel_err, to64, TOL_BF16, TOL_BF16_OUT

pytestmark = pytest.mark.gpu

DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


def _inputs(B, T, Hq, Hkv, D, seed, gated):
    g = inputs.generator(seed, DEV)
    q = inputs.normal((B, T, Hq, D), g, 1.0, dtype=torch.bfloat16, device=DEV)
    k = inputs.normal((B, T, Hkv, D), g, 1.0, dtype=torch.bfloat16, device=DEV)
    v = inputs.normal((B, T, Hkv, D), g, 1.0, dtype=torch.bfloat16, device=DEV)
    decay = None
    if gated:
        x = inputs.normal((B, T, Hkv), g, 1.0, dtype=torch.float32, device=DEV) + 3.0
        decay = torch.nn.functional.logsigmoid(x).to(torch.bfloat16)
    S0 = inputs.normal((B, Hkv, D, D), g, 1.0, dtype=torch.float32, device=DEV)
    Z0 = inputs.normal((B, Hkv, D), g, 1.0, dtype=torch.float32, device=DEV).abs() + 1.0
    return q, k, v, decay, S0, Z0


CASES = [
    # (B, T, Hq, Hkv, D, feature map, normalizer, rule, in-place state)
    (1, 2048, 2, 2, 64, "elu_plus_one", True, "linear", False),
    (2, 1000, 8, 2, 128, "none", False, "gated", True),
    (1, 4097, 1, 1, 128, "relu", True, "linear", True),
]


@pytest.mark.parametrize("B,T,Hq,Hkv,D,fmap,norm,rule,inplace", CASES)
def test_noalloc_matches_workspace_call(B, T, Hq, Hkv, D, fmap, norm, rule, inplace):
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm, update_rule=rule)
    p = la.make_params(batch=B, seq_len=T, q_heads=Hq, kv_heads=Hkv, key_dim=D, value_dim=D,
                       feature_map=fmap, use_normalizer=norm, update_rule=rule)
    need = la.la_workspace_bytes(p, True)
    assert 0 < need <= la.LA_NOALLOC_SCRATCH_BYTES, need  # split into segments, fits the scratch
    for call, seed in enumerate((11, 23)):  # two calls in a row
        q, k, v, decay, S0, Z0 = _inputs(B, T, Hq, Hkv, D, seed, rule == "gated")
        Z0 = Z0 if norm else None
        y_ref, (S_ref, Z_ref) = la.la_forward_causal(q, k, v, decay=decay, initial_state=(S0, Z0),
                                                     return_state=True, **kw)
        y = torch.empty_like(y_ref)
        if inplace:  # the final state overwrites the initial one
            S, Z = S0.clone(), (Z0.clone() if norm else None)
            la.la_forward_causal_noalloc(q, k, v, decay=decay, initial_state=(S, Z), out=y,
                                         state_out=(S, Z), **kw)
        else:
            S = torch.empty_like(S_ref)
            Z = torch.empty_like(Z_ref) if norm else None
            la.la_forward_causal_noalloc(q, k, v, decay=decay, initial_state=(S0, Z0), out=y,
                                         state_out=(S, Z), **kw)
        torch.cuda.synchronize()
        ey = rel_err(to64(y), to64(y_ref))
        eS = rel_err(to64(S), to64(S_ref))
        assert ey <= TOL_BF16_OUT, f"call {call}: y rel err {ey:.3e}"
        assert eS <= TOL_BF16, f"call {call}: S rel err {eS:.3e}"
        if norm:
            eZ = rel_err(to64(Z), to64(Z_ref))
            assert eZ <= TOL_BF16, f"call {call}: Z rel err {eZ:.3e}"


def test_scratch_size_covers_every_causal_problem_on_this_device():
    """The largest causal workspace on this device (head size 128, the
    (batch x kv head) count that maximises segments times state copies) fits
    the built-in scratch, and the header states the same size as the binding."""
    header = open(os.path.join(ROOT, "include", "linattn.h")).read()
    m = re.search(r"#define LA_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", header)
    assert m and int(m.group(1)) << int(m.group(2)) == la.LA_NOALLOC_SCRATCH_BYTES
    worst = 0
    for bh in range(1, 2 * torch.cuda.get_device_properties(0).multi_processor_count + 1):
        p = la.make_params(batch=bh, seq_len=1 << 20, q_heads=1, kv_heads=1, key_dim=128, value_dim=128,
                           feature_map="relu", use_normalizer=True)
        worst = max(worst, la.la_workspace_bytes(p, True))
    assert 0 < worst <= la.LA_NOALLOC_SCRATCH_BYTES, worst
