"""la_forward_causal_noalloc: the causal pass on the library's built-in
scratch must give what la_forward_causal gives with a caller workspace.

Each case makes two calls in a row on different inputs, so the second one
runs on scratch the first has filled (nothing may depend on it starting at
zero).  Shapes are chosen so the sequence is split into several segments:
the scratch is then really used.  This file sorts last so that it also runs
after every other test in one session; it passes on its own as well.
"""
import ctypes
import os
import re

import pytest
import torch

import kernelized_linear_attention_02_gb300 as la
import linattn_inputs as inputs
from parity_utils import assert_close, to64, tol_for

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


def _inputs(B, T, Hq, Hkv, D, seed, gated, dtype=torch.bfloat16, per_dim=False):
    g = inputs.generator(seed, DEV)
    q = inputs.normal((B, T, Hq, D), g, 1.0, dtype=dtype, device=DEV)
    k = inputs.normal((B, T, Hkv, D), g, 1.0, dtype=dtype, device=DEV)
    v = inputs.normal((B, T, Hkv, D), g, 1.0, dtype=dtype, device=DEV)
    decay = None
    if gated:
        shape = (B, T, Hkv, D) if per_dim else (B, T, Hkv)
        x = inputs.normal(shape, g, 1.0, dtype=torch.float32, device=DEV) + 3.0
        decay = torch.nn.functional.logsigmoid(x).to(dtype)
    S0 = inputs.normal((B, Hkv, D, D), g, 1.0, dtype=torch.float32, device=DEV)
    Z0 = inputs.normal((B, Hkv, D), g, 1.0, dtype=torch.float32, device=DEV).abs() + 1.0
    return q, k, v, decay, S0, Z0


CASES = [
    # (B, T, Hq, Hkv, D, feature map, normalizer, rule, in-place state, io dtype, per-key-dim decay)
    (1, 2048, 2, 2, 64, "elu_plus_one", True, "linear", False, torch.bfloat16, False),
    (2, 1000, 8, 2, 128, "none", False, "gated", True, torch.bfloat16, False),
    (1, 4097, 1, 1, 128, "relu", True, "linear", True, torch.bfloat16, False),
    # the CUDA-core recurrence, split into sequence segments on the scratch
    (1, 1500, 2, 2, 64, "elu_plus_one", True, "linear", True, torch.float32, False),
    (1, 1200, 4, 2, 64, "none", False, "gated", False, torch.bfloat16, True),
]


@pytest.mark.parametrize("B,T,Hq,Hkv,D,fmap,norm,rule,inplace,dtype,per_dim", CASES,
                         ids=lambda x: str(x).replace("torch.", ""))
def test_noalloc_matches_workspace_call(B, T, Hq, Hkv, D, fmap, norm, rule, inplace, dtype, per_dim):
    kw = dict(q_heads=Hq, kv_heads=Hkv, feature_map=fmap, use_normalizer=norm, update_rule=rule)
    p = la.make_params(batch=B, seq_len=T, q_heads=Hq, kv_heads=Hkv, key_dim=D, value_dim=D, io_dtype=dtype,
                       feature_map=fmap, use_normalizer=norm, update_rule=rule, decay_per_key_dim=per_dim)
    need = la.la_workspace_bytes(p, True)
    assert 0 < need <= la.LA_NOALLOC_SCRATCH_BYTES, need  # split into segments, fits the scratch
    for call, seed in enumerate((11, 23)):  # two calls in a row
        q, k, v, decay, S0, Z0 = _inputs(B, T, Hq, Hkv, D, seed, rule == "gated", dtype, per_dim)
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
        assert_close(to64(y), to64(y_ref), tol_for(dtype, dtype), f"call {call}: y")
        assert_close(to64(S), to64(S_ref), tol_for(dtype, torch.float32), f"call {call}: S")
        if norm:
            assert_close(to64(Z), to64(Z_ref), tol_for(dtype, torch.float32), f"call {call}: Z")


def test_scratch_size_covers_every_causal_problem_on_this_device():
    """The largest causal workspace on this device (head size 128, the
    (batch x kv head) count that maximises segments times state copies) fits
    the built-in scratch, and the header states the same size as the binding."""
    header = open(os.path.join(ROOT, "include", "linattn.h")).read()
    m = re.search(r"#define LA_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", header)
    assert m and int(m.group(1)) << int(m.group(2)) == la.LA_NOALLOC_SCRATCH_BYTES
    worst = 0
    # the tensor-core path (bf16, head size 128) and the CUDA-core recurrence
    # (float32 io; per-key-dimension decay), whose segment scratch is sized
    # differently (a segment cap plus a copy of the initial state)
    kinds = [dict(io_dtype=torch.bfloat16, feature_map="relu", use_normalizer=True),
             dict(io_dtype=torch.float32, feature_map="relu", use_normalizer=True),
             dict(io_dtype=torch.float32, feature_map="none", use_normalizer=False, update_rule="gated",
                  decay_per_key_dim=True)]
    for kind in kinds:
        for bh in range(1, 2 * torch.cuda.get_device_properties(0).multi_processor_count + 1):
            p = la.make_params(batch=bh, seq_len=1 << 20, q_heads=1, kv_heads=1, key_dim=128, value_dim=128, **kind)
            worst = max(worst, la.la_workspace_bytes(p, True))
    assert 0 < worst <= la.LA_NOALLOC_SCRATCH_BYTES, worst
    # bf16 with one decay per key dimension: its tensor-core form wants more
    # than the scratch on long sequences, and the call then takes the
    # recurrence, which fits: it gets past the scratch check to the pointer
    # check (nothing is launched)
    L = la.lib()
    for bh in (1, 8, 76, 152):
        p = la.make_params(batch=bh, seq_len=1 << 20, q_heads=1, kv_heads=1, key_dim=128, value_dim=128,
                           feature_map="none", use_normalizer=False, update_rule="gated", decay_per_key_dim=True)
        assert la.la_workspace_bytes(p, True) > la.LA_NOALLOC_SCRATCH_BYTES
        st = L.la_forward_causal_noalloc(ctypes.byref(p), None, None, None, None, None, None, None, None, None, None)
        assert st == la.LA_ERR_INVALID_ARG, (bh, st)
