"""CPU-only checks of the C ABI: the library loads, exports every entry point
the header declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import kernelized_linear_attention_02_gb300 as la
from kernelized_linear_attention_02_gb300 import build as la_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    la_build.build()
    return la.lib()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[\w\s\*]*?\b(la_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("la_forward_causal", "la_forward_noncausal", "la_decode_step", "la_get_initial_state",
              "la_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_params_struct_layout_matches_header():
    # int64 x2, int32 x8, float x2, int32 x2 -> 64 bytes, no padding surprises
    assert ctypes.sizeof(la.la_params) == 64
    assert la.la_params.epsilon.offset == 48


def _p(**kw):
    base = dict(batch=2, seq_len=8, q_heads=4, kv_heads=2, key_dim=64, value_dim=64)
    base.update(kw)
    return la.make_params(**base)


BAD = [
    (dict(batch=0), la.LA_ERR_INVALID_ARG),
    (dict(seq_len=-1), la.LA_ERR_INVALID_ARG),
    (dict(q_heads=3, kv_heads=2), la.LA_ERR_INVALID_ARG),
    (dict(key_dim=0), la.LA_ERR_INVALID_ARG),
    (dict(key_dim=256), la.LA_ERR_UNSUPPORTED),
    (dict(epsilon=-1.0), la.LA_ERR_INVALID_ARG),
    (dict(epsilon=float("nan")), la.LA_ERR_INVALID_ARG),
    (dict(update_rule="gated"), la.LA_ERR_UNSUPPORTED),  # gated with elu+1 and the normalizer
]


@pytest.mark.parametrize("kw,status", BAD, ids=[str(b[0]) for b in BAD])
def test_invalid_params_are_rejected_without_launch(L, kw, status):
    p = _p(**kw)
    dummy = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    rc = L.la_forward_causal(ctypes.byref(p), dummy, dummy, dummy, dummy, None, None, dummy, None,
                             None, None, 0, None)  # q k v decay S0 Z0 y S_out Z_out ws
    assert rc == status
    assert L.la_last_error().decode()


def test_bad_enum_values(L):
    p = _p()
    p.io_dtype = 7
    assert L.la_forward_causal(ctypes.byref(p), *([None] * 10), 0, None) == la.LA_ERR_INVALID_ARG
    p = _p()
    p.feature_map = 9
    assert L.la_forward_causal(ctypes.byref(p), *([None] * 10), 0, None) == la.LA_ERR_INVALID_ARG
    p = _p()
    p.decay_per_key_dim = 1  # needs the gated rule
    assert L.la_forward_causal(ctypes.byref(p), *([None] * 10), 0, None) == la.LA_ERR_INVALID_ARG


def test_null_pointers_rejected(L):
    p = _p()
    assert L.la_forward_causal(ctypes.byref(p), *([None] * 10), 0, None) == la.LA_ERR_INVALID_ARG
    assert L.la_forward_causal(None, *([None] * 10), 0, None) == la.LA_ERR_INVALID_ARG
    assert L.la_get_initial_state(ctypes.byref(p), None, None, None) == la.LA_ERR_INVALID_ARG


def test_gated_needs_decay(L):
    p = _p(update_rule="gated", feature_map="none", use_normalizer=False)
    d = ctypes.c_void_p(16)
    assert L.la_forward_causal(ctypes.byref(p), d, d, d, None, None, None, d, None, None, None, 0,
                               None) == la.LA_ERR_INVALID_ARG  # decay missing


def test_decode_needs_single_token(L):
    p = _p(seq_len=2)
    d = ctypes.c_void_p(16)
    assert L.la_decode_step(ctypes.byref(p), d, d, d, None, d, d, d, None) == la.LA_ERR_INVALID_ARG


def test_noncausal_rejects_gated(L):
    p = _p(update_rule="gated", feature_map="none", use_normalizer=False)
    d = ctypes.c_void_p(16)
    assert L.la_forward_noncausal(ctypes.byref(p), d, d, d, d, None, 0, None) == la.LA_ERR_UNSUPPORTED


def test_workspace_too_small_rejected(L):
    p = _p()
    need = L.la_workspace_bytes(ctypes.byref(p), 0)
    assert need > 0
    d = ctypes.c_void_p(256)
    assert L.la_forward_noncausal(ctypes.byref(p), d, d, d, d, d, need - 1, None) == la.LA_ERR_WORKSPACE
    assert L.la_forward_noncausal(ctypes.byref(p), d, d, d, d, ctypes.c_void_p(257), need,
                                  None) == la.LA_ERR_WORKSPACE


def test_status_strings(L):
    for s in range(6):
        assert L.la_status_string(s)
        assert L.la_status_str(s) == L.la_status_string(s)
    assert L.la_abi_version() == 3


def test_bounded_wait_selftest_rejects_bad_limits(L):
    assert L.la_check_bounded_wait(0, None) == la.LA_ERR_INVALID_ARG
    assert L.la_check_bounded_wait(1000001, None) == la.LA_ERR_INVALID_ARG


# ---- entry points added with the masks, the delta rules and the backward pass:
# each rejects bad arguments before it enqueues anything (no GPU needed)

def _delta(**kw):
    base = dict(feature_map="none", use_normalizer=False, update_rule="delta")
    base.update(kw)
    return _p(**base)


def test_plain_calls_refuse_the_delta_rules(L):
    p = _delta()
    d = ctypes.c_void_p(16)
    assert L.la_forward_causal(ctypes.byref(p), d, d, d, None, None, None, d, None, None, None, 0,
                               None) == la.LA_ERR_INVALID_ARG
    assert "la_forward_causal_delta" in L.la_last_error().decode()
    p1 = _delta(seq_len=1)
    assert L.la_decode_step(ctypes.byref(p1), d, d, d, None, d, None, d, None) == la.LA_ERR_INVALID_ARG


def test_delta_entry_point_checks(L):
    d = ctypes.c_void_p(16)
    call = lambda p, beta, bph=1, decay=None: L.la_forward_causal_delta(ctypes.byref(p), d, d, d, decay, beta, bph,
                                                                        None, None, d, None, None)
    assert call(_delta(), None) == la.LA_ERR_INVALID_ARG                     # beta missing
    assert call(_delta(), d, bph=2) == la.LA_ERR_INVALID_ARG                 # beta layout flag
    assert call(_delta(update_rule="gated_delta"), d) == la.LA_ERR_INVALID_ARG  # gated_delta without decay
    assert call(_delta(update_rule="linear"), d) == la.LA_ERR_INVALID_ARG    # not a delta rule
    assert call(_delta(feature_map="elu_plus_one"), d) == la.LA_ERR_UNSUPPORTED
    assert call(_delta(use_normalizer=True, feature_map="none"), d) == la.LA_ERR_UNSUPPORTED
    p2 = _delta(seq_len=2)
    assert L.la_decode_step_delta(ctypes.byref(p2), d, d, d, None, d, 1, None, d, d, None) == la.LA_ERR_INVALID_ARG
    p1 = _delta(seq_len=1)
    assert L.la_decode_step_delta(ctypes.byref(p1), d, d, d, None, d, 1, None, None, d, None) == la.LA_ERR_INVALID_ARG


def test_masked_entry_points_validate_like_the_plain_ones(L):
    d = ctypes.c_void_p(16)
    p = _p(batch=0)
    assert L.la_forward_causal_masked(ctypes.byref(p), d, d, d, None, d, None, None, d, None, None, None, 0,
                                      None) == la.LA_ERR_INVALID_ARG
    assert L.la_forward_noncausal_masked(ctypes.byref(p), d, d, d, d, d, None, 0, None) == la.LA_ERR_INVALID_ARG
    p = _p(seq_len=3)
    assert L.la_decode_step_masked(ctypes.byref(p), d, d, d, None, d, d, d, d, None) == la.LA_ERR_INVALID_ARG


def test_backward_checks(L):
    d = ctypes.c_void_p(256)
    p = _p(update_rule="gated", feature_map="none", use_normalizer=False)
    assert L.la_backward_causal(ctypes.byref(p), d, d, d, None, None, d, d, d, d, None, None, d, 1 << 20,
                                None) == la.LA_ERR_UNSUPPORTED
    p = _p()
    need = L.la_backward_workspace_bytes(ctypes.byref(p))
    assert need > 0
    assert L.la_backward_causal(ctypes.byref(p), d, d, d, None, None, d, d, d, d, None, None, d, need - 1,
                                None) == la.LA_ERR_WORKSPACE
    assert L.la_backward_causal(ctypes.byref(p), d, d, d, None, None, None, d, d, d, None, None, d, need,
                                None) == la.LA_ERR_INVALID_ARG  # dy missing


def test_decay_per_key_dim_accepted_only_for_gated_rules(L):
    d = ctypes.c_void_p(16)
    p = _p(update_rule="gated", feature_map="none", use_normalizer=False, decay_per_key_dim=True)
    # valid parameters: only the missing decay is reported
    assert L.la_forward_causal(ctypes.byref(p), d, d, d, None, None, None, d, None, None, None, 0,
                               None) == la.LA_ERR_INVALID_ARG
    assert "decay" in L.la_last_error().decode()
    p = _p(decay_per_key_dim=True)
    assert L.la_forward_causal(ctypes.byref(p), d, d, d, d, None, None, d, None, None, None, 0,
                               None) == la.LA_ERR_INVALID_ARG
    assert "gated" in L.la_last_error().decode()
