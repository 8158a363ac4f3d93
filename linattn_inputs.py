"""Seeded synthetic inputs for kernelized linear attention.

This module is shared by the tests, the benchmark and the smoke check; it
feeds both the CUDA library and the CPU oracle.  It draws random tensors and
nothing else: it holds none of the method's arithmetic.

The workloads below are the shapes and value distributions the library is
measured and checked on.  No dataset is involved; every tensor is drawn from a
seeded ``torch.Generator`` on the requested device.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    q_heads: int
    kv_heads: int
    Dk: int
    Dv: int
    dtype: torch.dtype
    feature_map: str          # "elu_plus_one" | "relu" | "none"
    use_normalizer: bool
    eps: float
    scale: float              # 0.0 -> 1/sqrt(Dk) (ONNX convention)
    rule: str                 # "linear" | "gated" | "delta" | "gated_delta"
    qk_std: float = 1.0       # q, k ~ N(0, qk_std^2)
    v_std: float = 1.0
    k_l2_normalize: bool = False
    decay_mu: float = 4.0     # gated: g = log(sigmoid(x)), x ~ N(decay_mu, 1)
    seed: int = 0
    mask: str = ""            # "" (no mask) or a validity_mask kind, e.g. "right"
    decay_per_dim: bool = False  # gated: decay (B,T,Hkv,Dk) per key dimension instead of (B,T,Hkv)


TINY = Workload("tiny_B1_H2_T64_D16_f32", 1, 64, 2, 2, 16, 16, torch.float32,
                "elu_plus_one", True, 1e-6, 1.0, "linear", qk_std=0.5, seed=42)
PREFILL_2K = Workload("causal_prefill_B4_H8_T2048_D64_bf16", 4, 2048, 8, 8, 64, 64,
                      torch.bfloat16, "elu_plus_one", True, 1e-6, 1.0, "linear", qk_std=0.5)
LONG_8K = Workload("long_prefill_B8_H16_T8192_D128_bf16_relu", 8, 8192, 16, 16, 128, 128,
                   torch.bfloat16, "relu", True, 1e-6, 1.0, "linear")
LONG_8K_UNNORM = dataclasses.replace(LONG_8K, name=LONG_8K.name + "_unnormalized",
                                     use_normalizer=False)
DECODE = Workload("decode_B256_H32_D128_prefill4096", 256, 4096, 32, 32, 128, 128,
                  torch.bfloat16, "elu_plus_one", True, 1e-6, 1.0, "linear")
DECODE_STEPS = 1024
ONNX_LINEAR = Workload("onnx_linear_gqa_B2_T32768_Hq32_Hkv8_D128_bf16", 2, 32768, 32, 8,
                       128, 128, torch.bfloat16, "none", False, 0.0, 1.0 / math.sqrt(128),
                       "linear", k_l2_normalize=True)
ONNX_GATED = dataclasses.replace(ONNX_LINEAR, name="onnx_gated_gqa_B2_T32768_Hq32_Hkv8_D128_bf16",
                                 rule="gated")

# the 2k prefill as a right-padded batch: sequence b is valid for its first
# L_b steps, L_b uniform in [T/2, T] (Keras request, Masking: right padding)
PREFILL_2K_RIGHTPAD = dataclasses.replace(PREFILL_2K, name=PREFILL_2K.name + "_rightpad_mask", mask="right")

# the gated rule with one log decay per key dimension (ONNX decay layout
# (B, T, H_kv*d_k)), on a shorter sequence: it runs on the CUDA-core recurrence
GATED_PERDIM = dataclasses.replace(ONNX_GATED, name="gated_perdim_gqa_B2_T4096_Hq32_Hkv8_D128_bf16", T=4096,
                                   decay_per_dim=True)

# the ONNX operator's default rule, gated_delta (beta per kv head), on the
# CUDA-core recurrence
GATED_DELTA = dataclasses.replace(ONNX_GATED, name="gated_delta_gqa_B2_T4096_Hq32_Hkv8_D128_bf16", T=4096,
                                  rule="gated_delta")

ALL = [TINY, PREFILL_2K, LONG_8K, LONG_8K_UNNORM, DECODE, ONNX_LINEAR, ONNX_GATED, PREFILL_2K_RIGHTPAD,
       GATED_PERDIM, GATED_DELTA]

MASK_KINDS = ("right", "left", "gaps", "random", "none_valid", "all_valid")


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, gen: torch.Generator, std=1.0, mean=0.0, dtype=torch.float32, device="cpu"):
    """N(mean, std^2) drawn in fp32 on ``device``, then rounded to ``dtype``."""
    x = torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    if mean != 0.0:
        x = x + mean
    return x.to(dtype)


def make_qkv(w: Workload, device="cpu", T=None, B=None, seed=None):
    """q (B,T,Hq,Dk), k (B,T,Hkv,Dk), v (B,T,Hkv,Dv) and, for the gated rule,
    decay (B,T,Hkv) (or (B,T,Hkv,Dk) per key dimension) -- contiguous, the
    packed [B,T,H*D] memory of the ONNX op.

    Draw order q, k, v, decay.  Keys are L2-normalised over Dk in fp32 before
    rounding when the workload asks for it (the ONNX page recommends
    normalised keys); the log-decay is log(sigmoid(x)), x ~ N(decay_mu, 1)."""
    T = w.T if T is None else T
    B = w.B if B is None else B
    g = generator(w.seed if seed is None else seed, device)
    q = normal((B, T, w.q_heads, w.Dk), g, w.qk_std, dtype=w.dtype, device=device)
    if w.k_l2_normalize:
        k32 = normal((B, T, w.kv_heads, w.Dk), g, w.qk_std, dtype=torch.float32, device=device)
        k = (k32 / k32.norm(dim=-1, keepdim=True).clamp_min(1e-12)).to(w.dtype)
    else:
        k = normal((B, T, w.kv_heads, w.Dk), g, w.qk_std, dtype=w.dtype, device=device)
    v = normal((B, T, w.kv_heads, w.Dv), g, w.v_std, dtype=w.dtype, device=device)
    decay = None
    if w.rule in ("gated", "gated_delta"):
        dshape = (B, T, w.kv_heads, w.Dk) if w.decay_per_dim else (B, T, w.kv_heads)
        x = normal(dshape, g, 1.0, mean=w.decay_mu, dtype=torch.float32, device=device)
        decay = torch.nn.functional.logsigmoid(x).to(w.dtype)
    return q, k, v, decay


def make_beta(w: Workload, device="cpu", seed=None) -> torch.Tensor:
    """Update rate of the delta rules, (B, T, Hkv): sigmoid(x), x ~ N(0, 1)
    (the ONNX page's beta is a sigmoid output), drawn after the other inputs'
    generator (its own seed offset)."""
    g = generator((w.seed if seed is None else seed) + 7919, device)
    return torch.sigmoid(normal((w.B, w.T, w.kv_heads), g, 1.0, dtype=torch.float32, device=device)).to(w.dtype)


def validity_mask(kind: str, B: int, T: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """A (B, T) bool sequence-validity mask of one of the layouts the Keras
    request's tests name (Mask and state behavior):

    right       sequence b valid for its first L_b steps, L_b ~ U[T/2, T]
    left        valid for its last L_b steps
    gaps        valid except 1-3 interior runs of 1..T/4 steps per sequence
    random      each step valid with probability 0.7
    none_valid  all false;  all_valid  all true."""
    g = generator(seed, "cpu")
    t = torch.arange(T)
    if kind in ("right", "left"):
        L = torch.randint(T // 2, T + 1, (B,), generator=g) if T > 0 else torch.zeros(B, dtype=torch.long)
        m = t[None, :] < L[:, None] if kind == "right" else t[None, :] >= (T - L)[:, None]
    elif kind == "gaps":
        m = torch.ones(B, T, dtype=torch.bool)
        for b in range(B):
            for _ in range(int(torch.randint(1, 4, (1,), generator=g))):
                n = int(torch.randint(1, max(2, T // 4 + 1), (1,), generator=g))
                s = int(torch.randint(0, max(1, T - n + 1), (1,), generator=g))
                m[b, s:s + n] = False
    elif kind == "random":
        m = torch.rand(B, T, generator=g) < 0.7
    elif kind == "none_valid":
        m = torch.zeros(B, T, dtype=torch.bool)
    elif kind == "all_valid":
        m = torch.ones(B, T, dtype=torch.bool)
    else:
        raise ValueError(kind)
    return m.to(device)


def tiny_paper_inputs(seed=42, n=32, d=16):
    """The n=32, d=16 draw of the 'Causal Linear Attention' notebook, replayed
    with numpy's legacy seeded generator (order Q, K, V; Q and K times 0.5)."""
    import numpy as np
    np.random.seed(seed)
    Q = np.random.randn(n, d).astype(np.float32) * 0.5
    K = np.random.randn(n, d).astype(np.float32) * 0.5
    V = np.random.randn(n, d).astype(np.float32)
    return Q, K, V
