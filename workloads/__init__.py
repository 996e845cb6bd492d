"""Seeded synthetic inputs shaped like the pages' decode workloads.

This module is the one piece shared by the tests, the benchmark, the oracle
side and the CUDA side: it only draws random numbers and lays them out.  It
holds none of the method's arithmetic (no decode, no GEMM, no acceptance).

Workloads (shapes from "Module 11. Speculative Decoding and Quantization",
§1 and §10: an 8B dense decoder read once per verification step; the 70B case
from "Inference at the Memory Wall ...", section "The physical reality of the
memory bandwidth wall"):

* tiny      -- one 256x512 MXFP4 layer, X 4x512 (batch 1, K_spec 3),
               acceptance over vocab 1024.
* llama8b   -- hidden 4096: QKV 4096->6144, O 4096->4096, gate+up 4096->28672,
               down 14336->4096, 32 layers, lm_head 4096->128256, vocab 128256.
* llama70b  -- hidden 8192: QKV 8192->10240, O 8192->8192, gate+up
               8192->57344, down 28672->8192, 80 layers, lm_head 8192->128256.

Distributions: packed nibble bytes uniform over 0..255 (so each E2M1 code is
uniform over its 16 values), E8M0 exponents uniform over an inclusive range,
X ~ N(0, 1) rounded to bf16 (round to nearest even), logits ~ N(0, sigma)
with sigma the standard deviation, softmax in float64 then stored as fp32,
draft tokens drawn from q by inverse CDF, uniforms U[0, 1) in fp32.
Every host tensor has its own stream PCG64(SeedSequence([seed, tensor_id])).
"""
from __future__ import annotations

import numpy as np

# (name, K in_features, N out_features)
LLAMA8B_LAYER = (("qkv", 4096, 6144), ("o", 4096, 4096),
                 ("gate_up", 4096, 28672), ("down", 14336, 4096))
LLAMA8B_LM_HEAD = ("lm_head", 4096, 128256)
LLAMA8B_LAYERS = 32
LLAMA70B_LAYER = (("qkv", 8192, 10240), ("o", 8192, 8192),
                  ("gate_up", 8192, 57344), ("down", 28672, 8192))
LLAMA70B_LM_HEAD = ("lm_head", 8192, 128256)
LLAMA70B_LAYERS = 80
VOCAB_LLAMA = 128256

TINY = dict(N=256, K=512, M=4, exp_lo=120, exp_hi=130, B=1, K_spec=3, V=1024,
            logit_std=2.0, seed=0)
LLAMA_EXP_RANGE = (118, 132)


def stack_shapes(model: str):
    """List of (name, K, N) for every GEMM of one verification step, in order."""
    if model == "llama8b":
        layer, head, nl = LLAMA8B_LAYER, LLAMA8B_LM_HEAD, LLAMA8B_LAYERS
    elif model == "llama70b":
        layer, head, nl = LLAMA70B_LAYER, LLAMA70B_LM_HEAD, LLAMA70B_LAYERS
    else:
        raise ValueError(model)
    out = []
    for li in range(nl):
        for name, K, N in layer:
            out.append((f"l{li}.{name}", K, N))
    out.append(head)
    return out


def host_rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id])))


# --------------------------------------------------------------------------
# GEMM inputs
# --------------------------------------------------------------------------

def mxfp4_weights(N: int, K: int, exp_lo: int, exp_hi: int, seed: int,
                  tensor_id: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Random packed MXFP4 weights: (nibbles uint8 [N, K/2], scales uint8 [N, K/32])."""
    assert K % 32 == 0
    g = host_rng(seed, tensor_id)
    nib = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sc = g.integers(exp_lo, exp_hi + 1, size=(N, K // 32), dtype=np.uint8)
    return nib, sc


def nvfp4_weights(N: int, K: int, seed: int, tensor_id: int = 0, exp_lo: int = 4,
                  exp_hi: int = 10) -> tuple[np.ndarray, np.ndarray]:
    """Random packed NVFP4 weights: (nibbles uint8 [N, K/2], E4M3 scale bytes
    uint8 [N, K/16]); positive scales with exponent field in [exp_lo, exp_hi]
    (<= 14: no NaN) and a random 3-bit fraction."""
    assert K % 16 == 0 and 0 <= exp_lo <= exp_hi <= 14
    g = host_rng(seed, tensor_id)
    nib = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    e = g.integers(exp_lo, exp_hi + 1, size=(N, K // 16), dtype=np.uint8)
    f = g.integers(0, 8, size=(N, K // 16), dtype=np.uint8)
    return nib, ((e << 3) | f).astype(np.uint8)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_normal(M: int, K: int, seed: int, tensor_id: int = 1, std: float = 1.0) -> np.ndarray:
    """X ~ N(0, std) rounded to bf16, as uint16 bit patterns [M, K]."""
    g = host_rng(seed, tensor_id)
    return f32_to_bf16_bits(g.standard_normal((M, K), dtype=np.float32) * np.float32(std))


def tiny_gemm_inputs(seed: int = 0):
    t = TINY
    nib, sc = mxfp4_weights(t["N"], t["K"], t["exp_lo"], t["exp_hi"], seed, 0)
    x = bf16_normal(t["M"], t["K"], seed, 1)
    return x, nib, sc


def device_mxfp4_weights(N: int, K: int, exp_lo: int, exp_hi: int, seed: int, device):
    """Random packed MXFP4 weights generated directly in device memory (torch RNG).

    Used for the multi-GB stacks; sampled rows are copied back to the host
    when the oracle needs them.
    """
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    nib = torch.randint(0, 256, (N, K // 2), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
    sc = torch.randint(exp_lo, exp_hi + 1, (N, K // 32), generator=gen, device=device,
                       dtype=torch.int32).to(torch.uint8)
    return nib, sc


def device_nvfp4_weights(N: int, K: int, seed: int, device, exp_lo: int = 4, exp_hi: int = 10):
    """nvfp4_weights' distribution, generated in device memory (torch RNG)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    nib = torch.randint(0, 256, (N, K // 2), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
    e = torch.randint(exp_lo, exp_hi + 1, (N, K // 16), generator=gen, device=device, dtype=torch.int32)
    f = torch.randint(0, 8, (N, K // 16), generator=gen, device=device, dtype=torch.int32)
    return nib, ((e << 3) | f).to(torch.uint8)


def device_bf16_normal(M: int, K: int, seed: int, device, std: float = 1.0):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return (torch.randn((M, K), generator=gen, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


# --------------------------------------------------------------------------
# Acceptance inputs
# --------------------------------------------------------------------------

def _softmax_f64(logits: np.ndarray) -> np.ndarray:
    z = logits.astype(np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def _draw_from(probs_row: np.ndarray, uni: float) -> int:
    c = np.cumsum(probs_row.astype(np.float64))
    idx = int(np.searchsorted(c, uni * c[-1], side="right"))
    return min(idx, probs_row.shape[0] - 1)


def spec_inputs(B: int, K: int, V: int, seed: int, *, logit_std: float = 2.0,
                draft_noise: float | None = None):
    """p [B,K+1,V] f32, q [B,K,V] f32, draft [B,K] int32, u [B,K+1] f32.

    Target logits ~ N(0, logit_std).  Draft logits are independent
    N(0, logit_std) when ``draft_noise`` is None, else target + N(0, draft_noise).
    Draft token i is drawn from q_i; u ~ U[0, 1).
    """
    g_t = host_rng(seed, 10)
    g_d = host_rng(seed, 11)
    g_x = host_rng(seed, 12)
    g_u = host_rng(seed, 13)
    tl = g_t.standard_normal((B, K + 1, V), dtype=np.float32) * np.float32(logit_std)
    if draft_noise is None:
        dl = g_d.standard_normal((B, K, V), dtype=np.float32) * np.float32(logit_std)
    else:
        dl = tl[:, :K, :] + g_d.standard_normal((B, K, V), dtype=np.float32) * np.float32(draft_noise)
    p = _softmax_f64(tl).astype(np.float32)
    q = _softmax_f64(dl).astype(np.float32)
    draws = g_x.random((B, K))
    draft = np.empty((B, K), dtype=np.int32)
    for b in range(B):
        for i in range(K):
            draft[b, i] = _draw_from(q[b, i], draws[b, i])
    u = g_u.random((B, K + 1), dtype=np.float32)
    return p, q, draft, u


def tune_draft_noise(target_alpha: float, V: int, logit_std: float, seed: int,
                     samples: int = 16) -> float:
    """Noise sigma for which the mean overlap sum_t min(p_t, q_t) of
    softmax(l) and softmax(l + N(0, sigma)) is ``target_alpha`` (bisection on
    seeded samples; this only shapes the synthetic draft law)."""
    g = host_rng(seed, 20)
    base = g.standard_normal((samples, V), dtype=np.float32) * np.float32(logit_std)
    noise = g.standard_normal((samples, V), dtype=np.float32)
    p = _softmax_f64(base)

    def overlap(sig):
        q = _softmax_f64(base + noise * np.float32(sig))
        return float(np.minimum(p, q).sum(axis=-1).mean())

    lo, hi = 0.0, 4.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if overlap(mid) > target_alpha:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)
