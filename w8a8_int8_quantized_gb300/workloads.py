"""Seeded synthetic inputs for the W8A8 INT8 linear workloads.

This module only draws random numbers and casts them to the storage formats the
layer consumes (bf16, FP8 E4M3, int32 routing tables).  It contains none of the
quantization arithmetic; both the CUDA library's tests and the CPU oracle take
their inputs from here.  All tensors are CPU torch tensors; ``bits()`` gives the
uint16 numpy view that the oracle reads.

Every tensor gets its own generator stream (seed, stream id), drawn in a fixed
order, so that a workload is reproducible element for element.
"""

import math

import numpy as np
import torch

__all__ = [
    "bits", "tiny_linear", "llama_shapes", "llama_activations", "weight_bf16",
    "asym_activations", "moe_workload", "fp8_block_matrix", "requant_workload",
]


def _gen(seed, stream):
    g = torch.Generator()
    g.manual_seed(int(seed) * 1_000_003 + int(stream))
    return g


def _normal(shape, mean, std, seed, stream):
    t = torch.randn(*shape, generator=_gen(seed, stream), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def bits(t):
    """uint16 bit patterns of a bf16 CPU tensor (numpy view, no copy)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def tiny_linear(seed=0):
    """x[16,512] ~ N(0,1), W[512,512] ~ N(0,0.02), bias[512] ~ N(0,0.1), all bf16."""
    x = _normal((16, 512), 0.0, 1.0, seed, 1).to(torch.bfloat16)
    w = _normal((512, 512), 0.0, 0.02, seed, 2).to(torch.bfloat16)
    b = _normal((512,), 0.0, 0.1, seed, 3).to(torch.bfloat16)
    return dict(x=x, w=w, bias=b)


def llama_shapes():
    """(name, N, K) of the four Llama-3-8B linear layers."""
    return [("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 28672, 4096), ("down", 4096, 14336)]


def llama_activations(M, K, seed=0, stream=10):
    """x[M,K] ~ N(0,1) with 1% of the K channels (seeded choice) scaled by 20 before bf16 rounding."""
    x = _normal((M, K), 0.0, 1.0, seed, stream)
    n_out = int(round(0.01 * K))
    ch = torch.randperm(K, generator=_gen(seed, stream + 1))[:n_out]
    x[:, ch] *= 20.0
    return x.to(torch.bfloat16)


def weight_bf16(N, K, seed=0, stream=20, std=0.02):
    """W[N,K] ~ N(0, std) in bf16."""
    return _normal((N, K), 0.0, std, seed, stream).to(torch.bfloat16)


def asym_activations(M, K, seed=0, stream=30):
    """x[M,K] ~ N(0.5, 1) in bf16: rows with non-zero mean."""
    return _normal((M, K), 0.5, 1.0, seed, stream).to(torch.bfloat16)


def moe_workload(T=4096, H=4096, E=32, topk=4, inter=1408, seed=0, with_weights=True):
    """MoE inputs: tokens, skewed top-k routing and bf16 expert weights.

    logits[t, e] = Gumbel noise + log p_e with p_e proportional to (e+1)**-1.1
    (a Zipf-like expert load); each token takes its top-k experts without
    replacement, with weights = softmax over all E logits evaluated at the chosen
    experts (not renormalised).  W13[e] = [gate rows; up rows] is [2*inter, H],
    W2[e] is [H, inter], both ~ N(0, 0.02).
    """
    x = _normal((T, H), 0.0, 1.0, seed, 40).to(torch.bfloat16)
    u = torch.rand(T, E, generator=_gen(seed, 41), dtype=torch.float64)
    u = u.clamp_(1e-300, 1.0 - 1e-16)
    gumbel = -torch.log(-torch.log(u))
    p = torch.tensor([(e + 1) ** -1.1 for e in range(E)], dtype=torch.float64)
    p = p / p.sum()
    logits = gumbel + torch.log(p)[None, :]
    top = torch.topk(logits, topk, dim=1)
    probs = torch.softmax(logits, dim=1)
    ids = top.indices.to(torch.int32)
    w = torch.gather(probs, 1, top.indices).to(torch.float32)
    out = dict(x=x, topk_ids=ids, topk_w=w, E=E, topk=topk, inter=inter, H=H, T=T,
               logits=logits.to(torch.float32))
    if with_weights:
        out["w13"] = _normal((E, 2 * inter, H), 0.0, 0.02, seed, 42).to(torch.bfloat16)
        out["w2"] = _normal((E, H, inter), 0.0, 0.02, seed, 43).to(torch.bfloat16)
    return out


def fp8_block_matrix(N, K, seed=0, stream=50, zero_frac=0.001, block=128):
    """One FP8-block-scaled weight: E4M3 codes of N(0,1) samples (round to nearest,
    saturating cast), block scales exp(U(ln 1e-4, ln 1e-2)) of shape
    [ceil(N/128), ceil(K/128)], and round(zero_frac*N) all-zero rows (seeded).
    Returns (codes uint8 [N,K] torch, scale_inv float32 torch, zero_rows torch).
    """
    v = torch.randn(N, K, generator=_gen(seed, stream), dtype=torch.float32)
    codes = v.to(torch.float8_e4m3fn).view(torch.uint8)
    nb_r, nb_c = math.ceil(N / block), math.ceil(K / block)
    lu = torch.rand(nb_r, nb_c, generator=_gen(seed, stream + 1), dtype=torch.float64)
    sinv = torch.exp(math.log(1e-4) + lu * (math.log(1e-2) - math.log(1e-4))).to(torch.float32)
    nz = int(round(zero_frac * N))
    zero_rows = torch.randperm(N, generator=_gen(seed, stream + 2))[:nz]
    codes[zero_rows] = 0
    return codes, sinv, zero_rows


def requant_workload(n_big=64, n_ragged=8, big=(6144, 4096), ragged=(3000, 1500), seed=0):
    """The batched requantization set: n_big [6144,4096] plus n_ragged [3000,1500] matrices."""
    mats = []
    for i in range(n_big):
        mats.append(fp8_block_matrix(big[0], big[1], seed=seed, stream=1000 + 3 * i))
    for i in range(n_ragged):
        mats.append(fp8_block_matrix(ragged[0], ragged[1], seed=seed, stream=5000 + 3 * i))
    return mats
