"""Run one kernel of the library repeatedly on a fixed, seeded case, for profilers.

    python -m w8a8_int8_quantized_gb300.profile_cases CASE [--reps R]

Cases (inputs drawn on the device with a seeded generator; nothing is checked here):
  quant          w8a8_quantize_act, dynamic symmetric, M=8192, K=4096
  quant_packed   w8a8_quantize_act_packed, dynamic symmetric, M=8192, K=4096
  quant_asym     w8a8_quantize_act, dynamic asymmetric, M=8192, K=4096
  quant_asym_mean  the same on nonzero-mean rows N(0.5, 1) (many exact rounding ties)
  wquant         w8a8_quantize_weight (+ azp_adj), N=28672, K=4096
  wquant_o       the same on the o-projection weight, N=K=4096
  requant        fp8block_to_int8_rowwise_batched over 8 x [6144, 4096]
  gemm           w8a8_scaled_mm_packed, M=4096, N=28672, K=4096 (Llama-like activations, as the
                 bench: 1% outlier channels, so every tile runs the single fp32 pass)
  gemm_o         the same with N=4096
  gemm_chunked   M=4096, N=28672, K=4096 with N(0,1) activations: many rows' L1 norms exceed
                 2^17, so their tiles run the 1024-K chunked mode
  small          w8a8_linear at M=16 (warp-MMA engine), N=28672, K=4096
  decode1_o      w8a8_linear on one bf16 token row (quantizer fused into the small-M GEMM), N=K=4096
  decode1_qkv    the same with N=6144
  decode8        w8a8_scaled_mm on 8 quantized token rows (staged small-M kernel), N=28672, K=4096
  moe            the MoE layer: 4096 tokens, 32 experts, top-4 (expert weights' sums of squares given)
  moe_routed     the same layer behind w8a8_moe_route (router logits in, every step on the GPU)
  route          w8a8_moe_route alone: 4096 tokens, 32 experts, top-4
  requant_word   fp8block_to_int8_rowwise_batched over 8 x [3000, 1500] (rows on 4-byte words)
  max_scale      w8a8_requantize_max_scale on a fused q/k/v weight [4096+1024+1024, 4096]
  asym_linear    w8a8_linear, dynamic asymmetric, M=N=K=4096, with the weight's sums of squares
  split          w8a8_linear at M=128 on the down projection (N=4096, K=14336) with the K-split
                 scratch: 16 tiles in 4 parts each, then the reduce kernel

Every case uses a few GB of device memory at most, so a profiler capture of one launch
stays small.
"""

import argparse
import math

import torch

import w8a8_int8_quantized_gb300 as w8
from w8a8_int8_quantized_gb300 import workloads as wl


def _gen(seed):
    return torch.Generator(device="cuda").manual_seed(seed)


def _bf16(shape, std, seed):
    return torch.randn(*shape, device="cuda", generator=_gen(seed)).mul_(std).to(torch.bfloat16)


def case_fn(name):
    dev = "cuda"
    if name == "quant_asym_mean":
        x = torch.randn(8192, 4096, device=dev, generator=_gen(1)).add_(0.5).to(torch.bfloat16)
        return lambda: w8.quantize_act(x, "dyn_asym")
    if name == "wquant_o":
        w = _bf16((4096, 4096), 0.02, 2)
        return lambda: w8.quantize_weight(w, with_azp_adj=True)
    if name in ("quant", "quant_packed", "quant_asym"):
        x = _bf16((8192, 4096), 1.0, 1)
        if name == "quant":
            return lambda: w8.quantize_act(x, "dyn_sym")
        if name == "quant_asym":
            return lambda: w8.quantize_act(x, "dyn_asym")
        buf = torch.empty(w8.act_packed_size(8192, 4096), dtype=torch.uint8, device=dev)
        return lambda: w8.quantize_act_packed(x, "dyn_sym", buf=buf)
    if name == "wquant":
        w = _bf16((28672, 4096), 0.02, 2)
        return lambda: w8.quantize_weight(w, with_azp_adj=True)
    if name == "requant":
        g = _gen(3)
        mats = []
        for _ in range(8):
            c = torch.randn(6144, 4096, device=dev, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
            s = torch.exp(torch.empty(48, 32, device=dev).uniform_(math.log(1e-4), math.log(1e-2), generator=g))
            mats.append((c, s))
        outs = [(torch.empty(c.shape, dtype=torch.int8, device=dev), torch.empty(c.shape[0], device=dev))
                for c, _ in mats]
        return lambda: w8.fp8block_to_int8_rowwise_batched(mats, outs)
    if name in ("gemm", "gemm_o", "gemm_chunked"):
        N = 4096 if name == "gemm_o" else 28672
        x = _bf16((4096, 4096), 1.0, 4) if name == "gemm_chunked" else wl.llama_activations(4096, 4096, seed=4).to(dev)
        wq = torch.randint(-127, 128, (N, 4096), dtype=torch.int8, device=dev, generator=_gen(5))
        sw = torch.rand(N, device=dev, generator=_gen(6)).mul_(1e-3)
        pa = w8.quantize_act_packed(x)
        y = torch.empty(4096, N, dtype=torch.bfloat16, device=dev)
        return lambda: w8.scaled_mm_packed(pa, wq, sw, out=y)
    if name == "small":
        x = _bf16((16, 4096), 1.0, 7)
        wq = torch.randint(-127, 128, (28672, 4096), dtype=torch.int8, device=dev, generator=_gen(8))
        sw = torch.rand(28672, device=dev, generator=_gen(9)).mul_(1e-3)
        ws = torch.empty(w8.linear_workspace_size(16, 4096), dtype=torch.uint8, device=dev)
        y = torch.empty(16, 28672, dtype=torch.bfloat16, device=dev)
        return lambda: w8.linear(x, wq, sw, workspace=ws, out=y)
    if name in ("decode1_o", "decode1_qkv"):
        N = 4096 if name == "decode1_o" else 6144
        x = _bf16((1, 4096), 1.0, 25)
        wq = torch.randint(-127, 128, (N, 4096), dtype=torch.int8, device=dev, generator=_gen(26))
        sw = torch.rand(N, device=dev, generator=_gen(27)).mul_(1e-3)
        ws = torch.empty(w8.linear_workspace_size(1, 4096), dtype=torch.uint8, device=dev)
        y = torch.empty(1, N, dtype=torch.bfloat16, device=dev)
        return lambda: w8.linear(x, wq, sw, workspace=ws, out=y)
    if name == "decode8":
        xq = torch.randint(-127, 128, (8, 4096), dtype=torch.int8, device=dev, generator=_gen(18))
        sx = torch.rand(8, device=dev, generator=_gen(19)).mul_(1e-2)
        wq = torch.randint(-127, 128, (28672, 4096), dtype=torch.int8, device=dev, generator=_gen(20))
        sw = torch.rand(28672, device=dev, generator=_gen(21)).mul_(1e-3)
        y = torch.empty(8, 28672, dtype=torch.bfloat16, device=dev)
        return lambda: w8.scaled_mm(xq, wq, sx, sw, "dyn_sym", out=y)
    if name == "moe":
        T, H, E, k, inter = 4096, 4096, 32, 4, 1408
        g = _gen(10)
        ids = torch.stack([torch.randperm(E, device=dev, generator=g)[:k] for _ in range(T)]).reshape(-1)
        order = torch.argsort(ids, stable=True)
        seg = torch.zeros(E + 1, dtype=torch.int64, device=dev)
        seg[1:] = torch.cumsum(torch.bincount(ids, minlength=E), 0)
        row_of = torch.empty(T * k, dtype=torch.int64, device=dev)
        row_of[order] = torch.arange(T * k, device=dev)
        x = _bf16((T, H), 1.0, 11)
        w13q, s13 = w8.quantize_weight(_bf16((E * 2 * inter, H), 0.02, 12))
        w2q, s2 = w8.quantize_weight(_bf16((E * H, inter), 0.02, 13))
        tw = torch.rand(T, k, device=dev, generator=g)
        args = (x, order // k, seg, row_of.view(T, k), tw, w13q.view(E, 2 * inter, H), s13.view(E, 2 * inter),
                w2q.view(E, H, inter), s2.view(E, H))
        kw = dict(w13_sumsq=w8.weight_sumsq(w13q).view(E, 2 * inter), w2_sumsq=w8.weight_sumsq(w2q).view(E, H))
        return lambda: w8.moe_forward(*args, **kw)
    if name in ("moe_routed", "route"):
        T, H, E, k, inter = 4096, 4096, 32, 4, 1408
        logits = wl.moe_workload(T=T, H=64, E=E, topk=k, inter=64, seed=0, with_weights=False)["logits"].to(dev)
        ws = torch.empty(max(int(w8.lib().w8a8_moe_route_workspace_size(T, E, k)), 4), dtype=torch.uint8, device=dev)
        if name == "route":
            return lambda: w8.moe_route(logits, k, workspace=ws)
        x = _bf16((T, H), 1.0, 11)
        w13q, s13 = w8.quantize_weight(_bf16((E * 2 * inter, H), 0.02, 12))
        w2q, s2 = w8.quantize_weight(_bf16((E * H, inter), 0.02, 13))

        w13sq, w2sq = w8.weight_sumsq(w13q).view(E, 2 * inter), w8.weight_sumsq(w2q).view(E, H)

        def layer():
            ids, tw, seg, row_index, row_of = w8.moe_route(logits, k, workspace=ws)
            return w8.moe_forward(x, row_index, seg, row_of, tw, w13q.view(E, 2 * inter, H), s13.view(E, 2 * inter),
                                  w2q.view(E, H, inter), s2.view(E, H), w13_sumsq=w13sq, w2_sumsq=w2sq)
        return layer
    if name == "requant_word":
        g = _gen(14)
        mats = []
        for _ in range(8):
            c = torch.randn(3000, 1500, device=dev, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
            s = torch.exp(torch.empty(24, 12, device=dev).uniform_(math.log(1e-4), math.log(1e-2), generator=g))
            mats.append((c, s))
        outs = [(torch.empty(c.shape, dtype=torch.int8, device=dev), torch.empty(c.shape[0], device=dev))
                for c, _ in mats]
        return lambda: w8.fp8block_to_int8_rowwise_batched(mats, outs)
    if name == "max_scale":
        wq = torch.randint(-127, 128, (6144, 4096), dtype=torch.int8, device=dev, generator=_gen(15))
        sc = torch.tensor([1.1e-3, 1.7e-3, 1.3e-3], dtype=torch.float32, device=dev)
        return lambda: w8.requantize_max_scale(wq, sc, [4096, 1024, 1024])
    if name == "asym_linear":
        x = wl.asym_activations(4096, 4096, seed=16).to(dev)
        wq, sw, adj, wsq = w8.quantize_weight(_bf16((4096, 4096), 0.02, 17), with_azp_adj=True, with_sumsq=True)
        ws = torch.empty(w8.linear_workspace_size(4096, 4096, "dyn_asym"), dtype=torch.uint8, device=dev)
        y = torch.empty(4096, 4096, dtype=torch.bfloat16, device=dev)
        return lambda: w8.linear(x, wq, sw, act_mode="dyn_asym", azp_adj=adj, w_sumsq=wsq, workspace=ws, out=y)
    if name == "split":
        x = wl.llama_activations(128, 14336, seed=22).to(dev)
        wq = torch.randint(-127, 128, (4096, 14336), dtype=torch.int8, device=dev, generator=_gen(23))
        sw = torch.rand(4096, device=dev, generator=_gen(24)).mul_(1e-3)
        ws = torch.empty(w8.linear_workspace_size(128, 14336, "dyn_sym", 4096), dtype=torch.uint8, device=dev)
        y = torch.empty(128, 4096, dtype=torch.bfloat16, device=dev)
        return lambda: w8.linear(x, wq, sw, workspace=ws, out=y)
    raise SystemExit(f"unknown case {name}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--reps", type=int, default=5)
    a = ap.parse_args()
    fn = case_fn(a.case)
    for _ in range(a.reps):
        fn()
    torch.cuda.synchronize()
    print(f"{a.case}: ran {a.reps} times")


if __name__ == "__main__":
    main()
