"""The bounds-checked build (libw8a8_debug.so, -DW8A8_DEBUG) on odd shapes.

Its kernels check the index invariants of their global-memory accesses and record a
violated one in a registered device word instead of trapping.  These cases run the hot path
through that build on shapes that exercise every tail: M = 1, 3, 17 token rows, K = 16, 48,
1040, 1500 and 3088, N = 5, 257, 520, a K-split launch, the requantizer's three row paths, a
grouped GEMM with empty segments and a small MoE layer.  Results must equal the oracle as in
the release build, and the error word must stay 0.
"""

import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_quantized_gb300 as w8
from w8a8_int8_quantized_gb300 import _binding
from w8a8_int8_quantized_gb300 import build as wbuild
from w8a8_int8_quantized_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module")
def debug_lib():
    L = _binding.load_library(wbuild.build(debug=True))
    assert L.w8a8_debug_build() == 1
    word = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert L.w8a8_debug_set_error_word(_binding._ptr(word)) == 0
    yield L, word
    L.w8a8_debug_set_error_word(None)


def _check_word(word):
    torch.cuda.synchronize()
    assert int(word.item()) == 0, f"bounds check site {int(word.item())} failed"


@pytest.mark.parametrize("M,K", [(1, 16), (3, 48), (17, 1500), (17, 1040)])
@pytest.mark.parametrize("mode", ["dyn_sym", "dyn_asym"])
def test_debug_quantize_act(debug_lib, M, K, mode):
    L, word = debug_lib
    x = wl.llama_activations(M, K, seed=M + K)
    with _binding.using_library(L):
        q, s, z = w8.quantize_act(x.to(DEV), mode)
    _check_word(word)
    xf = x.float().numpy()
    if mode == "dyn_sym":
        rq, rs = oracle.quantize_act_dynamic_symmetric(xf)
        np.testing.assert_array_equal(q.cpu().numpy(), rq)
        np.testing.assert_array_equal(s.cpu().numpy(), rs)
    else:
        rq, rs, rz = oracle.quantize_act_dynamic_asymmetric(xf)
        np.testing.assert_array_equal(q.cpu().numpy(), rq)
        np.testing.assert_array_equal(z.cpu().numpy(), rz)


@pytest.mark.parametrize("M,N,K", [(1, 5, 16), (3, 257, 48), (17, 520, 1040), (3, 520, 1040), (17, 257, 3088)])
@pytest.mark.parametrize("engine", [0, 1])
def test_debug_linear(debug_lib, M, N, K, engine):
    """Both GEMM engines (auto: warp MMA for M <= 16; 1: tcgen05), with the K-split scratch
    the binding adds where a launch splits (M = 17, K = 3088)."""
    L, word = debug_lib
    x = wl.llama_activations(M, K, seed=M * N + K)
    w = wl.weight_bf16(N, K, seed=N + K)
    b = wl.weight_bf16(1, N, seed=N, std=0.1)[0]
    with _binding.using_library(L):
        L.w8a8_set_gemm_engine(engine)
        try:
            wq, sw = w8.quantize_weight(w.to(DEV))
            y = w8.linear(x.to(DEV), wq, sw, bias=b.to(DEV))
        finally:
            L.w8a8_set_gemm_engine(0)
    _check_word(word)
    rq, rs = oracle.quantize_weight_per_channel(w.float().numpy())
    r = oracle.w8a8_linear(wl.bits(x), rq, rs, bias_bits=wl.bits(b))
    np.testing.assert_array_equal(_bits(y), r["y_bits"])


@pytest.mark.parametrize("N,K", [(5, 17), (300, 1500), (9, 4096)])
def test_debug_fp8_requant(debug_lib, N, K):
    """The generic byte path (K = 17), the word path (K = 1500) and the bulk-copy ring (K = 4096)."""
    L, word = debug_lib
    codes, sinv, _ = wl.fp8_block_matrix(N, K, seed=11, stream=N + K, zero_frac=0.05)
    with _binding.using_library(L):
        q, s = w8.fp8block_to_int8_rowwise(codes.to(DEV), sinv.to(DEV))
    _check_word(word)
    rq, rs, bad = oracle.fp8_block_to_int8_rowwise(codes.numpy(), sinv.numpy())
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)


def test_debug_grouped_and_moe(debug_lib):
    L, word = debug_lib
    E, N, K = 5, 257, 48
    seg = torch.tensor([0, 0, 130, 130, 131, 300], dtype=torch.int64)
    xq = torch.randint(-127, 128, (300, K), dtype=torch.int8)
    wq = torch.randint(-127, 128, (E, N, K), dtype=torch.int8)
    sx = torch.rand(300, dtype=torch.float32)
    sw = torch.rand(E, N, dtype=torch.float32) * 1e-3
    T, H, Ex, k, inter = 40, 256, 8, 2, 128
    d = wl.moe_workload(T=T, H=H, E=Ex, topk=k, inter=inter, seed=3)
    ids = d["topk_ids"].numpy()
    tok, slot, sg = oracle.moe_sort(ids, Ex)
    row_of = np.zeros((T, k), np.int64)
    row_of[tok, slot] = np.arange(len(tok))
    with _binding.using_library(L):
        y = w8.grouped_mm(xq.to(DEV), sx.to(DEV), wq.to(DEV), sw.to(DEV), seg.to(DEV))
        w13q, s13 = w8.quantize_weight(d["w13"].reshape(Ex * 2 * inter, H).to(DEV))
        w2q, s2 = w8.quantize_weight(d["w2"].reshape(Ex * H, inter).to(DEV))
        ym, h, o = w8.moe_forward(d["x"].to(DEV), torch.from_numpy(tok).to(DEV), torch.from_numpy(sg).to(DEV),
                                  torch.from_numpy(row_of).to(DEV), d["topk_w"].to(DEV), w13q.view(Ex, 2 * inter, H),
                                  s13.view(Ex, 2 * inter), w2q.view(Ex, H, inter), s2.view(Ex, H))
    _check_word(word)
    for e in range(E):
        a, b = int(seg[e]), int(seg[e + 1])
        if a == b:
            continue
        acc = oracle.int8_gemm(xq[a:b].numpy(), wq[e].numpy())
        yb, _ = oracle.scaled_mm_epilogue(acc, sx[a:b].numpy(), sw[e].numpy())
        np.testing.assert_array_equal(_bits(y[a:b]), yb)
    r = oracle.moe_forward(wl.bits(d["x"]), ids, d["topk_w"].numpy(), w13q.view(Ex, 2 * inter, H).cpu().numpy(),
                           s13.view(Ex, 2 * inter).cpu().numpy(), w2q.view(Ex, H, inter).cpu().numpy(),
                           s2.view(Ex, H).cpu().numpy())
    np.testing.assert_array_equal(_bits(h), r["h_bits"])
