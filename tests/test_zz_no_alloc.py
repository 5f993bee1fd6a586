"""w8a8_scaled_mm_noalloc, the allocation-free GEMM entry point, against w8a8_scaled_mm.

Callers that cannot allocate device memory (no allocator of their own to lend, or no
cudaMalloc allowed on their path) use w8a8_scaled_mm_noalloc, which stages activations in a
library-owned device buffer instead of a caller workspace.  Its output must equal the
workspace entry point's, call after call, since every call shares and rewrites that buffer.
This file is collected last so a failure here never hides the other tests' results.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_quantized_gb300 as w8
from w8a8_int8_quantized_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
P = ctypes.c_void_p


def _ptr(t):
    return None if t is None else P(t.data_ptr())


def _within_tolerance(y, y_ref):
    a = y.float().cpu().numpy().astype(np.float64)
    r = y_ref.float().cpu().numpy().astype(np.float64)
    rownorm = np.linalg.norm(r, axis=1, keepdims=True)
    err = np.abs(a - r)
    return bool(np.all((err <= 1e-2 * np.abs(r)) | (err <= 1e-3 * rownorm)))


def _case(M, N, K, seed, act):
    x = (wl.asym_activations if act == "dyn_asym" else wl.llama_activations)(M, K, seed=seed)
    w = wl.weight_bf16(N, K, seed=seed + 1)
    b = wl.weight_bf16(1, N, seed=seed + 2, std=0.1)[0].to(DEV)
    wq, sw, adj = w8.quantize_weight(w.to(DEV), with_azp_adj=True)
    xq, sx, zp = w8.quantize_act(x.to(DEV), act)
    return xq, wq, sx, sw, zp, (adj if act == "dyn_asym" else None), b


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    lib = w8.lib()
    stream = P(torch.cuda.current_stream().cuda_stream)
    # two calls in a row with different shapes and modes: the second reuses the shared buffer
    for M, N, K, act, seed in [(300, 520, 2048, "dyn_sym", 3), (1000, 384, 4096, "dyn_asym", 4)]:
        xq, wq, sx, sw, zp, adj, b = _case(M, N, K, seed, act)
        mode = 1 if act == "dyn_asym" else 0
        y_ref = w8.scaled_mm(xq, wq, sx, sw, act, zp=zp, azp_adj=adj, bias=b)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = lib.w8a8_scaled_mm_noalloc(_ptr(xq), _ptr(wq), M, N, K, mode, _ptr(sx), _ptr(zp), _ptr(adj), 0,
                                        _ptr(sw), _ptr(b), _ptr(y), _ptr(status), stream)
        assert rc == 0, lib.w8a8_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert _within_tolerance(y, y_ref)
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
        # and against the oracle on a few rows
        rows = np.array([0, M // 2, M - 1])
        acc = oracle.int8_gemm(xq.cpu().numpy()[rows], wq.cpu().numpy())
        kw = {}
        if act == "dyn_asym":
            kw = dict(zp=zp.cpu().numpy()[rows], adj=adj.cpu().numpy())
        yb, _ = oracle.scaled_mm_epilogue(acc, sx.cpu().numpy()[rows], sw.cpu().numpy(),
                                          bias_bits=wl.bits(b.cpu()), **kw)
        got = y.cpu()[torch.from_numpy(rows)].contiguous().view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(got, yb)


def test_noalloc_rejects_problems_beyond_its_buffer():
    lib = w8.lib()
    stream = P(torch.cuda.current_stream().cuda_stream)
    M, K, N = 8192, 4096, 16  # 64 MiB of staged codes: more than the 36 MiB buffer
    xq = torch.zeros((M, K), dtype=torch.int8, device=DEV)
    wq = torch.zeros((N, K), dtype=torch.int8, device=DEV)
    sx = torch.ones(M, dtype=torch.float32, device=DEV)
    sw = torch.ones(N, dtype=torch.float32, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    rc = lib.w8a8_scaled_mm_noalloc(_ptr(xq), _ptr(wq), M, N, K, 0, _ptr(sx), None, None, 0, _ptr(sw), None,
                                    _ptr(y), None, stream)
    assert rc == 7  # W8A8_ERR_WORKSPACE


def test_noalloc_rejects_a_misaligned_bias():
    """The bf16 bias must be 2-byte aligned, as for w8a8_scaled_mm: an odd pointer is refused
    before anything is launched."""
    lib = w8.lib()
    stream = P(torch.cuda.current_stream().cuda_stream)
    M, N, K = 32, 64, 256
    xq = torch.zeros((M, K), dtype=torch.int8, device=DEV)
    wq = torch.zeros((N, K), dtype=torch.int8, device=DEV)
    sx = torch.ones(M, dtype=torch.float32, device=DEV)
    sw = torch.ones(N, dtype=torch.float32, device=DEV)
    bias = torch.zeros(N + 1, dtype=torch.bfloat16, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    odd = P(bias.data_ptr() + 1)
    rc = lib.w8a8_scaled_mm_noalloc(_ptr(xq), _ptr(wq), M, N, K, 0, _ptr(sx), None, None, 0, _ptr(sw), odd,
                                    _ptr(y), None, stream)
    assert rc == 3  # W8A8_ERR_MISALIGNED
