"""ctypes binding of libw8a8.so: argument marshalling only.

Every function here checks tensor devices/dtypes/shapes, allocates outputs with torch
(device memory is PyTorch's job), and calls the C entry point of the same name on the
current CUDA stream.  All arithmetic runs in the library's CUDA kernels; if the library
is missing or fails to load, every call raises.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw8a8.so")

ACT_DYN_TOKEN_SYM = 0
ACT_DYN_TOKEN_ASYM = 1
ACT_STATIC_TENSOR_SYM = 2
ACT_STATIC_TENSOR_ASYM = 3
W_CHANNEL = 0
W_TENSOR = 1

_ACT_NAMES = {"dyn_sym": 0, "dyn_asym": 1, "static_sym": 2, "static_asym": 3}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_SZ = ctypes.c_size_t

# name -> (restype, argtypes)
SIGNATURES = {
    "w8a8_status_string": (ctypes.c_char_p, [_I]),
    "w8a8_version": (_I, []),
    "w8a8_set_gemm_engine": (_I, [_I]),
    "w8a8_test_requant_wait_fault": (_I, [ctypes.c_uint32, ctypes.c_uint64]),
    "w8a8_debug_set_error_word": (_I, [_P]),
    "w8a8_debug_build": (_I, []),
    "w8a8_quantize_act": (_I, [_P, _I64, _I64, _I64, _I, _P, _P, _P, _P]),
    "w8a8_scaled_mm_workspace_size": (_SZ, [_I64, _I64]),
    "w8a8_scaled_mm": (_I, [_P, _P, _I64, _I64, _I64, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "w8a8_linear_workspace_size": (_SZ, [_I64, _I64, _I]),
    "w8a8_splitk_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "w8a8_linear": (_I, [_P, _I64, _I64, _I64, _I, _P, _P, _P, _I64, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "w8a8_quantize_weight": (_I, [_P, _I64, _I64, _P, _P, _P, _P, _P]),
    "w8a8_weight_sumsq": (_I, [_P, _I64, _I64, _P, _P]),
    "w8a8_azp_adj": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "fp8block_to_int8_rowwise": (_I, [_P, _P, _I64, _I64, _P, _P, _P, _P]),
    "fp8block_to_int8_rowwise_batched": (_I, [_I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "fp8block_to_int8_rowwise_batched_adj": (_I, [_I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "w8a8_requantize_max_scale": (_I, [_P, _I64, _I64, _P, _P, _I, _P, _P, _P]),
    "w8a8_moe_route_workspace_size": (_SZ, [_I64, _I, _I]),
    "w8a8_moe_route": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "w8a8_grouped_mm_workspace_size": (_SZ, [_I64, _I64]),
    "w8a8_grouped_mm": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _P, _SZ, _P, _P]),
    "w8a8_moe_quantize_gather": (_I, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P]),
    "w8a8_silu_mul_quant": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "w8a8_moe_combine": (_I, [_P, _P, _P, _I64, _I, _I64, _P, _P]),
    "w8a8_act_packed_size": (_SZ, [_I64, _I64]),
    "w8a8_quantize_act_packed": (_I, [_P, _I64, _I64, _I64, _I, _P, _P, _P, _P]),
    "w8a8_scaled_mm_packed": (_I, [_P, _P, _I64, _I64, _I64, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "w8a8_grouped_mm_packed": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _P, _P]),
    "w8a8_moe_quantize_gather_packed": (_I, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P]),
    "w8a8_moe_quantize_scatter_packed": (_I, [_P, _I64, _I64, _I64, _P, _I, _I64, _P, _P, _P]),
    "w8a8_silu_mul_quant_packed": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "w8a8_scaled_mm_noalloc": (_I, [_P, _P, _I64, _I64, _I64, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P]),
}

_lib = None


class W8A8Error(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


def load_library(path):
    """Load a build of the library (libw8a8.so, or the bounds-checked libw8a8_debug.so) with
    the C signatures declared."""
    L = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


def lib():
    """Load libw8a8.so (raises if it is not built or cannot be loaded)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m w8a8_int8_quantized_gb300.build`")
        _lib = load_library(LIB_PATH)
    return _lib


class using_library:
    """Context manager: every call of this module goes to library `L` (for example the
    bounds-checked build) until the block ends."""

    def __init__(self, L):
        self.L = L

    def __enter__(self):
        global _lib
        self.prev = lib()
        _lib = self.L
        return self.L

    def __exit__(self, *exc):
        global _lib
        _lib = self.prev
        return False


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(name, code):
    if code != 0:
        raise W8A8Error(name, code, lib().w8a8_status_string(code).decode())


def _need(t, dtype, name, dim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _mode(m):
    return _ACT_NAMES[m] if isinstance(m, str) else int(m)


def set_gemm_engine(engine):
    """0 automatic, 1 tcgen05, 2 warp-MMA (applies to the calling thread)."""
    _check("w8a8_set_gemm_engine", lib().w8a8_set_gemm_engine(int(engine)))


def quantize_act(x, mode="dyn_sym", scale=None, zp=None):
    """Quantize bf16 activations [M, K].  Returns (q int8, scale float32, zp int32|None)."""
    _need(x, torch.bfloat16, "x", 2)
    m = _mode(mode)
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if m in (ACT_DYN_TOKEN_SYM, ACT_DYN_TOKEN_ASYM):
        scale = torch.empty(M, dtype=torch.float32, device=x.device)
        zp = torch.empty(M, dtype=torch.int32, device=x.device) if m == ACT_DYN_TOKEN_ASYM else None
    else:
        _need(scale, torch.float32, "scale")
        if m == ACT_STATIC_TENSOR_ASYM:
            _need(zp, torch.int32, "zp")
    _check("w8a8_quantize_act", lib().w8a8_quantize_act(_ptr(x), M, K, K, m, _ptr(q), _ptr(scale), _ptr(zp),
                                                        _stream()))
    return q, scale, zp


def _workspace(nbytes, device, given):
    if given is not None:
        return given
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def scaled_mm(xq, wq, s_x, s_w, act_mode="dyn_sym", zp=None, azp_adj=None, w_mode=W_CHANNEL, bias=None,
              out=None, status=None, workspace=None, w_sumsq=None):
    """y[M, N] bf16 = epilogue(xq @ wq.T) (see w8a8_scaled_mm in include/w8a8.h)."""
    _need(xq, torch.int8, "xq", 2)
    _need(wq, torch.int8, "wq", 2)
    M, K = xq.shape
    N = wq.shape[0]
    if wq.shape[1] != K:
        raise ValueError("K mismatch")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    ws = _workspace(lib().w8a8_scaled_mm_workspace_size(M, K) + splitk_workspace_size(M, N, K), xq.device,
                    workspace)
    code = lib().w8a8_scaled_mm(_ptr(xq), _ptr(wq), M, N, K, _mode(act_mode), _ptr(s_x), _ptr(zp), _ptr(azp_adj),
                                int(w_mode), _ptr(s_w), _ptr(w_sumsq), _ptr(bias), _ptr(out), _ptr(ws), ws.numel(),
                                _ptr(status), _stream())
    _check("w8a8_scaled_mm", code)
    return out


def splitk_workspace_size(M, N, K):
    """Extra workspace bytes with which a GEMM of few tiles splits along K (0: no split)."""
    return int(lib().w8a8_splitk_workspace_size(M, N, K))


def linear_workspace_size(M, K, act_mode="dyn_sym", N=None):
    """Workspace of w8a8_linear; with N, including the K-split scratch for that shape."""
    n = int(lib().w8a8_linear_workspace_size(M, K, _mode(act_mode)))
    return n + (splitk_workspace_size(M, N, K) if N is not None else 0)


def linear(x, wq, s_w, act_mode="dyn_sym", input_scale=None, input_zero_point=None, azp_adj=None, bias=None,
           w_mode=W_CHANNEL, workspace=None, out=None, status=None, w_sumsq=None):
    """Whole W8A8 linear: y = epilogue(quant(x) @ wq.T)."""
    _need(x, torch.bfloat16, "x", 2)
    _need(wq, torch.int8, "wq", 2)
    M, K = x.shape
    N = wq.shape[0]
    m = _mode(act_mode)
    workspace = _workspace(linear_workspace_size(M, K, m, N), x.device, workspace)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    code = lib().w8a8_linear(_ptr(x), M, K, K, m, _ptr(input_scale), _ptr(input_zero_point), _ptr(wq), N,
                             int(w_mode), _ptr(s_w), _ptr(azp_adj), _ptr(w_sumsq), _ptr(bias), _ptr(out),
                             _ptr(workspace), workspace.numel(), _ptr(status), _stream())
    _check("w8a8_linear", code)
    return out


def quantize_weight(w, with_azp_adj=False, with_sumsq=False):
    """Per-channel symmetric int8 weight.  Returns (wq, s_w[, azp_adj][, w_sumsq])."""
    _need(w, torch.bfloat16, "w", 2)
    N, K = w.shape
    wq = torch.empty((N, K), dtype=torch.int8, device=w.device)
    s = torch.empty(N, dtype=torch.float32, device=w.device)
    adj = torch.empty(N, dtype=torch.int32, device=w.device) if with_azp_adj else None
    sq = torch.empty(N, dtype=torch.int32, device=w.device) if with_sumsq else None
    _check("w8a8_quantize_weight", lib().w8a8_quantize_weight(_ptr(w), N, K, _ptr(wq), _ptr(s), _ptr(adj), _ptr(sq),
                                                              _stream()))
    return (wq, s) + ((adj,) if with_azp_adj else ()) + ((sq,) if with_sumsq else ())


def weight_sumsq(wq):
    """int32 [N] row sums of squares of an int8 weight (the GEMM's optional w_sumsq)."""
    _need(wq, torch.int8, "wq", 2)
    N, K = wq.shape
    out = torch.empty(N, dtype=torch.int32, device=wq.device)
    _check("w8a8_weight_sumsq", lib().w8a8_weight_sumsq(_ptr(wq), N, K, _ptr(out), _stream()))
    return out


def azp_adj(wq, input_zero_point=None):
    """azp_adj[n] = (zp *) sum_k wq[n, k], int32."""
    _need(wq, torch.int8, "wq", 2)
    N, K = wq.shape
    out = torch.empty(N, dtype=torch.int32, device=wq.device)
    _check("w8a8_azp_adj", lib().w8a8_azp_adj(_ptr(wq), N, K, _ptr(input_zero_point), _ptr(out), _stream()))
    return out


def fp8block_to_int8_rowwise(codes, scale_inv, status=None):
    """FP8 E4M3 codes (uint8 [N, K]) + block scales -> (q int8 [N, K], s float32 [N])."""
    _need(codes, torch.uint8, "codes", 2)
    _need(scale_inv, torch.float32, "scale_inv", 2)
    N, K = codes.shape
    q = torch.empty((N, K), dtype=torch.int8, device=codes.device)
    s = torch.empty(N, dtype=torch.float32, device=codes.device)
    _check("fp8block_to_int8_rowwise", lib().fp8block_to_int8_rowwise(_ptr(codes), _ptr(scale_inv), N, K, _ptr(q),
                                                                      _ptr(s), _ptr(status), _stream()))
    return q, s


def fp8block_to_int8_rowwise_batched(mats, outs=None, status=None, azp_adj=False):
    """mats: list of (codes, scale_inv) CUDA tensors.  Returns list of (q, s), or of
    (q, s, azp_adj) when azp_adj is True (int32 [N] row sums of q, written in the same pass)."""
    n = len(mats)
    if outs is None:
        outs = []
        for c, _ in mats:
            o = (torch.empty(c.shape, dtype=torch.int8, device=c.device),
                 torch.empty(c.shape[0], dtype=torch.float32, device=c.device))
            if azp_adj:
                o = o + (torch.empty(c.shape[0], dtype=torch.int32, device=c.device),)
            outs.append(o)
    for c, si in mats:
        _need(c, torch.uint8, "codes", 2)
        _need(si, torch.float32, "scale_inv", 2)
    arr = ctypes.c_void_p * n
    ai = ctypes.c_int64 * n
    w = arr(*[c.data_ptr() for c, _ in mats])
    si = arr(*[s.data_ptr() for _, s in mats])
    Ns = ai(*[c.shape[0] for c, _ in mats])
    Ks = ai(*[c.shape[1] for c, _ in mats])
    qs = arr(*[o[0].data_ptr() for o in outs])
    ss = arr(*[o[1].data_ptr() for o in outs])
    if azp_adj:
        for o in outs:
            _need(o[2], torch.int32, "azp_adj", 1)
        adj = arr(*[o[2].data_ptr() for o in outs])
        code = lib().fp8block_to_int8_rowwise_batched_adj(
            n, ctypes.cast(w, _P), ctypes.cast(si, _P), ctypes.cast(Ns, _P), ctypes.cast(Ks, _P),
            ctypes.cast(qs, _P), ctypes.cast(ss, _P), ctypes.cast(adj, _P), _ptr(status), _stream())
    else:
        code = lib().fp8block_to_int8_rowwise_batched(n, ctypes.cast(w, _P), ctypes.cast(si, _P),
                                                      ctypes.cast(Ns, _P), ctypes.cast(Ks, _P),
                                                      ctypes.cast(qs, _P), ctypes.cast(ss, _P), _ptr(status),
                                                      _stream())
    _check("fp8block_to_int8_rowwise_batched", code)
    return outs


def moe_route(logits, topk, workspace=None):
    """Router logits float32 [T, E] -> (topk_ids int32 [T, k], topk_w float32 [T, k],
    seg_offsets int64 [E+1], row_index int64 [T*k], row_of int64 [T, k]): top-k by logit
    (ties to the lower expert), softmax weights over all experts, and the stable counting
    sort of the routed rows by expert -- the inputs moe_forward takes."""
    _need(logits, torch.float32, "logits", 2)
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    T, E = logits.shape
    dev = logits.device
    ids = torch.empty((T, topk), dtype=torch.int32, device=dev)
    w = torch.empty((T, topk), dtype=torch.float32, device=dev)
    seg = torch.empty(E + 1, dtype=torch.int64, device=dev)
    row_index = torch.empty(T * topk, dtype=torch.int64, device=dev)
    row_of = torch.empty((T, topk), dtype=torch.int64, device=dev)
    need = lib().w8a8_moe_route_workspace_size(T, E, topk)
    if workspace is None:
        workspace = torch.empty(max(need, 4), dtype=torch.uint8, device=dev)
    _check("w8a8_moe_route", lib().w8a8_moe_route(_ptr(logits), T, E, topk, _ptr(ids), _ptr(w), _ptr(seg),
                                                  _ptr(row_index), _ptr(row_of), _ptr(workspace),
                                                  workspace.numel(), _stream()))
    return ids, w, seg, row_index, row_of


def requantize_max_scale(wq, scales, logical_widths, status=None):
    """Fused weight wq int8 [N, K] with per-partition tensor scales (float32 [P]) and
    logical_widths (P row counts summing to N): requantized IN PLACE against the largest
    scale, which is returned as a float32 [1] tensor."""
    _need(wq, torch.int8, "wq", 2)
    _need(scales, torch.float32, "scales", 1)
    if not wq.is_contiguous() or not scales.is_contiguous():
        raise ValueError("wq and scales must be contiguous")
    N, K = wq.shape
    widths = [int(w) for w in logical_widths]
    arr = (ctypes.c_int64 * len(widths))(*widths)
    s_max = torch.empty(1, dtype=torch.float32, device=wq.device)
    _check("w8a8_requantize_max_scale",
           lib().w8a8_requantize_max_scale(_ptr(wq), N, K, _ptr(scales), ctypes.cast(arr, _P),
                                           len(widths), _ptr(s_max), _ptr(status), _stream()))
    return s_max


def grouped_mm(xq_sorted, s_x, w, s_w, seg_offsets, out=None, status=None, workspace=None, w_sumsq=None):
    """Per-segment W8A8 GEMMs: rows [seg[e], seg[e+1]) use expert e's weight.  w_sumsq: int32
    [E, N] row sums of squares of the expert weights (enables the Cauchy-Schwarz test)."""
    _need(xq_sorted, torch.int8, "xq_sorted", 2)
    _need(w, torch.int8, "w", 3)
    _need(seg_offsets, torch.int64, "seg_offsets", 1)
    R, K = xq_sorted.shape
    E, N, K2 = w.shape
    if K2 != K or seg_offsets.numel() != E + 1:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((R, N), dtype=torch.bfloat16, device=w.device)
    ws = _workspace(lib().w8a8_grouped_mm_workspace_size(R, K), w.device, workspace)
    code = lib().w8a8_grouped_mm(_ptr(xq_sorted), _ptr(s_x), _ptr(w), _ptr(s_w), _ptr(w_sumsq), _ptr(seg_offsets), E,
                                 R, N, K, _ptr(out), _ptr(ws), ws.numel(), _ptr(status), _stream())
    _check("w8a8_grouped_mm", code)
    return out


def moe_quantize_gather(x, row_index):
    _need(x, torch.bfloat16, "x", 2)
    _need(row_index, torch.int64, "row_index", 1)
    T, K = x.shape
    R = row_index.numel()
    q = torch.empty((R, K), dtype=torch.int8, device=x.device)
    s = torch.empty(R, dtype=torch.float32, device=x.device)
    _check("w8a8_moe_quantize_gather", lib().w8a8_moe_quantize_gather(_ptr(x), T, K, K, _ptr(row_index), R, _ptr(q),
                                                                      _ptr(s), _stream()))
    return q, s


def silu_mul_quant(h):
    _need(h, torch.bfloat16, "h", 2)
    R, twoI = h.shape
    inter = twoI // 2
    q = torch.empty((R, inter), dtype=torch.int8, device=h.device)
    s = torch.empty(R, dtype=torch.float32, device=h.device)
    _check("w8a8_silu_mul_quant", lib().w8a8_silu_mul_quant(_ptr(h), R, inter, _ptr(q), _ptr(s), _stream()))
    return q, s


def moe_combine(out_rows, row_of, topk_w):
    _need(out_rows, torch.bfloat16, "out", 2)
    _need(row_of, torch.int64, "row_of", 2)
    _need(topk_w, torch.float32, "topk_w", 2)
    T, k = row_of.shape
    H = out_rows.shape[1]
    y = torch.empty((T, H), dtype=torch.bfloat16, device=out_rows.device)
    _check("w8a8_moe_combine", lib().w8a8_moe_combine(_ptr(out_rows), _ptr(row_of), _ptr(topk_w), T, k, H, _ptr(y),
                                                      _stream()))
    return y


class PackedActivations:
    """Quantized activations in the tensor-core engine's format (fp16 codes, row L1 norms and,
    for the affine modes, row sums of squares).

    buf: uint8 CUDA tensor of w8a8_act_packed_size(M, K) bytes; scale / zp as produced by the
    quantizer.  codes(), norms() and sumsq() are views for inspection.
    """

    def __init__(self, buf, M, K, scale, zp=None):
        self.buf, self.M, self.K, self.scale, self.zp = buf, M, K, scale, zp

    def codes(self):
        return self.buf[: self.M * self.K * 2].view(torch.float16).view(self.M, self.K)

    def norms(self):
        off = (self.M * self.K * 2 + 255) // 256 * 256
        return self.buf[off: off + 4 * self.M].view(torch.int32)

    def sumsq(self):
        off = (self.M * self.K * 2 + 255) // 256 * 256 + 4 * self.M
        return self.buf[off: off + 4 * self.M].view(torch.int32)


def act_packed_size(M, K):
    return int(lib().w8a8_act_packed_size(M, K))


def _packed_buf(M, K, device, buf):
    return buf if buf is not None else torch.empty(max(act_packed_size(M, K), 256), dtype=torch.uint8, device=device)


def quantize_act_packed(x, mode="dyn_sym", scale=None, zp=None, buf=None):
    """Quantize bf16 activations into the packed format.  Returns PackedActivations."""
    _need(x, torch.bfloat16, "x", 2)
    m = _mode(mode)
    M, K = x.shape
    if m in (ACT_DYN_TOKEN_SYM, ACT_DYN_TOKEN_ASYM):
        scale = torch.empty(M, dtype=torch.float32, device=x.device)
        zp = torch.empty(M, dtype=torch.int32, device=x.device) if m == ACT_DYN_TOKEN_ASYM else None
    pk = _packed_buf(M, K, x.device, buf)
    _check("w8a8_quantize_act_packed", lib().w8a8_quantize_act_packed(_ptr(x), M, K, K, m, _ptr(pk), _ptr(scale),
                                                                      _ptr(zp), _stream()))
    return PackedActivations(pk, M, K, scale, zp)


def scaled_mm_packed(pa, wq, s_w, act_mode="dyn_sym", azp_adj=None, w_mode=W_CHANNEL, bias=None, out=None,
                     status=None, w_sumsq=None, split_ws=None):
    """y = epilogue(A @ wq.T) with A given as PackedActivations (scales taken from it).
    split_ws: optional uint8 CUDA tensor of splitk_workspace_size(M, N, K) bytes."""
    _need(wq, torch.int8, "wq", 2)
    N = wq.shape[0]
    if out is None:
        out = torch.empty((pa.M, N), dtype=torch.bfloat16, device=wq.device)
    code = lib().w8a8_scaled_mm_packed(_ptr(pa.buf), _ptr(wq), pa.M, N, pa.K, _mode(act_mode), _ptr(pa.scale),
                                       _ptr(pa.zp), _ptr(azp_adj), int(w_mode), _ptr(s_w), _ptr(w_sumsq), _ptr(bias),
                                       _ptr(out), _ptr(split_ws), split_ws.numel() if split_ws is not None else 0,
                                       _ptr(status), _stream())
    _check("w8a8_scaled_mm_packed", code)
    return out


def grouped_mm_packed(pa, w, s_w, seg_offsets, out=None, status=None, w_sumsq=None):
    _need(w, torch.int8, "w", 3)
    E, N, K = w.shape
    if out is None:
        out = torch.empty((pa.M, N), dtype=torch.bfloat16, device=w.device)
    code = lib().w8a8_grouped_mm_packed(_ptr(pa.buf), _ptr(pa.scale), _ptr(w), _ptr(s_w), _ptr(w_sumsq),
                                        _ptr(seg_offsets), E, pa.M, N, K, _ptr(out), _ptr(status), _stream())
    _check("w8a8_grouped_mm_packed", code)
    return out


def moe_quantize_gather_packed(x, row_index, buf=None):
    _need(x, torch.bfloat16, "x", 2)
    _need(row_index, torch.int64, "row_index", 1)
    T, K = x.shape
    R = row_index.numel()
    pk = _packed_buf(R, K, x.device, buf)
    s = torch.empty(R, dtype=torch.float32, device=x.device)
    _check("w8a8_moe_quantize_gather_packed",
           lib().w8a8_moe_quantize_gather_packed(_ptr(x), T, K, K, _ptr(row_index), R, _ptr(pk), _ptr(s), _stream()))
    return PackedActivations(pk, R, K, s)


def moe_quantize_scatter_packed(x, row_of, R=None, buf=None):
    """Each token row quantized once, its codes written to the routed rows row_of[t, j]."""
    _need(x, torch.bfloat16, "x", 2)
    _need(row_of, torch.int64, "row_of", 2)
    T, K = x.shape
    topk = row_of.shape[1]
    R = T * topk if R is None else R
    pk = _packed_buf(R, K, x.device, buf)
    s = torch.empty(R, dtype=torch.float32, device=x.device)
    _check("w8a8_moe_quantize_scatter_packed",
           lib().w8a8_moe_quantize_scatter_packed(_ptr(x), T, K, K, _ptr(row_of), topk, R, _ptr(pk), _ptr(s),
                                                  _stream()))
    return PackedActivations(pk, R, K, s)


def silu_mul_quant_packed(h, buf=None):
    _need(h, torch.bfloat16, "h", 2)
    R, twoI = h.shape
    inter = twoI // 2
    pk = _packed_buf(R, inter, h.device, buf)
    s = torch.empty(R, dtype=torch.float32, device=h.device)
    _check("w8a8_silu_mul_quant_packed",
           lib().w8a8_silu_mul_quant_packed(_ptr(h), R, inter, _ptr(pk), _ptr(s), _stream()))
    return PackedActivations(pk, R, inter, s)


def moe_forward(x, row_index, seg_offsets, row_of, topk_w, w13, s13, w2, s2, w13_sumsq=None, w2_sumsq=None):
    """MoE layer with W8A8 expert GEMMs over token-sorted segments (routing given).

    x bf16 [T, H]; row_index int64 [R] (token of each sorted row); seg_offsets int64 [E+1];
    row_of int64 [T, k] (sorted row of each (token, slot)); topk_w float32 [T, k];
    w13 int8 [E, 2I, H] with s13 [E, 2I]; w2 int8 [E, H, I] with s2 [E, H]; optional row sums
    of squares of the expert weights (int32 [E, 2I] and [E, H], weight_sumsq) for the GEMMs'
    Cauchy-Schwarz exactness test.
    Five launches: quantize (each token once, written to its routed rows), expert GEMM 1,
    SiLU*up + quantize, expert GEMM 2, combine.
    Returns (y [T, H], h [R, 2I], out [R, H]).
    """
    xa = moe_quantize_scatter_packed(x, row_of.reshape(x.shape[0], -1), row_index.numel())
    h = grouped_mm_packed(xa, w13, s13, seg_offsets, w_sumsq=w13_sumsq)
    ga = silu_mul_quant_packed(h)
    o = grouped_mm_packed(ga, w2, s2, seg_offsets, w_sumsq=w2_sumsq)
    return moe_combine(o, row_of, topk_w), h, o
