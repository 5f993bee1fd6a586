"""Plain numpy restatement of the W8A8 INT8 linear hot path -- test infrastructure only.

Every floating-point step is an explicit float32 (or float64) numpy operation in
the order written here, so that a reader can check each line against the rule it
cites.  bf16 tensors are carried as uint16 bit patterns.  Integer products use
float64 BLAS on int8 operands, which is exact because every partial sum is an
integer far below 2**53.

Short names of the sources are defined in oracle/__init__.py.
"""

import numpy as np

F32 = np.float32
F64 = np.float64


# ---------------------------------------------------------------------------
# bf16 <-> fp32 (format definition: bf16 is the top half of an IEEE fp32)
# ---------------------------------------------------------------------------

def bf16_bits_to_f32(bits):
    """bf16 bit patterns (uint16) -> exact float32 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16_bits(x):
    """float32 -> bf16 bit patterns, round to nearest, ties to even.

    Written from the definition: keep the top 16 bits after adding half an ulp
    of the kept part (0x7FFF plus the kept LSB for the tie case).  NaN stays a
    quiet NaN.
    """
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r = r.copy()
        r[nan] = ((u[nan] >> np.uint64(16)).astype(np.uint16) | np.uint16(0x0040))
    return r


def _rint_int(q_f):
    """Round half to even, as float64 (exact for float32 inputs)."""
    return np.rint(np.asarray(q_f, dtype=F64))


# ---------------------------------------------------------------------------
# S1: dynamic per-token symmetric activation quantization
# ---------------------------------------------------------------------------

def quantize_act_dynamic_symmetric(x):
    """Per-token symmetric INT8 quantization of activations.

    [SGLang-CT] item 3 names the step (``per_token_quant_int8(x)`` returning
    ``x_q, x_scale``) without a formula; the rule applied is the per-row rule of
    [Kunlun-INT8] 转换关系, applied to each token row:
        s[m]      = max_k |x[m,k]| / 127                 (float32 division)
        q[m,k]    = clamp(rint(x[m,k] / s[m]), -127, 127) (float32 division, ties-to-even)
    and an all-zero row gives q = 0, s = 1 ([Kunlun-INT8] 转换关系, last paragraph).

    x: float32 [M, K] (exact bf16 values).  Returns (q int8 [M,K], s float32 [M]).
    """
    x = np.asarray(x, dtype=F32)
    M, K = x.shape
    q = np.zeros((M, K), dtype=np.int8)
    s = np.ones(M, dtype=F32)
    for m in range(M):
        a = F32(np.max(np.abs(x[m]))) if K > 0 else F32(0)
        if a == F32(0):
            continue                      # zero row: q = 0, s = 1
        sm = F32(a / F32(127))            # one float32 division
        t = x[m] / sm                     # float32 division, element by element
        q[m] = np.clip(_rint_int(t), -127, 127).astype(np.int8)
        s[m] = sm
    return q, s


# ---------------------------------------------------------------------------
# S2: dynamic per-token asymmetric activation quantization
# ---------------------------------------------------------------------------

def quantize_act_dynamic_asymmetric(x):
    """Per-token asymmetric INT8 quantization (scale + int32 zero point).

    [vLLM-W8A8] 4.1 (table row 对称性) allows asymmetric activations; 4.2 says the
    zero point is used as int32 ("azp").  No formula is printed; the reading
    applied is the plain affine min/max map onto [-128, 127]:
        lo = min_k x, hi = max_k x
        s  = (hi - lo) / 255                      (float32 subtract, then divide)
        zp = rint(-128 - lo / s)                  (divide, subtract, ties-to-even), int32
        q  = clamp(rint(x / s) + zp, -128, 127)
    Degenerate rows (hi == lo): hi == 0 -> s = 1, zp = 0, q = 0; otherwise
    s = |hi| / 127, zp = 0 and q = clamp(rint(x / s), -127, 127).

    Returns (q int8 [M,K], s float32 [M], zp int32 [M]).
    """
    x = np.asarray(x, dtype=F32)
    M, K = x.shape
    q = np.zeros((M, K), dtype=np.int8)
    s = np.ones(M, dtype=F32)
    zp = np.zeros(M, dtype=np.int32)
    for m in range(M):
        if K == 0:
            continue
        lo = F32(np.min(x[m]))
        hi = F32(np.max(x[m]))
        if hi == lo:
            if hi == F32(0):
                continue
            sm = F32(F32(np.abs(hi)) / F32(127))
            t = x[m] / sm
            q[m] = np.clip(_rint_int(t), -127, 127).astype(np.int8)
            s[m] = sm
            continue
        sm = F32(F32(hi - lo) / F32(255))
        z = int(_rint_int(F32(F32(-128) - F32(lo / sm))))
        t = x[m] / sm
        q[m] = np.clip(_rint_int(t) + z, -128, 127).astype(np.int8)
        s[m] = sm
        zp[m] = z
    return q, s, zp


# ---------------------------------------------------------------------------
# S3: static per-tensor activation quantization
# ---------------------------------------------------------------------------

def quantize_act_static_symmetric(x, input_scale):
    """Static per-tensor symmetric quantization with a calibrated ``input_scale``.

    [vLLM-W8A8] 4.1 (static per-tensor branch) and 4.2 (input_scale registered
    only for the static scheme).  q = clamp(rint(x / input_scale), -127, 127).
    """
    x = np.asarray(x, dtype=F32)
    t = x / F32(input_scale)
    return np.clip(_rint_int(t), -127, 127).astype(np.int8)


def quantize_act_static_asymmetric(x, input_scale, input_zero_point):
    """Static per-tensor asymmetric quantization.

    [vLLM-W8A8] 4.2: the zero point is stored as int8 and used as an int32 azp.
    q = clamp(rint(x / input_scale) + zp, -128, 127).
    """
    x = np.asarray(x, dtype=F32)
    t = x / F32(input_scale)
    return np.clip(_rint_int(t) + int(input_zero_point), -128, 127).astype(np.int8)


def static_scale_from_tensor(x):
    """Calibration stand-in for the static scheme: one (scale, zero point) for a tensor.

    The pages obtain static scales from calibration data ([vLLM-W8A8] 3.2); with
    synthetic inputs the plainest stand-in is the affine min/max map of the whole
    tensor: s = (max - min) / 255, zp = clamp(rint(-128 - min / s), -128, 127)
    (the zero point must fit the int8 it is stored as, [vLLM-W8A8] 4.2).
    Returns (scale float32, zero_point int).
    """
    x = np.asarray(x, dtype=F32)
    lo = F32(np.min(x))
    hi = F32(np.max(x))
    s = F32(F32(hi - lo) / F32(255))
    z = int(np.clip(_rint_int(F32(F32(-128) - F32(lo / s))), -128, 127))
    return s, z


# ---------------------------------------------------------------------------
# S4: INT8 x INT8 -> INT32 GEMM
# ---------------------------------------------------------------------------

def int8_gemm(q_x, q_w):
    """acc[m, n] = sum_k q_x[m, k] * q_w[n, k], exact, as int32.

    [SGLang-CT] item 3: ``int8_scaled_mm(x_q, layer.weight, ...)`` multiplies the
    int8 activations by the int8 weight laid out [out_features, in_features]
    ([vLLM-W8A8] 4.2).  float64 BLAS is exact here: every product and partial
    sum is an integer below 2**31 < 2**53.
    """
    a = np.asarray(q_x, dtype=np.int8).astype(F64)
    b = np.asarray(q_w, dtype=np.int8).astype(F64)
    acc = a @ b.T
    return acc.astype(np.int64).astype(np.int32)


# ---------------------------------------------------------------------------
# S6: azp_adj
# ---------------------------------------------------------------------------

def azp_adj(q_w, input_zero_point=None):
    """Per-output-channel sum of the int8 weight over K, as int32.

    [SGLang-CT] item 4: ``azp_adj = weight.sum(...)``, multiplied by
    ``input_zero_point`` for the static scheme.  The sum runs over K for each
    output channel n: that is the only reading under which
    sum_k (q[m,k] - zp) * w[n,k] == acc[m,n] - zp * azp_adj[n].
    """
    w = np.asarray(q_w, dtype=np.int8).astype(np.int64)
    adj = w.sum(axis=1)
    if input_zero_point is not None:
        adj = adj * int(input_zero_point)
    return adj.astype(np.int32)


# ---------------------------------------------------------------------------
# S5: scale / azp / bias epilogue
# ---------------------------------------------------------------------------

def scaled_mm_epilogue(acc, s_x, s_w, zp=None, adj=None, adj_premultiplied=False, bias_bits=None):
    """y = bf16( (s_x[m] * s_w[n]) * f32(acc - zp*azp_adj) + bias[n] ).

    [SGLang-CT] item 3: ``int8_scaled_mm(x_q, W, x_scale, weight_scale,
    out_dtype=x.dtype, bias=bias)`` and item 4 (the azp correction).  Operation
    order, all float32 with one rounding each and no fused multiply-add:
        c = acc - zp[m] * azp_adj[n]     exact integer, then rounded to float32
            (premultiplied static form: acc - azp_adj'[n])
        t = s_x[m] * s_w[n]
        y = t * c   (+ bias[n] when a bias is given)
        out = bf16 round-to-nearest-even of y
    s_x: float32 [M] or scalar; s_w: float32 [N] or scalar; zp: int32 [M], scalar
    or None; bias_bits: bf16 bits [N] or None.
    Returns (y_bits uint16 [M, N], y float32 [M, N] before the bf16 rounding).
    """
    acc = np.asarray(acc, dtype=np.int32).astype(np.int64)
    M, N = acc.shape
    c = acc
    if adj is not None:
        a = np.asarray(adj, dtype=np.int32).astype(np.int64).reshape(1, N)
        if adj_premultiplied:
            c = c - a
        else:
            z = np.asarray(zp, dtype=np.int32).astype(np.int64).reshape(-1, 1)
            c = c - z * a
    cf = c.astype(F32)
    sx = np.broadcast_to(np.asarray(s_x, dtype=F32).reshape(-1, 1), (M, 1))
    sw = np.broadcast_to(np.asarray(s_w, dtype=F32).reshape(1, -1), (1, N))
    t = (sx * sw).astype(F32)
    y = (t * cf).astype(F32)
    if bias_bits is not None:
        y = (y + bf16_bits_to_f32(bias_bits).reshape(1, N)).astype(F32)
    return f32_to_bf16_bits(y), y


def w8a8_linear(x_bits, q_w, s_w, bias_bits=None, mode="dyn_sym", input_scale=None,
                input_zero_point=None, adj=None):
    """Whole linear: quantize activations, integer GEMM, epilogue.

    [SGLang-CT] item 3 ``apply_weights``: ``x_q, x_scale = per_token_quant_int8(x)``
    then ``int8_scaled_mm(...)``; item 4 for the asymmetric correction;
    [vLLM-W8A8] 4.1 for the four activation modes.
    Returns a dict with q, s_x, zp, acc, y_bits, y32.
    """
    x = bf16_bits_to_f32(x_bits)
    zp = None
    if mode == "dyn_sym":
        q, sx = quantize_act_dynamic_symmetric(x)
    elif mode == "dyn_asym":
        q, sx, zp = quantize_act_dynamic_asymmetric(x)
    elif mode == "static_sym":
        q = quantize_act_static_symmetric(x, input_scale)
        sx = F32(input_scale)
    elif mode == "static_asym":
        q = quantize_act_static_asymmetric(x, input_scale, input_zero_point)
        sx = F32(input_scale)
    else:
        raise ValueError(mode)
    acc = int8_gemm(q, q_w)
    if mode == "dyn_asym":
        a = azp_adj(q_w) if adj is None else adj
        y_bits, y32 = scaled_mm_epilogue(acc, sx, s_w, zp=zp, adj=a, bias_bits=bias_bits)
    elif mode == "static_asym":
        a = azp_adj(q_w, input_zero_point) if adj is None else adj
        y_bits, y32 = scaled_mm_epilogue(acc, sx, s_w, adj=a, adj_premultiplied=True,
                                         bias_bits=bias_bits)
    else:
        y_bits, y32 = scaled_mm_epilogue(acc, sx, s_w, bias_bits=bias_bits)
    return dict(q=q, s_x=sx, zp=zp, acc=acc, y_bits=y_bits, y32=y32)


# ---------------------------------------------------------------------------
# S7: per-output-channel symmetric weight quantization
# ---------------------------------------------------------------------------

def quantize_weight_per_channel(w):
    """Per-output-channel symmetric INT8 weights.

    [vLLM-W8A8] 4.2: weight int8 [out_features, in_features], weight_scale
    float32 [out_features, 1] (one scale per weight row); [Kunlun-INT8] 转换关系:
    s[i] = max_j |W[i,j]| / 127, q = clamp(round(W / s), -127, 127), zero row ->
    q = 0, s = 1.  Same arithmetic as quantize_act_dynamic_symmetric, per row.
    w: float32 [N, K].  Returns (q int8 [N,K], s float32 [N]).
    """
    return quantize_act_dynamic_symmetric(w)


# ---------------------------------------------------------------------------
# Fused modules with per-tensor scales: one scale for the whole weight
# ---------------------------------------------------------------------------

def requantize_with_max_scale(q_w, scales, logical_widths):
    """Unify the per-tensor scales of a fused weight (e.g. Q/K/V) to their maximum.

    [SGLang-CT] item 7 (텐서별 스케일 후처리: requantize_with_max_scale) and
    설계 근거 3 (Fused 모듈 호환): the logical partitions of a fused weight may carry
    different per-tensor scales; the largest becomes the module's single scale and
    the weights are quantized again against it.  The page prints only the call, so
    the arithmetic is our reading: partition p covers the next logical_widths[p]
    rows; each code is dequantized with one float32 multiply and requantized with
    the weight rule (float32 division, ties to even, clamp to +-127):
        s_max   = max_p scales[p]
        w'[n,k] = clamp(rint(f32(f32(q[n,k]) * scales[p]) / s_max), -127, 127)
    q_w int8 [N, K]; scales float32 [P] (positive, finite); sum(logical_widths) == N.
    Returns (w' int8 [N, K], s_max float32).
    """
    q = np.asarray(q_w, dtype=np.int8)
    sc = np.asarray(scales, dtype=F32).reshape(-1)
    widths = [int(w) for w in logical_widths]
    if len(widths) != sc.size or sum(widths) != q.shape[0] or any(w < 0 for w in widths):
        raise ValueError("logical_widths must give one non-negative width per scale, summing to N")
    if not np.all(np.isfinite(sc)) or not np.all(sc > 0):
        raise ValueError("per-tensor scales must be positive and finite")
    s_max = F32(sc.max())
    out = np.empty_like(q)
    r0 = 0
    for p, wdt in enumerate(widths):
        deq = (q[r0:r0 + wdt].astype(F32) * sc[p]).astype(F32)   # one float32 multiply
        t = (deq / s_max).astype(F32)                             # IEEE float32 division
        out[r0:r0 + wdt] = np.clip(_rint_int(t), -127, 127).astype(np.int8)
        r0 += wdt
    return out, s_max


# ---------------------------------------------------------------------------
# S8: FP8 E4M3 block-scaled -> INT8 per-row requantization
# ---------------------------------------------------------------------------

def e4m3_to_f32(codes):
    """Decode FP8 E4M3 (the "fn" variant: no infinities) from its definition.

    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.  Exponent field 0
    is subnormal: m * 2**-9.  Otherwise (1 + m/8) * 2**(e-7).  The pattern
    S.1111.111 is NaN; there is no infinity.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.power(2.0, e - 7))
    v = sign * mag
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return v.astype(F32)


def fp8_block_to_int8_rowwise(codes, scale_inv, block=128):
    """FP8 block-scaled weight -> INT8 weight with one float32 scale per row.

    [Kunlun-INT8] 转换关系:
        W_fp32[i,j] = W_fp8[i,j] * weight_scale_inv[i//128, j//128]   (multiply;
                      the "_inv" scale is never inverted)
        s[i]        = max_j |W_fp32[i,j]| / 127
        q[i,j]      = clamp(round(W_fp32[i,j] / s[i]), -127, 127)
        all-zero row -> q = 0, s = 1.
    Illegal input ([Kunlun-INT8] 验证 lists an illegal-scale test without a
    definition; reading applied): a row is bad when any block scale it touches
    is non-finite or <= 0, any of its codes is the NaN pattern, or any
    dequantized value is non-finite.  Bad rows give q = 0, s = 1 and are
    reported.
    codes: uint8 [N, K]; scale_inv: float32 [ceil(N/128), ceil(K/128)].
    Returns (q int8 [N,K], s float32 [N], bad bool [N]).
    """
    codes = np.asarray(codes, dtype=np.uint8)
    sinv = np.asarray(scale_inv, dtype=F32)
    N, K = codes.shape
    q = np.zeros((N, K), dtype=np.int8)
    s = np.ones(N, dtype=F32)
    bad = np.zeros(N, dtype=bool)
    col_block = np.arange(K) // block
    for i in range(N):
        row_scales = sinv[i // block, col_block]               # [K]
        with np.errstate(invalid="ignore", over="ignore"):
            wf = (e4m3_to_f32(codes[i]) * row_scales).astype(F32)  # one float32 multiply
        blocks_used = sinv[i // block, :((K + block - 1) // block)]
        if (not np.all(np.isfinite(blocks_used))) or np.any(blocks_used <= 0) \
                or (not np.all(np.isfinite(wf))):
            bad[i] = True
            continue
        a = F32(np.max(np.abs(wf))) if K > 0 else F32(0)
        if a == F32(0):
            continue
        si = F32(a / F32(127))
        t = wf / si
        q[i] = np.clip(_rint_int(t), -127, 127).astype(np.int8)
        s[i] = si
    return q, s, bad


# ---------------------------------------------------------------------------
# S9: MoE expert GEMMs over token-sorted segments
# ---------------------------------------------------------------------------

def silu_mul_bf16(gate_bits, up_bits):
    """g = bf16( silu(gate) * up ), evaluated in float64 and rounded once to bf16.

    The glue between the two expert GEMMs.  The pages name the MoE W8A8 method
    ([SGLang-CT] file tree; [Kunlun-INT8] w1/w2/w3) without its arithmetic; the
    gated form silu(w1 x) * (w3 x) with w1/w3 fused as one GEMM is the reading
    applied.  silu(a) = a / (1 + exp(-a)).
    """
    a = bf16_bits_to_f32(gate_bits).astype(F64)
    b = bf16_bits_to_f32(up_bits).astype(F64)
    g = a / (1.0 + np.exp(-a)) * b
    return f32_to_bf16_bits(g.astype(F32))


def moe_sort(topk_ids, num_experts):
    """Stable sort of the (token, slot) pairs by expert id.

    Returns (sorted_token [R], sorted_slot [R], seg_offsets [E+1]), R = T * topk.
    Entries of one expert keep token order.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=num_experts)
    seg = np.zeros(num_experts + 1, dtype=np.int64)
    seg[1:] = np.cumsum(counts)
    return (order // k).astype(np.int64), (order % k).astype(np.int64), seg


def moe_route(logits, topk):
    """Per-token expert choice and routing weight from router logits.

    The MoE INT8 scheme ([SGLang-CT] file tree: compressed_tensors_w8a8_int8_moe;
    [Kunlun-INT8] MoE method with experts w1/w2/w3) runs each token through the
    experts it is routed to; the pages leave the router itself to the framework.
    Our reading (the plainest one): ids[t] = the topk experts with the largest
    logits, in descending order, equal logits broken by the lower expert index;
    w[t, j] = softmax(logits[t])[ids[t, j]] over all E experts (not renormalised
    over the chosen ones), evaluated in float64.
    logits float32 [T, E].  Returns (ids int32 [T, topk], w float64 [T, topk]).
    """
    lg = np.asarray(logits, dtype=F32)
    T, E = lg.shape
    if not 1 <= topk <= E:
        raise ValueError("topk must be in [1, E]")
    ids = np.empty((T, topk), dtype=np.int32)
    w = np.empty((T, topk), dtype=F64)
    for t in range(T):
        row = lg[t].astype(F64)
        # stable sort of -logit keeps the lower index first among equal logits
        order = np.argsort(-row, kind="stable")[:topk]
        ids[t] = order
        e = np.exp(row - row.max())
        w[t] = e[order] / e.sum()
    return ids, w


def moe_forward(x_bits, topk_ids, topk_w, w13_q, s13, w2_q, s2, rows=None):
    """MoE layer with W8A8 INT8 expert GEMMs.

    Per expert e over its token segment: h = W8A8(x, W13_e) -> bf16 [n_e, 2I]
    (gate rows first), g = bf16(silu(h[:, :I]) * h[:, I:]), out = W8A8(g, W2_e)
    -> bf16 [n_e, H]; then y[t] = bf16( sum over the token's top-k slots, in
    slot order, of w[t, slot] * out ) with one float32 multiply and one float32
    add per slot.  Activations are quantized per token, dynamic symmetric
    ([Kunlun-INT8]: per-token dynamic symmetric INT8 activations).
    rows: optional token indices to evaluate (others left zero) so that large
    cases can be sampled.
    Returns dict(y_bits [T, H], y32 [T, H] (the float32 sums before the bf16 rounding),
    h_bits [R, 2I], out_bits [R, H]) where h/out are in sorted-row order (zero for rows
    not evaluated).
    """
    x = bf16_bits_to_f32(x_bits)
    T, H = x.shape
    E, twoI, _ = w13_q.shape
    inter = twoI // 2
    k = topk_ids.shape[1]
    tok, slot, seg = moe_sort(topk_ids, E)
    R = tok.shape[0]
    want = np.ones(T, dtype=bool) if rows is None else np.isin(np.arange(T), rows)
    h_bits = np.zeros((R, twoI), dtype=np.uint16)
    out_bits = np.zeros((R, H), dtype=np.uint16)
    row_of = np.zeros((T, k), dtype=np.int64)
    row_of[tok, slot] = np.arange(R)
    for e in range(E):
        r0, r1 = int(seg[e]), int(seg[e + 1])
        sel = [r for r in range(r0, r1) if want[tok[r]]]
        if not sel:
            continue
        sel = np.asarray(sel)
        xq, sx = quantize_act_dynamic_symmetric(x[tok[sel]])
        acc1 = int8_gemm(xq, w13_q[e])
        hb, _ = scaled_mm_epilogue(acc1, sx, s13[e])
        h_bits[sel] = hb
        g = silu_mul_bf16(hb[:, :inter], hb[:, inter:])
        gq, sg = quantize_act_dynamic_symmetric(bf16_bits_to_f32(g))
        acc2 = int8_gemm(gq, w2_q[e])
        ob, _ = scaled_mm_epilogue(acc2, sg, s2[e])
        out_bits[sel] = ob
    y_bits, y = moe_combine(out_bits, row_of, topk_w, rows=np.nonzero(want)[0])
    return dict(y_bits=y_bits, y32=y, h_bits=h_bits, out_bits=out_bits, seg=seg, tok=tok, slot=slot)


def moe_combine(out_bits, row_of, topk_w, rows=None):
    """The combine step of the MoE layer: y[t] = bf16( sum over the token's top-k slots,
    in slot order, of w[t, slot] * out[row_of[t, slot]] ), one float32 multiply and one
    float32 add per slot, starting from zero.
    out_bits: bf16 bits [R, H] (expert outputs in sorted-row order); row_of int [T, k];
    topk_w float32 [T, k]; rows: optional token indices to evaluate (others zero).
    Returns (y_bits [T, H], y32 [T, H] the float32 sums before the bf16 rounding).
    """
    T, k = row_of.shape
    H = out_bits.shape[1]
    y = np.zeros((T, H), dtype=F32)
    for t in (range(T) if rows is None else rows):
        acc = np.zeros(H, dtype=F32)
        for j in range(k):
            o = bf16_bits_to_f32(out_bits[row_of[t, j]])
            acc = (acc + (F32(topk_w[t, j]) * o).astype(F32)).astype(F32)
        y[t] = acc
    return f32_to_bf16_bits(y), y
