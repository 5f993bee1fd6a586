"""Parity of the CUDA kernels (through the C ABI) with the CPU oracle.

Integer results (int8 codes, int32 zero points and column sums) and float32 scales must
match bit for bit.  bf16 outputs must satisfy the stated tolerance -- |y - y_ref| <=
1e-2*|y_ref| or <= 1e-3*||y_ref32[m, :]||_2 per row -- and, because the epilogue follows
the oracle's float32 operation order, are also checked for exact equality where the
inputs to the epilogue are identical.
"""

import time

import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_quantized_gb300 as w8
from w8a8_int8_quantized_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def npbits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_bf16(y_gpu, y_bits_ref, y32_ref, exact=True):
    got = oracle.bf16_bits_to_f32(npbits(y_gpu)).astype(np.float64)
    ref = oracle.bf16_bits_to_f32(y_bits_ref).astype(np.float64)
    rownorm = np.linalg.norm(y32_ref.astype(np.float64), axis=1, keepdims=True)
    err = np.abs(got - ref)
    ok = (err <= 1e-2 * np.abs(ref)) | (err <= 1e-3 * rownorm)
    assert ok.all(), f"{(~ok).sum()} outputs outside tolerance; max err {err.max()}"
    if exact:
        mism = (npbits(y_gpu) != y_bits_ref).sum()
        assert mism == 0, f"{mism} bf16 outputs differ from the oracle bit pattern"


@pytest.fixture(autouse=True)
def _engine_reset():
    w8.set_gemm_engine(0)
    yield
    w8.set_gemm_engine(0)


# ------------------------------------------------------------------ quantizers

@pytest.mark.parametrize("M,K", [(16, 512), (37, 4096), (5, 14336), (3, 1500), (2, 20000), (1, 8)])
def test_quantize_act_dyn_sym(M, K):
    x = wl.llama_activations(M, K, seed=M + K)
    x[0, : min(K, 7)] = 0
    if M > 2:
        x[2] = 0  # all-zero row
    q, s, _ = w8.quantize_act(x.to(DEV), "dyn_sym")
    rq, rs = oracle.quantize_act_dynamic_symmetric(x.float().numpy())
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("M,K", [(16, 512), (64, 4096), (3, 1500)])
def test_quantize_act_dyn_asym(M, K):
    x = wl.asym_activations(M, K, seed=K)
    x[1] = 2.0          # constant row
    if M > 2:
        x[2] = 0.0      # zero row
    q, s, zp = w8.quantize_act(x.to(DEV), "dyn_asym")
    rq, rs, rz = oracle.quantize_act_dynamic_asymmetric(x.float().numpy())
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(zp.cpu().numpy(), rz)


def test_division_free_codes_equal_ieee_quotient_exhaustively():
    """The symmetric row rule's codes come from a division-free rounding (Markstein's
    correction step on RN(x * RN(1/s))).  Run on every bf16 absmax a and every bf16 x with
    |x| <= a (s = RN(a / 127)), the library's own device function gives rint of the IEEE
    float32 quotient x / s in every case ([Kunlun-INT8] 转换关系: round(W / s)).  The affine
    rule's division-free codes (window test and exact near-tie decision) are checked the same
    way over every bf16 value of 65536 row ranges, a quarter of them with exact ties."""
    from w8a8_int8_quantized_gb300 import quotient_check
    out = quotient_check.run()
    r = out["symmetric_rule"]
    assert r["values"] > 800_000_000
    assert r["code_mismatches"] == 0
    a = out["affine_rule"]
    assert a["values"] > 100_000_000
    assert a["code_mismatches"] == 0
    assert a["exact_resolver_mismatches"] == 0


def _asym_stress_rows(K):
    """bf16 rows that stress the affine rule's fast path: rows far from zero (|x/s| up to
    about 2^16), constant rows, rows of two values, tiny magnitudes, rows of exact
    multiples of a power of two (many exact ties), exact ties under an odd zero point and
    near-ties under an inexact scale."""
    g = torch.Generator().manual_seed(K)
    rows = [
        1000.0 + torch.randint(0, 8, (K,), generator=g).float() * 4.0,      # bf16 step 4 at 1000
        -3.0e4 + torch.rand(K, generator=g) * 300.0,
        torch.full((K,), -7.5),
        torch.where(torch.rand(K, generator=g) < 0.5, torch.tensor(1.0), torch.tensor(3.0)),
        torch.randn(K, generator=g) * 1e-30,
        torch.randint(-64, 64, (K,), generator=g).float() * 0.125,
        torch.randn(K, generator=g) * 5.0 + 40.0,
        torch.linspace(-1.0, 1.0, K),
    ]
    # exact ties with an odd zero point: s = 1/8 exactly (lo = -13/8, hi = lo + 255/8, zp = -115)
    # and x = (m + 1/2) s
    r = (torch.randint(-13, 128, (K,), generator=g).float() + 0.5) * 0.125
    r[0], r[1 % K] = -1.625, 30.25
    rows.append(r)
    # lo = -13.6875, hi = 36.25: x = +-1.46875 has RN(x * RN(1/s)) = +-7.5 exactly but
    # x / s = +-7.4999995, and the exact product x * RN(1/s) lies just above the midpoint below
    # 7.5, so a multiply-add fused into one rounding and the separately rounded product break
    # the value different ways
    r = torch.where(torch.rand(K, generator=g) < 0.5, torch.tensor(1.46875), torch.tensor(-1.46875))
    r[0], r[1 % K] = -13.6875, 36.25
    rows.append(r)
    # near-ties with inexact scales: of every bf16 value in [lo, hi], the 64 whose quotients
    # x / s lie closest to a half-integer, drawn at random
    for lo, hi in ((-3.5, 4.5), (-1.0, 7.25), (0.5, 1.5)):
        s_ = np.float32(np.float32(hi) - np.float32(lo)) / np.float32(255.0)
        pos = np.arange(0, 0x7F80, dtype=np.uint32) << 16
        cand = np.concatenate([pos.view(np.float32), (pos | 0x80000000).view(np.float32)])
        cand = cand[(cand >= lo) & (cand <= hi)]
        t = cand.astype(np.float64) / np.float64(s_)
        dist = np.abs(np.abs(t - np.floor(t)) - 0.5)
        near = torch.from_numpy(cand[np.argsort(dist, kind="stable")[:64]].copy())
        r = near[torch.randint(0, 64, (K,), generator=g)]
        r[0], r[1 % K] = lo, hi
        rows.append(r)
    return torch.stack(rows).to(torch.bfloat16)


def _sym_tie_rows(K):
    """bf16 rows whose quotients x/s sit on or next to half-integers: s = 1 and s = 2 with
    x = (k + 1/2) s (exact ties), absmax 100 (s not a power of two) with x the bf16 values
    nearest (k + 1/2) s and their neighbours, and values around +-s/2 and +-3s/2."""
    g = torch.Generator().manual_seed(K)
    k = torch.randint(-127, 127, (K,), generator=g).float()
    rows = []
    r = k + 0.5
    r[0] = 127.0
    rows.append(r)                                   # s = 1: every value an exact tie
    r = 2.0 * k + 1.0
    r[0] = 254.0
    rows.append(r)                                   # s = 2
    s100 = np.float32(100.0) / np.float32(127.0)
    base = torch.from_numpy(((k.numpy() + 0.5) * s100).astype(np.float32))
    b16 = base.to(torch.bfloat16).float()
    step = torch.randint(-2, 3, (K,), generator=g).float()
    near = (b16.view(torch.int32) + (step.to(torch.int32) << 16)).view(torch.float32)
    near[0] = 100.0
    rows.append(near)                                # near-ties, s = RN(100/127)
    small = torch.tensor([0.5, -0.5, 1.5, -1.5, 0.49, 0.51, 1.49, 1.51], dtype=torch.float32)
    r = small[torch.randint(0, 8, (K,), generator=g)] * s100
    r[0] = 100.0
    rows.append(r)                                   # |h| < 1.5 and its edges
    return torch.stack(rows).to(torch.bfloat16)


@pytest.mark.parametrize("K", [512, 4096])
def test_quantize_sym_near_ties(K):
    """The exact near-tie decision (residual sign and size against s*ulp(h)/2) against the
    oracle's IEEE division, through the activation and the weight quantizers."""
    x = _sym_tie_rows(K)
    rq, rs = oracle.quantize_act_dynamic_symmetric(x.float().numpy())
    q, s, _ = w8.quantize_act(x.to(DEV), "dyn_sym")
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    wq, sw, adj = w8.quantize_weight(x.to(DEV), with_azp_adj=True)
    wr, wsr = oracle.quantize_weight_per_channel(x.float().numpy())
    np.testing.assert_array_equal(sw.cpu().numpy(), wsr)
    np.testing.assert_array_equal(wq.cpu().numpy(), wr)
    np.testing.assert_array_equal(adj.cpu().numpy(), wr.astype(np.int64).sum(1))


@pytest.mark.parametrize("K", [512, 4096, 1500])
def test_quantize_act_dyn_asym_stress(K):
    x = _asym_stress_rows(K)
    q, s, zp = w8.quantize_act(x.to(DEV), "dyn_asym")
    rq, rs, rz = oracle.quantize_act_dynamic_asymmetric(x.float().numpy())
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(zp.cpu().numpy(), rz)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("M,K", [(16, 512), (128, 4096), (3, 1500)])
def test_quantize_act_static(M, K):
    x = wl.asym_activations(M, K, seed=K + 1)
    xs = x.float().numpy()
    sc, z = oracle.static_scale_from_tensor(xs)
    scale = torch.tensor([sc], dtype=torch.float32, device=DEV)
    zp = torch.tensor([z], dtype=torch.int32, device=DEV)
    q, _, _ = w8.quantize_act(x.to(DEV), "static_sym", scale=scale)
    np.testing.assert_array_equal(q.cpu().numpy(), oracle.quantize_act_static_symmetric(xs, sc))
    q, _, _ = w8.quantize_act(x.to(DEV), "static_asym", scale=scale, zp=zp)
    np.testing.assert_array_equal(q.cpu().numpy(), oracle.quantize_act_static_asymmetric(xs, sc, z))
    # a tiny static scale drives every value into the clamp
    tiny = torch.tensor([1e-30], dtype=torch.float32, device=DEV)
    q, _, _ = w8.quantize_act(x.to(DEV), "static_asym", scale=tiny, zp=zp)
    np.testing.assert_array_equal(q.cpu().numpy(), oracle.quantize_act_static_asymmetric(xs, np.float32(1e-30), z))


@pytest.mark.parametrize("mode", ["dyn_sym", "dyn_asym", "static_sym", "static_asym"])
@pytest.mark.parametrize("M,K", [(16, 512), (37, 4096), (3, 14336)])
def test_quantize_act_packed(mode, M, K):
    """The packed format holds the same integer codes as fp16, plus each row's L1 norm (and, for
    the affine modes, its sum of squares)."""
    x = (wl.asym_activations if "asym" in mode else wl.llama_activations)(M, K, seed=M + 3)
    if M > 2:
        x[2] = 0
    xs = x.float().numpy()
    sc, z = oracle.static_scale_from_tensor(xs)
    kw = {}
    if mode.startswith("static"):
        kw["scale"] = torch.tensor([sc], dtype=torch.float32, device=DEV)
        kw["zp"] = torch.tensor([z], dtype=torch.int32, device=DEV)
    pa = w8.quantize_act_packed(x.to(DEV), mode, **kw)
    if mode == "dyn_sym":
        rq, rs = oracle.quantize_act_dynamic_symmetric(xs)
    elif mode == "dyn_asym":
        rq, rs, rz = oracle.quantize_act_dynamic_asymmetric(xs)
        np.testing.assert_array_equal(pa.zp.cpu().numpy(), rz)
    elif mode == "static_sym":
        rq, rs = oracle.quantize_act_static_symmetric(xs, sc), None
    else:
        rq, rs = oracle.quantize_act_static_asymmetric(xs, sc, z), None
    codes = pa.codes().float().cpu().numpy()
    np.testing.assert_array_equal(codes, rq.astype(np.float32))
    np.testing.assert_array_equal(pa.norms().cpu().numpy(), np.abs(rq.astype(np.int64)).sum(1))
    if "asym" in mode:  # the affine modes also carry each row's sum of squares
        np.testing.assert_array_equal(pa.sumsq().cpu().numpy(), (rq.astype(np.int64) ** 2).sum(1))
    if rs is not None:
        np.testing.assert_array_equal(pa.scale.cpu().numpy(), rs)


@pytest.mark.parametrize("N,K", [(512, 512), (300, 4096), (64, 1500)])
def test_quantize_weight_and_azp(N, K):
    w = wl.weight_bf16(N, K, seed=N)
    w[3] = 0
    wq, s, adj = w8.quantize_weight(w.to(DEV), with_azp_adj=True)
    rq, rs = oracle.quantize_weight_per_channel(w.float().numpy())
    np.testing.assert_array_equal(wq.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(adj.cpu().numpy(), oracle.azp_adj(rq))
    z = torch.tensor([-37], dtype=torch.int32, device=DEV)
    np.testing.assert_array_equal(w8.azp_adj(wq, z).cpu().numpy(), oracle.azp_adj(rq, -37))
    np.testing.assert_array_equal(w8.azp_adj(wq).cpu().numpy(), oracle.azp_adj(rq))


# ------------------------------------------------------------------ GEMM + epilogue

def _gemm_case(M, N, K, seed, act="dyn_sym", bias=True, w_mode=w8.W_CHANNEL):
    x = wl.asym_activations(M, K, seed=seed) if "asym" in act else wl.llama_activations(M, K, seed=seed)
    w = wl.weight_bf16(N, K, seed=seed + 1)
    b = wl.weight_bf16(1, N, seed=seed + 2, std=0.1)[0] if bias else None
    xb = wl.bits(x)
    rq, rs = oracle.quantize_weight_per_channel(w.float().numpy())
    if w_mode == w8.W_TENSOR:
        rs = np.array([np.float32(rs.max())], dtype=np.float32)
    inputs = dict(x=x, w=w, b=b, xb=xb, rq=rq, rs=rs)
    return inputs


@pytest.mark.parametrize("engine", [1, 2])
@pytest.mark.parametrize("M,N,K", [(16, 512, 512), (1, 256, 64), (300, 520, 1040), (129, 257, 2064),
                                   (17, 8, 16), (16, 24, 16), (2, 5, 32), (257, 1, 48), (600, 300, 16),
                                   (256, 512, 4096), (7, 1000, 4112)])
def test_scaled_mm_dyn_sym(engine, M, N, K):
    d = _gemm_case(M, N, K, seed=M * 7 + N)
    w8.set_gemm_engine(engine)
    xq, sx, _ = w8.quantize_act(d["x"].to(DEV), "dyn_sym")
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    bias = d["b"].to(DEV) if d["b"] is not None else None
    y = w8.scaled_mm(xq, wq, sx, sw, "dyn_sym", bias=bias)
    r = oracle.w8a8_linear(d["xb"], d["rq"], d["rs"], bias_bits=wl.bits(d["b"]) if d["b"] is not None else None)
    check_bf16(y, r["y_bits"], r["y32"])


@pytest.mark.parametrize("act", ["dyn_sym", "dyn_asym", "static_sym", "static_asym"])
@pytest.mark.parametrize("w_mode", [w8.W_CHANNEL, w8.W_TENSOR])
@pytest.mark.parametrize("M,N,K", [(1, 520, 4112), (2, 8, 16), (2, 2500, 4096), (2, 300, 14336), (1, 5000, 4096),
                                   (1, 17, 12304)])
def test_gemv_rows(act, w_mode, M, N, K):
    """One or two token rows take the dp4a GEMV (K % 16 == 0): units of 4096 weight bytes
    with a ragged last one (K = 4112, 12304), K = 16 (one partial unit), weights with fewer
    rows than warps (N = 8, 17) and more rows than warps (N = 5000), every activation mode
    through the pre-quantized path; bit-exact against the oracle."""
    d = _gemm_case(M, N, K, seed=M * 31 + K, act=act, w_mode=w_mode)
    xs = d["x"].float().numpy()
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    bias = d["b"].to(DEV)
    sc, z = oracle.static_scale_from_tensor(xs)
    kw = {}
    if act == "dyn_sym":
        xq, sx, _ = w8.quantize_act(d["x"].to(DEV), "dyn_sym")
    elif act == "dyn_asym":
        xq, sx, zq = w8.quantize_act(d["x"].to(DEV), "dyn_asym")
        kw = dict(zp=zq, azp_adj=w8.azp_adj(wq))
    else:
        sx = torch.tensor([sc], dtype=torch.float32, device=DEV)
        zt = torch.tensor([z], dtype=torch.int32, device=DEV)
        xq, _, _ = w8.quantize_act(d["x"].to(DEV), act, scale=sx, zp=zt if act == "static_asym" else None)
        if act == "static_asym":
            kw = dict(zp=zt, azp_adj=w8.azp_adj(wq, zt))
    y = w8.scaled_mm(xq, wq, sx, sw, act, bias=bias, w_mode=w_mode, **kw)
    r = oracle.w8a8_linear(d["xb"], d["rq"], d["rs"], bias_bits=wl.bits(d["b"]), mode=act,
                           input_scale=sc, input_zero_point=z)
    check_bf16(y, r["y_bits"], r["y32"])


def test_gemv_extremes_exact():
    """Largest int32 magnitudes through the GEMV: acc = +-128*127*K at K = 65536 (one row)
    and 14336 (two rows) must be exact, with the asymmetric epilogue."""
    for M, K in ((1, 65536), (2, 14336)):
        N = 40
        xq = torch.full((M, K), -128, dtype=torch.int8)
        xq[1::2] = 127
        wq = torch.full((N, K), 127, dtype=torch.int8)
        wq[1::2] = -127
        wq[7, 1000:] = 3
        sx = torch.full((M,), 1.0, dtype=torch.float32)
        sw = torch.full((N,), 2.0 ** -24, dtype=torch.float32)
        zp = torch.arange(M, dtype=torch.int32) - 2
        adj = torch.from_numpy(oracle.azp_adj(wq.numpy()))
        y = w8.scaled_mm(xq.to(DEV), wq.to(DEV), sx.to(DEV), sw.to(DEV), "dyn_asym", zp=zp.to(DEV),
                         azp_adj=adj.to(DEV))
        acc = oracle.int8_gemm(xq.numpy(), wq.numpy())
        yb, y32 = oracle.scaled_mm_epilogue(acc, sx.numpy(), sw.numpy(), zp=zp.numpy(), adj=adj.numpy())
        check_bf16(y, yb, y32)


@pytest.mark.parametrize("M,N,K", [(1, 520, 4112), (2, 520, 14336), (1, 520, 30016), (2, 520, 30016),
                                   (5, 5000, 4096), (8, 5000, 11200), (8, 300, 64)])
def test_decode_rows_staged(M, N, K):
    """Launches of at most 8 token rows stage the rows in shared memory (more than 48 KB at
    K = 30016) and walk 16-channel blocks persistently (N = 5000: more blocks than CTAs, a
    ragged last block; K = 11200: warps own unequal numbers of K-chunks; K = 64: most warps
    own none); bit-exact against the oracle."""
    d = _gemm_case(M, N, K, seed=M + K)
    xq, sx, _ = w8.quantize_act(d["x"].to(DEV), "dyn_sym")
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    y = w8.scaled_mm(xq, wq, sx, sw, "dyn_sym", bias=d["b"].to(DEV))
    r = oracle.w8a8_linear(d["xb"], d["rq"], d["rs"], bias_bits=wl.bits(d["b"]))
    check_bf16(y, r["y_bits"], r["y32"])


@pytest.mark.parametrize("engine", [1, 2])
@pytest.mark.parametrize("act", ["dyn_asym", "static_sym", "static_asym"])
@pytest.mark.parametrize("w_mode", [w8.W_CHANNEL, w8.W_TENSOR])
@pytest.mark.parametrize("M,N", [(130, 384), (6, 5000)])
def test_linear_modes(engine, act, w_mode, M, N):
    K = 1088
    d = _gemm_case(M, N, K, seed=11, act=act, w_mode=w_mode)
    w8.set_gemm_engine(engine)
    xs = d["x"].float().numpy()
    sc, z = oracle.static_scale_from_tensor(xs)
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    bias = d["b"].to(DEV)
    kw = {}
    if act == "dyn_asym":
        kw["azp_adj"] = w8.azp_adj(wq)
    if act.startswith("static"):
        kw["input_scale"] = torch.tensor([sc], dtype=torch.float32, device=DEV)
    if act == "static_asym":
        kw["input_zero_point"] = torch.tensor([z], dtype=torch.int32, device=DEV)
        kw["azp_adj"] = w8.azp_adj(wq, kw["input_zero_point"])
    y = w8.linear(d["x"].to(DEV), wq, sw, act_mode=act, bias=bias, w_mode=w_mode, **kw)
    r = oracle.w8a8_linear(d["xb"], d["rq"], d["rs"], bias_bits=wl.bits(d["b"]), mode=act,
                           input_scale=sc, input_zero_point=z)
    check_bf16(y, r["y_bits"], r["y32"])


@pytest.mark.parametrize("engine", [1, 2])
def test_gemm_extremes_exact(engine):
    """Largest int32 magnitudes: acc = +-128*127*K at K = 14336 must be exact."""
    w8.set_gemm_engine(engine)
    M, N, K = 130, 260, 14336
    xq = torch.full((M, K), -128, dtype=torch.int8)
    xq[1::2] = 127
    xq[5, ::3] = -1
    wq = torch.full((N, K), 127, dtype=torch.int8)
    wq[1::2] = -127
    wq[7, 1000:] = 3
    sx = torch.full((M,), 1.0, dtype=torch.float32)
    sw = torch.full((N,), 2.0 ** -20, dtype=torch.float32)
    zp = torch.arange(M, dtype=torch.int32) - 60
    adj = torch.from_numpy(oracle.azp_adj(wq.numpy()))
    y = w8.scaled_mm(xq.to(DEV), wq.to(DEV), sx.to(DEV), sw.to(DEV), "dyn_asym", zp=zp.to(DEV), azp_adj=adj.to(DEV))
    acc = oracle.int8_gemm(xq.numpy(), wq.numpy())
    yb, y32 = oracle.scaled_mm_epilogue(acc, sx.numpy(), sw.numpy(), zp=zp.numpy(), adj=adj.numpy())
    check_bf16(y, yb, y32)


@pytest.mark.parametrize("K,fill", [(1024, 127), (1040, None), (1040, "edge"), (4096, "mixed")])
def test_gemm_single_pass_bound(K, fill):
    """Tiles whose activation rows have L1 norm < 2^17 run one fp32 pass over K; rows at or
    above the bound switch the whole tile to 1024-K chunks.  Both must be exact."""
    M, N = 300, 272
    rng = np.random.default_rng(K)
    xq = rng.integers(-3, 4, size=(M, K)).astype(np.int8)
    if fill == 127:
        xq[:] = 127                       # norm 130048 < 2^17: single pass, |acc| = 127*127*1024
    elif fill == "edge":
        xq[:] = 0
        xq[0, :1032] = 127                # norm 131064 + 7 = 131071: single pass
        xq[0, 1032:1039] = 1
        xq[258, :1032] = 127              # norm 131072, second row tile: chunked
        xq[258, 1032:1040] = 1
        xq[260, :] = -128
    elif fill == "mixed":
        xq[7, :] = -128                   # one big row forces chunks for its tile only
    wq = np.full((N, K), 127, dtype=np.int8)
    wq[1::3] = -127
    wq[5] = rng.integers(-127, 128, size=K).astype(np.int8)
    sx = np.full(M, 2.0 ** -10, dtype=np.float32)
    sw = np.full(N, 2.0 ** -12, dtype=np.float32)
    w8.set_gemm_engine(1)
    y = w8.scaled_mm(torch.from_numpy(xq).to(DEV), torch.from_numpy(wq).to(DEV), torch.from_numpy(sx).to(DEV),
                     torch.from_numpy(sw).to(DEV))
    acc = oracle.int8_gemm(xq, wq)
    yb, y32 = oracle.scaled_mm_epilogue(acc, sx, sw)
    check_bf16(y, yb, y32)


def _split_bytes_expected(M, N, K):
    """The K-split scratch from the plan stated in include/w8a8.h: the tiles past a launch's
    last full wave of CTA pairs (all of them when there is none) are cut into as many parts
    as fill the pairs that wave leaves idle, at most one per 1024-K chunk."""
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    tiles = -(-M // 256) * -(-N // 256)
    if M <= 16:
        return 0
    tail = tiles % pairs
    if tail == 0:
        return 0
    f = min(pairs // tail, -(-K // 1024))
    if f < 2:
        return 0
    return tail * f * 256 * 256 * 4


@pytest.mark.parametrize("M,N,K", [(128, 4096, 4096), (300, 1000, 14336), (256, 20480, 2048), (17, 520, 3072),
                                   (130, 8, 1040), (512, 4104, 4096), (64, 256, 1024), (4096, 6144, 4096),
                                   (4096, 4096, 14336), (4096, 28672, 4096)])
def test_splitk_workspace_size(M, N, K):
    assert w8.splitk_workspace_size(M, N, K) == _split_bytes_expected(M, N, K)


@pytest.mark.parametrize("M,N,K,act", [(1024, 10240, 2048, "dyn_sym"), (4096, 6144, 4096, "dyn_sym"),
                                       (1024, 10240, 2048, "dyn_asym")])
def test_split_last_wave(M, N, K, act):
    """Launches of several waves cut only the tiles past their last full wave along K
    (1024 x 10240: 160 tiles = two waves of 76 pairs + 8, in parts; the qkv shape at
    M = 4096: 384 tiles = five waves + 4).  The result equals the unsplit call bit for bit
    and, on sampled rows, the oracle."""
    assert _split_bytes_expected(M, N, K) > 0
    x = wl.asym_activations(M, K, seed=K + 3) if act == "dyn_asym" else wl.llama_activations(M, K, seed=K + 3)
    w = wl.weight_bf16(N, K, seed=N + 5)
    rq, rs = oracle.quantize_weight_per_channel(w.float().numpy())
    wq = torch.from_numpy(rq).to(DEV)
    sw = torch.from_numpy(rs).to(DEV)
    kw = {"azp_adj": w8.azp_adj(wq)} if act == "dyn_asym" else {}
    xd = x.to(DEV)
    base = w8.linear_workspace_size(M, K, act)
    ws_split = torch.empty(base + w8.splitk_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    ws_plain = torch.empty(base, dtype=torch.uint8, device=DEV)
    y_split = w8.linear(xd, wq, sw, act_mode=act, workspace=ws_split, **kw)
    y_plain = w8.linear(xd, wq, sw, act_mode=act, workspace=ws_plain, **kw)
    assert torch.equal(y_split, y_plain)
    rows = np.concatenate([np.arange(0, M, 61), [M - 1]])
    r = oracle.w8a8_linear(wl.bits(x)[rows], rq, rs, mode=act)
    check_bf16(y_split[torch.from_numpy(rows).to(DEV)], r["y_bits"], r["y32"])


@pytest.mark.parametrize("act", ["dyn_sym", "dyn_asym", "static_asym"])
@pytest.mark.parametrize("M,N,K,acts", [(128, 4096, 4096, "llama"), (300, 1000, 14336, "llama"),
                                        (256, 20480, 2048, "llama"), (77, 520, 3072, "normal"),
                                        (130, 264, 5120, "normal")])
def test_linear_split_k(act, M, N, K, acts):
    """Launches with fewer tiles than two waves split tiles along K when the workspace holds
    the split scratch: only one row tile (M = 128: 16 tiles in 4 parts), unequal parts
    (K = 14336: 14 chunks in parts of 3 and 4), a full first wave plus split tail tiles
    (256 x 20480: 80 tiles), ragged rows and columns, and N(0, 1) rows whose L1 norms exceed
    2^17 so each part runs 1024-K chunks.  Bit-exact against the oracle and against the same
    call without the scratch."""
    if _split_bytes_expected(M, N, K) == 0:
        pytest.skip("shape does not split on this device")
    rng = np.random.default_rng(M + N + K)
    if acts == "normal":
        x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
        if "asym" in act:
            x = x + 0.5
    elif "asym" in act:
        x = wl.asym_activations(M, K, seed=K)
    else:
        x = wl.llama_activations(M, K, seed=K)
    w = wl.weight_bf16(N, K, seed=N)
    b = wl.weight_bf16(1, N, seed=N + 1, std=0.1)[0]
    rq, rs = oracle.quantize_weight_per_channel(w.float().numpy())
    xs = x.float().numpy()
    sc, z = oracle.static_scale_from_tensor(xs)
    wq = torch.from_numpy(rq).to(DEV)
    sw = torch.from_numpy(rs).to(DEV)
    kw = {}
    if act == "dyn_asym":
        kw["azp_adj"] = w8.azp_adj(wq)
    if act == "static_asym":
        kw["input_scale"] = torch.tensor([sc], dtype=torch.float32, device=DEV)
        kw["input_zero_point"] = torch.tensor([z], dtype=torch.int32, device=DEV)
        kw["azp_adj"] = w8.azp_adj(wq, kw["input_zero_point"])
    xd = x.to(DEV)
    base = w8.linear_workspace_size(M, K, act)
    extra = w8.splitk_workspace_size(M, N, K)
    ws_split = torch.full((base + extra,), 0xA5, dtype=torch.uint8, device=DEV)  # stale scratch
    ws_plain = torch.empty(base, dtype=torch.uint8, device=DEV)
    ws_short = torch.empty(base + extra - 256, dtype=torch.uint8, device=DEV)  # too small: no split
    y_split = w8.linear(xd, wq, sw, act_mode=act, bias=b.to(DEV), workspace=ws_split, **kw)
    y_again = w8.linear(xd, wq, sw, act_mode=act, bias=b.to(DEV), workspace=ws_split, **kw)
    y_plain = w8.linear(xd, wq, sw, act_mode=act, bias=b.to(DEV), workspace=ws_plain, **kw)
    y_short = w8.linear(xd, wq, sw, act_mode=act, bias=b.to(DEV), workspace=ws_short, **kw)
    torch.cuda.synchronize()
    r = oracle.w8a8_linear(wl.bits(x), rq, rs, bias_bits=wl.bits(b), mode=act, input_scale=sc, input_zero_point=z)
    check_bf16(y_split, r["y_bits"], r["y32"])
    for y in (y_again, y_plain, y_short):
        assert torch.equal(y.view(torch.int16), y_split.view(torch.int16))


@pytest.mark.parametrize("case", ["ragged_k_one_step_part", "ragged_n_scalar_stores", "static_sym_tensor_scale",
                                  "scaled_mm_dyn_asym"])
def test_split_k_edges(case):
    """Edges of the K split: a last part of one 64-wide step with a ragged K tail (M = 5 on the
    tensor-core engine, K = 3088: 49 steps in parts of 16/16/16/1), an output width that is
    not a multiple of 8 (the reduce kernel's scalar stores), a per-tensor weight scale
    without bias, and w8a8_scaled_mm with per-row zero points.  Bit-exact against the oracle
    and against the unsplit call."""
    if case == "ragged_k_one_step_part":
        M, N, K, act, w_mode, bias = 5, 520, 3088, "dyn_sym", w8.W_CHANNEL, True
        w8.set_gemm_engine(1)
    elif case == "ragged_n_scalar_stores":
        M, N, K, act, w_mode, bias = 200, 777, 2048, "dyn_sym", w8.W_CHANNEL, True
    elif case == "static_sym_tensor_scale":
        M, N, K, act, w_mode, bias = 96, 1000, 4096, "static_sym", w8.W_TENSOR, False
    else:
        M, N, K, act, w_mode, bias = 64, 768, 5120, "dyn_asym", w8.W_CHANNEL, True
    assert w8.splitk_workspace_size(M, N, K) > 0
    d = _gemm_case(M, N, K, seed=M + N, act=act, bias=bias, w_mode=w_mode)
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    b = d["b"].to(DEV) if bias else None
    bb = wl.bits(d["b"]) if bias else None
    extra = w8.splitk_workspace_size(M, N, K)
    if case == "scaled_mm_dyn_asym":
        xq, sx, zp = w8.quantize_act(d["x"].to(DEV), "dyn_asym")
        adj = w8.azp_adj(wq)
        base = w8.lib().w8a8_scaled_mm_workspace_size(M, K)
        run = lambda ws: w8.scaled_mm(xq, wq, sx, sw, "dyn_asym", zp=zp, azp_adj=adj, bias=b, workspace=ws)
        r = oracle.w8a8_linear(d["xb"], d["rq"], d["rs"], bias_bits=bb, mode="dyn_asym")
    else:
        sc, z = oracle.static_scale_from_tensor(d["x"].float().numpy())
        kw = {"input_scale": torch.tensor([sc], dtype=torch.float32, device=DEV)} if act == "static_sym" else {}
        base = w8.linear_workspace_size(M, K, act)
        run = lambda ws: w8.linear(d["x"].to(DEV), wq, sw, act_mode=act, bias=b, w_mode=w_mode, workspace=ws, **kw)
        r = oracle.w8a8_linear(d["xb"], d["rq"], d["rs"], bias_bits=bb, mode=act, input_scale=sc)
    y_split = run(torch.full((base + extra,), 0x5A, dtype=torch.uint8, device=DEV))
    y_plain = run(torch.empty(base, dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    check_bf16(y_split, r["y_bits"], r["y32"])
    assert torch.equal(y_plain.view(torch.int16), y_split.view(torch.int16))


@pytest.mark.parametrize("w_mode", [w8.W_CHANNEL, w8.W_TENSOR])
def test_scaled_mm_split_k_extremes(w_mode):
    """acc = +-128*127*K at K = 14336 through split parts (2 tiles in 14 one-chunk parts),
    with zero points on every row: exact."""
    M, N, K = 130, 260, 14336
    xq = torch.full((M, K), -128, dtype=torch.int8)
    xq[1::2] = 127
    xq[5, ::3] = -1
    wq = torch.full((N, K), 127, dtype=torch.int8)
    wq[1::2] = -127
    wq[7, 1000:] = 3
    sx = torch.full((M,), 1.0, dtype=torch.float32)
    sw = torch.full((N if w_mode == w8.W_CHANNEL else 1,), 2.0 ** -20, dtype=torch.float32)
    zp = torch.arange(M, dtype=torch.int32) - 60
    adj = torch.from_numpy(oracle.azp_adj(wq.numpy()))
    assert w8.splitk_workspace_size(M, N, K) > 0
    ws = torch.empty(w8.lib().w8a8_scaled_mm_workspace_size(M, K) + w8.splitk_workspace_size(M, N, K),
                     dtype=torch.uint8, device=DEV)
    y = w8.scaled_mm(xq.to(DEV), wq.to(DEV), sx.to(DEV), sw.to(DEV), "dyn_asym", zp=zp.to(DEV), azp_adj=adj.to(DEV),
                     w_mode=w_mode, workspace=ws)
    acc = oracle.int8_gemm(xq.numpy(), wq.numpy())
    swn = sw.numpy() if w_mode == w8.W_CHANNEL else np.full(N, sw.numpy()[0], dtype=np.float32)
    yb, y32 = oracle.scaled_mm_epilogue(acc, sx.numpy(), swn, zp=zp.numpy(), adj=adj.numpy())
    check_bf16(y, yb, y32)


def test_packed_linear_matches_int8_path():
    d = _gemm_case(200, 512, 2048, seed=21)
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    pa = w8.quantize_act_packed(d["x"].to(DEV))
    y1 = w8.scaled_mm_packed(pa, wq, sw, bias=d["b"].to(DEV))
    xq, sx, _ = w8.quantize_act(d["x"].to(DEV))
    y2 = w8.scaled_mm(xq, wq, sx, sw, bias=d["b"].to(DEV))
    y3 = w8.linear(d["x"].to(DEV), wq, sw, bias=d["b"].to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))
    r = oracle.w8a8_linear(d["xb"], d["rq"], d["rs"], bias_bits=wl.bits(d["b"]))
    check_bf16(y1, r["y_bits"], r["y32"])


def test_engines_agree_bitwise():
    d = _gemm_case(48, 768, 3072, seed=5)
    xq, sx, _ = w8.quantize_act(d["x"].to(DEV), "dyn_sym")
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    w8.set_gemm_engine(1)
    a = w8.scaled_mm(xq, wq, sx, sw)
    w8.set_gemm_engine(2)
    b = w8.scaled_mm(xq, wq, sx, sw)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------------ tiny config (config 1)

def test_tiny_linear_config():
    d = wl.tiny_linear(seed=0)
    wq, sw = w8.quantize_weight(d["w"].to(DEV))
    rq, rs = oracle.quantize_weight_per_channel(d["w"].float().numpy())
    np.testing.assert_array_equal(wq.cpu().numpy(), rq)
    y = w8.linear(d["x"].to(DEV), wq, sw, bias=d["bias"].to(DEV))
    r = oracle.w8a8_linear(wl.bits(d["x"]), rq, rs, bias_bits=wl.bits(d["bias"]))
    check_bf16(y, r["y_bits"], r["y32"])


# ------------------------------------------------------------------ Llama shapes at full size, sampled rows

@pytest.mark.parametrize("name,N,K", wl.llama_shapes())
def test_llama_full_size_sampled(name, N, K):
    M = 4096
    x = wl.llama_activations(M, K, seed=1)
    w = wl.weight_bf16(N, K, seed=2)
    wq, sw = w8.quantize_weight(w.to(DEV))
    y = w8.linear(x.to(DEV), wq, sw)
    torch.cuda.synchronize()
    rows = np.random.default_rng(N + K).choice(M, 24, replace=False)
    rows = np.concatenate([rows, [0, M - 1]])
    rq, rs = oracle.quantize_weight_per_channel(w.float().numpy())
    np.testing.assert_array_equal(sw.cpu().numpy(), rs)
    r = oracle.w8a8_linear(wl.bits(x)[rows], rq, rs)
    check_bf16(y[torch.from_numpy(rows).to(DEV)], r["y_bits"], r["y32"])


@pytest.mark.parametrize("M", [1, 16, 128, 1024, 8192])
@pytest.mark.parametrize("name,N,K", wl.llama_shapes())
def test_llama_grid(name, N, K, M):
    """The rest of the Llama-3-8B grid ([vLLM-W8A8] 3.3, dynamic per-token activations): every
    linear at M = 1 and 16 (weight-streaming engine, all rows compared), 128 and 1024 (the
    tensor-core engine with its K split over idle CTA pairs) and 8192 (two waves of row tiles
    more than the headline M = 4096; sampled rows), through w8a8_linear as a user calls it."""
    x = wl.llama_activations(M, K, seed=M)
    w = wl.weight_bf16(N, K, seed=3)
    wq, sw = w8.quantize_weight(w.to(DEV))
    y = w8.linear(x.to(DEV), wq, sw)
    torch.cuda.synchronize()
    if M <= 16:
        rows = np.arange(M)
    else:
        rows = np.random.default_rng(N + K + M).choice(M, 24, replace=False)
        rows = np.concatenate([rows, [0, M - 1]])
    rq, rs = oracle.quantize_weight_per_channel(w.float().numpy())
    r = oracle.w8a8_linear(wl.bits(x)[rows], rq, rs)
    check_bf16(y[torch.from_numpy(rows).to(DEV)], r["y_bits"], r["y32"])


# ------------------------------------------------------------------ FP8 -> INT8 requant

@pytest.mark.parametrize("N,K", [(256, 4096), (300, 1500), (129, 1500), (5, 17), (384, 512), (70, 4), (130, 516),
                                 (33, 4092), (20, 4100)])
def test_fp8_requant(N, K):
    codes, sinv, _ = wl.fp8_block_matrix(N, K, seed=3, stream=N + K, zero_frac=0.01)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, s = w8.fp8block_to_int8_rowwise(codes.to(DEV), sinv.to(DEV), status=st)
    rq, rs, bad = oracle.fp8_block_to_int8_rowwise(codes.numpy(), sinv.numpy())
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    assert int(st.item()) == 0 and not bad.any()


@pytest.mark.parametrize("K", [384, 1500])
@pytest.mark.parametrize("bad_val", [0.0, -1.0, float("inf"), float("nan")])
def test_fp8_requant_illegal_scale(bad_val, K):
    codes, sinv, _ = wl.fp8_block_matrix(256, K, seed=2, stream=9, zero_frac=0.0)
    c, si = codes.clone(), sinv.clone()
    si[1, 2] = bad_val
    c[5, 7] = 0x7F
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, s = w8.fp8block_to_int8_rowwise(c.to(DEV), si.to(DEV), status=st)
    rq, rs, bad = oracle.fp8_block_to_int8_rowwise(c.numpy(), si.numpy())
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    assert int(st.item()) == 4


def test_requant_bounded_wait_runs_out_and_recovers():
    """Failure detection on the device without a GPU fault ([Kunlun-INT8] 验证 lists tests of
    illegal inputs): the test hook makes the first row's barrier of a requantizer ring launch
    expect 16 bytes more than its bulk copy delivers and shortens the wait limit to 5 ms.  The
    copy lands as usual, the wait runs out, the launch records W8A8_ERR_TIMEOUT (5) and
    returns; the next ordinary call on the same GPU is bit-exact."""
    lib = w8.lib()
    codes, sinv, _ = wl.fp8_block_matrix(8, 4096, seed=5, stream=1, zero_frac=0.0)
    cd, sd = codes.to(DEV), sinv.to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    assert lib.w8a8_test_requant_wait_fault(16, 5_000_000) == 0
    try:
        t0 = time.perf_counter()
        w8.fp8block_to_int8_rowwise(cd, sd, status=st)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        assert lib.w8a8_test_requant_wait_fault(0, 0) == 0
    assert int(st.item()) == 5
    assert elapsed < 1.0  # ended by the shortened limit, not the default 2 s
    st.zero_()
    q, s = w8.fp8block_to_int8_rowwise(cd, sd, status=st)
    rq, rs, bad = oracle.fp8_block_to_int8_rowwise(codes.numpy(), sinv.numpy())
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    assert int(st.item()) == 0 and not bad.any()


@pytest.mark.parametrize("N,K", [(9, 8192), (9, 20480), (5, 65536), (140, 4112)])
def test_fp8_requant_long_rows(N, K):
    """Row lengths that take the 8- and 4-warp shared-memory rings, the streaming kernel
    (rows longer than a ring slot) and a partial last column block."""
    codes, sinv, _ = wl.fp8_block_matrix(N, K, seed=5, stream=K, zero_frac=0.0)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, s = w8.fp8block_to_int8_rowwise(codes.to(DEV), sinv.to(DEV), status=st)
    rq, rs, bad = oracle.fp8_block_to_int8_rowwise(codes.numpy(), sinv.numpy())
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    assert int(st.item()) == 0 and not bad.any()


@pytest.mark.parametrize("K,col,code", [(4112, 4100, 0x7F), (4096, 0, 0xFF), (65536, 65535, 0xFF)])
def test_fp8_requant_nan_code(K, col, code):
    """An E4M3 NaN code (either sign) anywhere in a row, including a partial last block and
    a streamed row, zeroes that row and reports a bad scale."""
    codes, sinv, _ = wl.fp8_block_matrix(3, K, seed=6, stream=col, zero_frac=0.0)
    c = codes.clone()
    c[1, col] = code
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, s = w8.fp8block_to_int8_rowwise(c.to(DEV), sinv.to(DEV), status=st)
    rq, rs, bad = oracle.fp8_block_to_int8_rowwise(c.numpy(), sinv.numpy())
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    assert bad[1] and not bad[0] and not bad[2]
    assert int(st.item()) == 4


def test_fp8_requant_batched_mixed():
    mats = [wl.fp8_block_matrix(*shape, seed=4, stream=i) for i, shape in
            enumerate([(512, 4096), (300, 1500), (64, 4096), (3000, 1500), (130, 4112)])]
    dev = [(c.to(DEV), s.to(DEV)) for c, s, _ in mats]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = w8.fp8block_to_int8_rowwise_batched(dev, status=st)
    for (c, s, _), (q, sq) in zip(mats, outs):
        rq, rs, _ = oracle.fp8_block_to_int8_rowwise(c.numpy(), s.numpy())
        np.testing.assert_array_equal(q.cpu().numpy(), rq)
        np.testing.assert_array_equal(sq.cpu().numpy(), rs)
    assert int(st.item()) == 0


def test_fp8_requant_batched_adj():
    """The requantizer's optional row sums (the converted weight's azp_adj) on every path:
    the shared-memory ring (K = 4096, 4112), the streaming kernel (K = 65536), the byte path
    (K = 1500), a zero row, and rows zeroed by an illegal block scale and a NaN code; the codes
    and scales must be unchanged by asking for the sums."""
    mats = [wl.fp8_block_matrix(*shape, seed=6, stream=i) for i, shape in
            enumerate([(512, 4096), (300, 1500), (5, 65536), (130, 4112)])]
    mats = [(c.clone(), si.clone()) for c, si, _ in mats]
    mats[0][1][1, 2] = 0.0      # rows 128..255 of the first matrix: illegal scale
    mats[3][0][5, 7] = 0x7F     # row 5 of the last: a NaN code
    mats[1][0][17, :] = 0       # an all-zero row
    dev = [(c.to(DEV), si.to(DEV)) for c, si in mats]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = w8.fp8block_to_int8_rowwise_batched(dev, status=st, azp_adj=True)
    plain = w8.fp8block_to_int8_rowwise_batched(dev)
    for (c, si), (q, sq, adj), (q0, s0) in zip(mats, outs, plain):
        rq, rs, _ = oracle.fp8_block_to_int8_rowwise(c.numpy(), si.numpy())
        np.testing.assert_array_equal(q.cpu().numpy(), rq)
        np.testing.assert_array_equal(sq.cpu().numpy(), rs)
        np.testing.assert_array_equal(adj.cpu().numpy(), oracle.azp_adj(rq))
        assert torch.equal(q, q0) and torch.equal(sq, s0)
    assert int(st.item()) == 4


def test_fp8_requant_full_config_sampled():
    """The requant workload (64 x [6144,4096] + 8 x [3000,1500]) in its batched launch;
    sampled rows of every matrix against the oracle, zero rows checked exactly."""
    mats = wl.requant_workload(n_big=64, n_ragged=8)
    dev = [(c.to(DEV), s.to(DEV)) for c, s, _ in mats]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = w8.fp8block_to_int8_rowwise_batched(dev, status=st)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    for (c, s, zr), (q, sq) in zip(mats, outs):
        N = c.shape[0]
        rows = np.unique(np.concatenate([rng.choice(N, 6, replace=False), zr.numpy()[:2], [N - 1]]))
        rb = (rows // 128)
        # oracle on the sampled rows: give each row its own block-row of scales
        rq = np.zeros((len(rows), c.shape[1]), np.int8)
        rs = np.zeros(len(rows), np.float32)
        cn, sn = c.numpy(), s.numpy()
        for j, i in enumerate(rows):
            qq, ss, _ = oracle.fp8_block_to_int8_rowwise(cn[i:i + 1], sn[rb[j]:rb[j] + 1])
            rq[j], rs[j] = qq[0], ss[0]
        idx = torch.from_numpy(rows).to(DEV)
        np.testing.assert_array_equal(q[idx].cpu().numpy(), rq)
        np.testing.assert_array_equal(sq[idx].cpu().numpy(), rs)
        zrows = zr.to(DEV)
        assert torch.all(sq[zrows] == 1.0) and not q[zrows].any()
    assert int(st.item()) == 0


# ------------------------------------------------------------------ MoE

def _moe_setup(T, H, E, topk, inter, seed):
    d = wl.moe_workload(T=T, H=H, E=E, topk=topk, inter=inter, seed=seed)
    ids = d["topk_ids"].numpy()
    tok, slot, seg = oracle.moe_sort(ids, E)
    row_of = np.zeros((T, topk), np.int64)
    row_of[tok, slot] = np.arange(len(tok))
    w13q, s13 = w8.quantize_weight(d["w13"].reshape(E * 2 * inter, H).to(DEV))
    w2q, s2 = w8.quantize_weight(d["w2"].reshape(E * H, inter).to(DEV))
    dev = dict(x=d["x"].to(DEV), row_index=torch.from_numpy(tok).to(DEV), seg=torch.from_numpy(seg).to(DEV),
               row_of=torch.from_numpy(row_of).to(DEV), topk_w=d["topk_w"].to(DEV),
               w13=w13q.view(E, 2 * inter, H), s13=s13.view(E, 2 * inter), w2=w2q.view(E, H, inter),
               s2=s2.view(E, H))
    return d, dev, tok, seg


@pytest.mark.parametrize("engine", [1, 2])
def test_moe_small_full_compare(engine):
    w8.set_gemm_engine(engine)
    T, H, E, k, inter = 96, 256, 8, 2, 128
    d, dev, tok, seg = _moe_setup(T, H, E, k, inter, seed=7)
    y, h, o = w8.moe_forward(dev["x"], dev["row_index"], dev["seg"], dev["row_of"], dev["topk_w"], dev["w13"],
                             dev["s13"], dev["w2"], dev["s2"])
    r = oracle.moe_forward(wl.bits(d["x"]), d["topk_ids"].numpy(), d["topk_w"].numpy(),
                           dev["w13"].cpu().numpy(), dev["s13"].cpu().numpy(), dev["w2"].cpu().numpy(),
                           dev["s2"].cpu().numpy())
    # the first expert GEMM sees identical int8 inputs: exact
    np.testing.assert_array_equal(npbits(h), r["h_bits"])
    # after the fp32 SiLU glue, compare within the stated bf16 tolerance
    check_bf16(y, r["y_bits"], r["y32"], exact=False)


def test_moe_weight_squares_exact():
    """With the expert weights' sums of squares, grouped tiles whose activation rows fail the
    L1 test (every 37th token made nearly constant in magnitude, so its codes are near +-127)
    may run one pass by the Cauchy-Schwarz test (weights indexed by expert): the expert GEMMs'
    outputs equal the runs without squares and the oracle, bit for bit."""
    T, H, E, k, inter = 512, 4096, 8, 2, 256
    d, dev, tok, seg = _moe_setup(T, H, E, k, inter, seed=9)
    x = d["x"].float()
    x[::37] = torch.where(x[::37] >= 0, 1.0, -1.0) * (1.0 + 0.01 * torch.rand(x[::37].shape,
                                                      generator=torch.Generator().manual_seed(3)))
    x = x.to(torch.bfloat16)
    xd = x.to(DEV)
    w13sq = w8.weight_sumsq(dev["w13"].reshape(E * 2 * inter, H)).view(E, 2 * inter)
    w2sq = w8.weight_sumsq(dev["w2"].reshape(E * H, inter)).view(E, H)
    args = (xd, dev["row_index"], dev["seg"], dev["row_of"], dev["topk_w"], dev["w13"], dev["s13"], dev["w2"],
            dev["s2"])
    y1, h1, o1 = w8.moe_forward(*args)
    y2, h2, o2 = w8.moe_forward(*args, w13_sumsq=w13sq, w2_sumsq=w2sq)
    assert torch.equal(h1, h2) and torch.equal(o1, o2) and torch.equal(y1, y2)
    r = oracle.moe_forward(wl.bits(x), d["topk_ids"].numpy(), d["topk_w"].numpy(),
                           dev["w13"].cpu().numpy(), dev["s13"].cpu().numpy(), dev["w2"].cpu().numpy(),
                           dev["s2"].cpu().numpy())
    np.testing.assert_array_equal(npbits(h2), r["h_bits"])
    check_bf16(y2, r["y_bits"], r["y32"], exact=False)


def test_moe_full_config_sampled():
    T, H, E, k, inter = 4096, 4096, 32, 4, 1408
    d, dev, tok, seg = _moe_setup(T, H, E, k, inter, seed=0)
    assert seg[-1] == T * k
    y, h, o = w8.moe_forward(dev["x"], dev["row_index"], dev["seg"], dev["row_of"], dev["topk_w"], dev["w13"],
                             dev["s13"], dev["w2"], dev["s2"])
    torch.cuda.synchronize()
    rows = np.concatenate([np.random.default_rng(1).choice(T, 6, replace=False), [0, T - 1]])
    r = oracle.moe_forward(wl.bits(d["x"]), d["topk_ids"].numpy(), d["topk_w"].numpy(),
                           dev["w13"].cpu().numpy(), dev["s13"].cpu().numpy(), dev["w2"].cpu().numpy(),
                           dev["s2"].cpu().numpy(), rows=rows)
    sel_rows = np.nonzero(np.isin(tok, rows))[0]
    np.testing.assert_array_equal(npbits(h)[sel_rows], r["h_bits"][sel_rows])
    # the second expert GEMM, exact at full size: the GPU's own SiLU*up codes and scales go
    # through w8a8_grouped_mm (int8 entry point) and, for the sampled tokens' rows, through the
    # oracle's int8 GEMM + epilogue; both must equal the layer's own expert-2 output bit for bit
    gq, sg = w8.silu_mul_quant(h)
    o2 = w8.grouped_mm(gq, sg, dev["w2"], dev["s2"], dev["seg"])
    torch.cuda.synchronize()
    assert torch.equal(o2.view(torch.int16), o.view(torch.int16))
    gqn, sgn, ob = gq.cpu().numpy(), sg.cpu().numpy(), npbits(o)
    w2n, s2n = dev["w2"].cpu().numpy(), dev["s2"].cpu().numpy()
    for e in range(E):
        sel = sel_rows[(sel_rows >= seg[e]) & (sel_rows < seg[e + 1])]
        if len(sel) == 0:
            continue
        acc = oracle.int8_gemm(gqn[sel], w2n[e])
        eb, _ = oracle.scaled_mm_epilogue(acc, sgn[sel], s2n[e])
        np.testing.assert_array_equal(ob[sel], eb)
    # the combined output against the oracle's float32 sums (before their bf16 rounding)
    check_bf16(y[torch.from_numpy(rows).to(DEV)], r["y_bits"][rows], r["y32"][rows], exact=False)


def test_grouped_mm_empty_segments():
    E, N, K = 5, 256, 512
    seg = torch.tensor([0, 0, 130, 130, 131, 300], dtype=torch.int64)
    R = 300
    xq = torch.randint(-127, 128, (R, K), dtype=torch.int8)
    wq = torch.randint(-127, 128, (E, N, K), dtype=torch.int8)
    sx = torch.rand(R, dtype=torch.float32)
    sw = torch.rand(E, N, dtype=torch.float32) * 1e-3
    y = w8.grouped_mm(xq.to(DEV), sx.to(DEV), wq.to(DEV), sw.to(DEV), seg.to(DEV))
    w8.set_gemm_engine(2)
    y2 = w8.grouped_mm(xq.to(DEV), sx.to(DEV), wq.to(DEV), sw.to(DEV), seg.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    for e in range(E):
        a, b = int(seg[e]), int(seg[e + 1])
        if a == b:
            continue
        acc = oracle.int8_gemm(xq[a:b].numpy(), wq[e].numpy())
        yb, y32 = oracle.scaled_mm_epilogue(acc, sx[a:b].numpy(), sw[e].numpy())
        check_bf16(y[a:b], yb, y32)


def test_grouped_mm_max_segments():
    """The largest segment count the tensor-core engine's work list holds (1024): mostly empty
    segments, single rows, a segment at the very end, and one of 300 rows (two row tiles);
    a segment count one past the limit is refused.  Bit-exact against the oracle per segment
    and against the warp-MMA engine."""
    E, N, K = 1024, 72, 96
    lens = np.zeros(E, dtype=np.int64)
    lens[[0, 1, 5, 511, 512, 1000]] = [1, 2, 3, 1, 300, 17]
    lens[E - 1] = 4
    seg = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int64))
    R = int(seg[-1])
    g = torch.Generator().manual_seed(11)
    xq = torch.randint(-127, 128, (R, K), dtype=torch.int8, generator=g)
    wq = torch.randint(-127, 128, (E, N, K), dtype=torch.int8, generator=g)
    sx = torch.rand(R, dtype=torch.float32, generator=g) * 1e-2
    sw = torch.rand(E, N, dtype=torch.float32, generator=g) * 1e-3
    y = w8.grouped_mm(xq.to(DEV), sx.to(DEV), wq.to(DEV), sw.to(DEV), seg.to(DEV))
    w8.set_gemm_engine(2)
    y2 = w8.grouped_mm(xq.to(DEV), sx.to(DEV), wq.to(DEV), sw.to(DEV), seg.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    for e in np.nonzero(lens)[0]:
        a, b = int(seg[e]), int(seg[e + 1])
        acc = oracle.int8_gemm(xq[a:b].numpy(), wq[e].numpy())
        yb, y32 = oracle.scaled_mm_epilogue(acc, sx[a:b].numpy(), sw[e].numpy())
        check_bf16(y[a:b], yb, y32)
    w8.set_gemm_engine(0)
    seg2 = torch.cat([seg, seg[-1:]])
    wq2 = torch.zeros((E + 1, N, K), dtype=torch.int8)
    sw2 = torch.zeros((E + 1, N), dtype=torch.float32)
    with pytest.raises(w8.W8A8Error):
        w8.grouped_mm(xq.to(DEV), sx.to(DEV), wq2.to(DEV), sw2.to(DEV), seg2.to(DEV))


@pytest.mark.parametrize("widths,K", [([4096, 1024, 1024], 4096), ([300, 77, 0, 129], 1500), ([64], 512),
                                      ([3, 5], 4112)])
def test_requantize_max_scale(widths, K):
    """Fused Q/K/V-style weights with per-partition tensor scales, requantized in place to
    the largest scale: bit-exact against the oracle (Llama-3-8B q/k/v widths; a ragged K on
    the byte path with an empty partition; one partition = no change; tiny partitions)."""
    N = sum(widths)
    rng = np.random.default_rng(N + K)
    q = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    sc = rng.uniform(1e-4, 3e-3, size=len(widths)).astype(np.float32)
    want, want_s = oracle.requantize_with_max_scale(q, sc, widths)
    wq = torch.from_numpy(q).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    s_max = w8.requantize_max_scale(wq, torch.from_numpy(sc).to(DEV), widths, status=st)
    np.testing.assert_array_equal(wq.cpu().numpy(), want)
    assert s_max.item() == float(want_s) and int(st.item()) == 0


@pytest.mark.parametrize("bad", [0.0, -1.0, float("inf"), float("nan")])
def test_requantize_max_scale_bad_scale(bad):
    q = torch.randint(-127, 128, (40, 64), dtype=torch.int8)
    wq = q.to(DEV)
    s_max = torch.full((1,), 7.0, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sc = torch.tensor([1e-3, bad, 2e-3], dtype=torch.float32, device=DEV)
    s_max = w8.requantize_max_scale(wq, sc, [10, 10, 20], status=st)
    assert torch.equal(wq.cpu(), q) and int(st.item()) == 4


def _route_expected(lg, k):
    ids, w = oracle.moe_route(lg, k)
    tok, slot, seg = oracle.moe_sort(ids, lg.shape[1])
    row_of = np.zeros(ids.shape, np.int64)
    row_of[tok, slot] = np.arange(len(tok))
    return ids, w, seg, tok, row_of


@pytest.mark.parametrize("T,E,k,kind", [(4096, 32, 4, "workload"), (300, 256, 8, "normal"), (777, 60, 3, "ties"),
                                        (1, 1, 1, "normal"), (5, 33, 2, "ties"), (0, 8, 2, "normal")])
def test_moe_route(T, E, k, kind):
    """Top-k ids, segment offsets and both row maps bit-exact against the oracle (ties to the
    lower expert; stable by token then slot); weights within 1e-5 relative (fp32 softmax with
    expf against the oracle's float64: a few fp32 roundings over at most 256 terms)."""
    if kind == "workload":
        lg = wl.moe_workload(T=T, H=64, E=E, topk=k, inter=64, seed=3, with_weights=False)["logits"].numpy()
    else:
        rng = np.random.default_rng(T * 1000 + E)
        lg = rng.standard_normal((T, E)).astype(np.float32)
        if kind == "ties":
            lg = np.round(lg * 2).astype(np.float32)
    ids, w, seg, row_index, row_of = w8.moe_route(torch.from_numpy(lg).to(DEV), k)
    rid, rw, rseg, rtok, rrow = _route_expected(lg, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_array_equal(seg.cpu().numpy(), rseg)
    np.testing.assert_array_equal(row_index.cpu().numpy(), rtok)
    np.testing.assert_array_equal(row_of.cpu().numpy(), rrow)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-5, atol=0)


@pytest.mark.parametrize("T,K,topk,E", [(4096, 4096, 4, 32), (37, 1040, 3, 5), (1, 16, 1, 1), (300, 14336, 8, 64)])
def test_moe_quantize_scatter_matches_gather(T, K, topk, E):
    """Each token quantized once and written to its routed rows gives the packed buffer
    (fp16 codes, L1 norms) and scales of quantizing every routed row from its token, bit for
    bit, and both equal the oracle's per-token quantization of the gathered rows."""
    g = torch.Generator().manual_seed(T + K)
    x = wl.llama_activations(T, K, seed=T * 3 + K)
    ids = torch.stack([torch.randperm(E, generator=g)[:topk] for _ in range(T)]).reshape(-1)
    order = torch.argsort(ids, stable=True)
    row_index = order // topk
    row_of = torch.empty(T * topk, dtype=torch.int64)
    row_of[order] = torch.arange(T * topk)
    xd = x.to(DEV)
    ga = w8.moe_quantize_gather_packed(xd, row_index.to(DEV))
    sa = w8.moe_quantize_scatter_packed(xd, row_of.view(T, topk).to(DEV))
    torch.cuda.synchronize()
    R = T * topk
    assert torch.equal(ga.buf[: R * K * 2], sa.buf[: R * K * 2])
    assert torch.equal(ga.norms(), sa.norms())
    assert torch.equal(ga.scale, sa.scale)
    rq, rs = oracle.quantize_act_dynamic_symmetric(x.float().numpy()[row_index.numpy()])
    np.testing.assert_array_equal(sa.codes().float().cpu().numpy().astype(np.int8), rq)
    np.testing.assert_array_equal(sa.scale.cpu().numpy(), rs)
    np.testing.assert_array_equal(sa.norms().cpu().numpy(), np.abs(rq.astype(np.int64)).sum(1))


@pytest.mark.parametrize("topk", [1, 3, 8, 9, 12])
def test_moe_combine_slots(topk):
    """The combine step bit for bit against the oracle: up to 8 slots take the kernel that
    reads a token's routed rows together, more slots (9, 12) the plain per-slot loop."""
    T, H = 300, 520
    R = T * topk
    g = np.random.default_rng(topk)
    out = torch.from_numpy(g.standard_normal((R, H)).astype(np.float32)).to(torch.bfloat16)
    row_of = torch.from_numpy(g.permutation(R).reshape(T, topk).astype(np.int64))
    tw = torch.from_numpy(g.random((T, topk)).astype(np.float32))
    y = w8.moe_combine(out.to(DEV), row_of.to(DEV), tw.to(DEV))
    yb, y32 = oracle.moe_combine(wl.bits(out), row_of.numpy(), tw.numpy())
    check_bf16(y, yb, y32)


def test_moe_route_feeds_moe_forward():
    """The routed outputs drive the MoE layer end to end: the same result as the oracle layer
    given the oracle's routing (the weights within the routing tolerance)."""
    T, H, E, k, inter = 96, 256, 8, 2, 128
    d = wl.moe_workload(T=T, H=H, E=E, topk=k, inter=inter, seed=9)
    ids, w, seg, row_index, row_of = w8.moe_route(d["logits"].to(DEV), k)
    w13q, s13 = w8.quantize_weight(d["w13"].reshape(E * 2 * inter, H).to(DEV))
    w2q, s2 = w8.quantize_weight(d["w2"].reshape(E * H, inter).to(DEV))
    y, h, o = w8.moe_forward(d["x"].to(DEV), row_index, seg, row_of, w, w13q.view(E, 2 * inter, H),
                             s13.view(E, 2 * inter), w2q.view(E, H, inter), s2.view(E, H))
    rid, rw = oracle.moe_route(d["logits"].numpy(), k)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    r = oracle.moe_forward(wl.bits(d["x"]), rid, rw.astype(np.float32), w13q.view(E, 2 * inter, H).cpu().numpy(),
                           s13.view(E, 2 * inter).cpu().numpy(), w2q.view(E, H, inter).cpu().numpy(),
                           s2.view(E, H).cpu().numpy())
    np.testing.assert_array_equal(npbits(h), r["h_bits"])
    check_bf16(y, r["y_bits"], r["y32"], exact=False)



@pytest.mark.parametrize("act", ["dyn_asym", "static_asym"])
@pytest.mark.parametrize("M", [300, 4096])
def test_asym_linear_cauchy_schwarz(act, M):
    """Affine codes of nonzero-mean rows at K = 4096 have L1 norms above 2^17, so without the
    weight's sums of squares every tile runs the chunked mode; with them the Cauchy-Schwarz
    bound admits single-pass tiles.  Both must equal the oracle bit for bit (M = 4096 on
    sampled rows)."""
    N, K = 520, 4096
    d = _gemm_case(M, N, K, seed=M + 17, act=act)
    xs = d["x"].float().numpy()
    sc, z = oracle.static_scale_from_tensor(xs)
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    kw = {}
    if act == "dyn_asym":
        kw["azp_adj"] = w8.azp_adj(wq)
    else:
        kw["input_scale"] = torch.tensor([sc], dtype=torch.float32, device=DEV)
        kw["input_zero_point"] = torch.tensor([z], dtype=torch.int32, device=DEV)
        kw["azp_adj"] = w8.azp_adj(wq, kw["input_zero_point"])
    wsq = w8.weight_sumsq(wq)
    np.testing.assert_array_equal(wsq.cpu().numpy(), (d["rq"].astype(np.int64) ** 2).sum(1))
    x = d["x"].to(DEV)
    y_cs = w8.linear(x, wq, sw, act_mode=act, bias=d["b"].to(DEV), w_sumsq=wsq, **kw)
    y_l1 = w8.linear(x, wq, sw, act_mode=act, bias=d["b"].to(DEV), **kw)
    assert torch.equal(y_cs, y_l1)
    rows = np.arange(M) if M <= 300 else np.concatenate([np.arange(0, M, 97), [M - 1]])
    r = oracle.w8a8_linear(d["xb"][rows], d["rq"], d["rs"], bias_bits=wl.bits(d["b"]), mode=act,
                           input_scale=sc, input_zero_point=z)
    check_bf16(y_cs[torch.from_numpy(rows).to(DEV)], r["y_bits"], r["y32"])


@pytest.mark.parametrize("qv,wv,cs_ok", [(40, 20, True), (127, 127, False), (-90, 31, True)])
def test_gemm_cauchy_schwarz_bound_exact(qv, wv, cs_ok):
    """Rows of |q| = qv over K = 4096 have L1 norm 4096 qv >= 2^17, so only the Cauchy-Schwarz
    test (K qv^2 * K wv^2 < 2^48) can make their tiles single pass; signs are chosen so that
    every product in a row/column pair has the same sign (the largest partial sums the bound
    allows).  (127, 127) fails both tests and runs chunked.  All exact."""
    M, N, K = 256, 512, 4096
    assert (K * qv * qv) * (K * wv * wv) < 2 ** 48 if cs_ok else (K * qv * qv) * (K * wv * wv) >= 2 ** 48
    rng = np.random.default_rng(abs(qv) + wv)
    sx = rng.choice([-1, 1], size=(M, 1)).astype(np.int64)
    sk = rng.choice([-1, 1], size=(1, K)).astype(np.int64)
    sn = rng.choice([-1, 1], size=(N, 1)).astype(np.int64)
    xq = (qv * sx * sk).astype(np.int8)
    wq = (wv * sn * sk).astype(np.int8)
    xq[7, :100] = 0  # a row of smaller norm in the same tile
    s_x = np.full(M, 2.0 ** -10, np.float32)
    s_w = np.full(N, 2.0 ** -12, np.float32)
    wq_d = torch.from_numpy(wq).to(DEV)
    y = w8.scaled_mm(torch.from_numpy(xq).to(DEV), wq_d, torch.from_numpy(s_x).to(DEV), torch.from_numpy(s_w).to(DEV),
                     "dyn_sym", w_sumsq=w8.weight_sumsq(wq_d))
    acc = oracle.int8_gemm(xq, wq)
    yb, y32 = oracle.scaled_mm_epilogue(acc, s_x, s_w)
    check_bf16(y, yb, y32)


@pytest.mark.parametrize("M,N,K", [(1, 520, 4112), (3, 5000, 4096), (8, 300, 64), (8, 1000, 11200), (5, 4104, 4096)])
def test_decode_linear_fused_quant(M, N, K):
    """Decode linears (dynamic symmetric, at most 8 rows) quantize inside the small-M GEMM:
    bf16 outputs equal the oracle's quantizer + GEMM + epilogue bit for bit, including a zero
    row and rows built on exact and near ties of x / s."""
    d = _gemm_case(M, N, K, seed=M * 31 + K)
    x = d["x"].clone()
    if M >= 3:
        x[1] = 0
        ties = _sym_tie_rows(K)
        x[2] = ties[2 % ties.shape[0]]
    if M >= 5:
        x[4] = ties[0]
    xb = wl.bits(x)
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    y = w8.linear(x.to(DEV), wq, sw, bias=d["b"].to(DEV))
    r = oracle.w8a8_linear(xb, d["rq"], d["rs"], bias_bits=wl.bits(d["b"]))
    check_bf16(y, r["y_bits"], r["y32"])


@pytest.mark.parametrize("kind", ["normal", "zero", "tie_s1", "tie_near", "tie_small"])
@pytest.mark.parametrize("N,K", [(520, 4112), (300, 64), (1000, 11200)])
def test_decode_linear_fused_single_row(kind, N, K):
    """A single token row takes the fused quantizer + small-M GEMM: bit-exact against the
    oracle for ordinary, zero and tie-heavy rows (exact ties with s = 1, bf16 near-ties with
    s = RN(100/127), values around +-s/2 and +-3s/2)."""
    d = _gemm_case(1, N, K, seed=K + N)
    x = d["x"].clone()
    ties = _sym_tie_rows(K)
    if kind == "zero":
        x[0] = 0
    elif kind != "normal":
        x[0] = ties[{"tie_s1": 0, "tie_near": 2, "tie_small": 3}[kind]]
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    y = w8.linear(x.to(DEV), wq, sw, bias=d["b"].to(DEV))
    r = oracle.w8a8_linear(wl.bits(x), d["rq"], d["rs"], bias_bits=wl.bits(d["b"]))
    check_bf16(y, r["y_bits"], r["y32"])


@pytest.mark.parametrize("kind", ["nonzero_mean", "zero", "stress0", "stress1", "stress2", "stress3", "stress4",
                                  "stress5", "stress6", "stress7"])
@pytest.mark.parametrize("N,K", [(520, 4112), (300, 64), (1000, 11200)])
def test_decode_linear_fused_asym_single_row(kind, N, K):
    """A single token row with dynamic asymmetric quantization ([vLLM-W8A8] 4.1; the zero
    point enters the epilogue through azp_adj, [SGLang-CT] item 4) takes the fused quantizer +
    small-M GEMM: bit-exact against the oracle and against the two-launch path (stand-alone
    quantizer, then the GEMM) for rows far from zero, constant rows (hi == lo: the symmetric
    fallback), rows of two values, tiny magnitudes, exact ties and an all-zero row."""
    d = _gemm_case(1, N, K, seed=3 * K + N, act="dyn_asym")
    x = d["x"].clone()
    if kind == "zero":
        x[0] = 0
    elif kind.startswith("stress"):
        x[0] = _asym_stress_rows(K)[int(kind[-1])]
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    adj = w8.azp_adj(wq)
    b = d["b"].to(DEV)
    y = w8.linear(x.to(DEV), wq, sw, act_mode="dyn_asym", azp_adj=adj, bias=b)
    xq, sx, zp = w8.quantize_act(x.to(DEV), "dyn_asym")
    y2 = w8.scaled_mm(xq, wq, sx, sw, "dyn_asym", zp=zp, azp_adj=adj, bias=b)
    r = oracle.w8a8_linear(wl.bits(x), d["rq"], d["rs"], bias_bits=wl.bits(d["b"]), mode="dyn_asym")
    check_bf16(y, r["y_bits"], r["y32"])
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("bias", [True, False])
def test_decode_linear_fused_tensor_scale(bias):
    """The fused single-row path with a per-tensor weight scale, with and without bias."""
    N, K = 1000, 4096
    d = _gemm_case(1, N, K, seed=77, bias=bias, w_mode=w8.W_TENSOR)
    wq = torch.from_numpy(d["rq"]).to(DEV)
    sw = torch.from_numpy(d["rs"]).to(DEV)
    b = d["b"].to(DEV) if bias else None
    y = w8.linear(d["x"].to(DEV), wq, sw, bias=b, w_mode=w8.W_TENSOR)
    r = oracle.w8a8_linear(d["xb"], d["rq"], d["rs"], bias_bits=wl.bits(d["b"]) if bias else None)
    check_bf16(y, r["y_bits"], r["y32"])


def test_concurrent_host_threads():
    """Two host threads, each on its own stream, call the library concurrently (the per-device
    launch caches are per thread): both results equal a single-threaded run bit for bit."""
    import threading
    cases = []
    for i, (M, N, K) in enumerate([(300, 520, 4096), (1, 4096, 4096)]):
        d = _gemm_case(M, N, K, seed=300 + i)
        wq = torch.from_numpy(d["rq"]).to(DEV)
        sw = torch.from_numpy(d["rs"]).to(DEV)
        x = d["x"].to(DEV)
        ref = w8.linear(x, wq, sw)
        cases.append((x, wq, sw, ref))
    torch.cuda.synchronize()
    errors = []

    def run(case):
        x, wq, sw, ref = case
        s = torch.cuda.Stream()
        try:
            with torch.cuda.stream(s):
                for _ in range(10):
                    y = w8.linear(x, wq, sw)
                    s.synchronize()
                    if not torch.equal(y, ref):
                        errors.append("mismatch")
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(c,)) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


@pytest.mark.parametrize("engine", [1, 2])
def test_static_asym_epilogue_ranges(engine):
    """Static asymmetric outputs are (s_x s_w) f32(acc - azp'[n]) with the premultiplied azp'.
    Groups of 8 columns put azp' below 2^22, in [2^22, 2^24) and beyond 2^24 (each handled
    differently by the tensor-core epilogue); every output equals the oracle's exact int64
    difference rounded once."""
    w8.set_gemm_engine(engine)
    M, N, K = 300, 512, 1024
    rng = np.random.default_rng(41)
    xq = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    wq = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    mags = np.array([2 ** 10, 2 ** 21 + 3, 2 ** 23 - 5, 2 ** 24 + 7, 2 ** 30 + 11], dtype=np.int64)
    adj = np.empty(N, dtype=np.int64)
    for gi in range(N // 8):
        m = mags[gi % len(mags)]
        adj[8 * gi: 8 * gi + 8] = rng.integers(-m, m, size=8)
    adj = adj.astype(np.int32)
    s_x = np.array([2.0 ** -9], dtype=np.float32)
    s_w = (rng.random(N) * 1e-3 + 1e-4).astype(np.float32)
    y = w8.scaled_mm(torch.from_numpy(xq).to(DEV), torch.from_numpy(wq).to(DEV), torch.from_numpy(s_x).to(DEV),
                     torch.from_numpy(s_w).to(DEV), "static_asym", azp_adj=torch.from_numpy(adj).to(DEV))
    acc = oracle.int8_gemm(xq, wq)
    yb, y32 = oracle.scaled_mm_epilogue(acc, np.repeat(s_x, M), s_w, adj=adj, adj_premultiplied=True)
    check_bf16(y, yb, y32)
