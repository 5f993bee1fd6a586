"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties one oracle function to a hand-worked example from the pages' rules
(tests/golden/*.txt), a closed-form bound, an invariant, a brute-force integer
loop, or a library routine -- chosen so that a dropped term, a wrong sign, a
wrong index or a transposed operand in the oracle fails at least one of them.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from w8a8_int8_quantized_gb300 import workloads as wl

F32 = np.float32


def _floats(rows):
    return np.array([[float(v) for v in r] for r in rows], dtype=np.float32)


def _ints(rows):
    return np.array([[int(v, 0) for v in r] for r in rows], dtype=np.int64)


# ------------------------------------------------------------------ S1 / S7

def test_act_sym_worked_example():
    g = read_golden("act_quant_worked_examples.txt")
    x = _floats(g["x"])
    q, s = oracle.quantize_act_dynamic_symmetric(x)
    np.testing.assert_array_equal(q, _ints(g["q"]).astype(np.int8))
    np.testing.assert_array_equal(s, _floats(g["s"])[0])
    # the weight quantizer follows the same per-row rule
    qw, sw = oracle.quantize_weight_per_channel(x)
    np.testing.assert_array_equal(qw, q)
    np.testing.assert_array_equal(sw, s)


def _half_step_check(x, q, s, lo=-127, hi=127, zp=None):
    """|x - s*(q - zp)| <= s/2 (+ float32 rounding of the quotient) for unclamped entries."""
    x64 = x.astype(np.float64)
    s64 = s.astype(np.float64)[:, None]
    z = 0 if zp is None else zp.astype(np.float64)[:, None]
    rec = s64 * (q.astype(np.float64) - z)
    err = np.abs(x64 - rec)
    # quotient x/s is rounded to float32 before rint: allow |x/s| * 2^-24 extra steps
    bound = s64 * (0.5 + np.abs(x64 / s64) * 2.0 ** -23)
    inside = (q > lo) & (q < hi)
    assert np.all(err[inside] <= bound[inside]), float((err - bound)[inside].max())


def test_act_sym_half_step_bound_and_absmax():
    x = wl.llama_activations(64, 4096, seed=3).float().numpy()
    q, s = oracle.quantize_act_dynamic_symmetric(x)
    _half_step_check(x, q, s)
    # the absmax element of each row maps to +-127
    for m in range(x.shape[0]):
        j = int(np.argmax(np.abs(x[m])))
        assert abs(int(q[m, j])) == 127
        assert np.sign(q[m, j]) == np.sign(x[m, j])
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    # scale is absmax/127 up to one float32 rounding
    a = np.max(np.abs(x), axis=1).astype(np.float64)
    assert np.all(np.abs(s.astype(np.float64) - a / 127) <= a / 127 * 2.0 ** -24)


def test_act_sym_zero_rows_and_padding():
    x = wl.llama_activations(8, 1500, seed=4).float().numpy()
    x[3] = 0.0
    q, s = oracle.quantize_act_dynamic_symmetric(x)
    assert s[3] == 1.0 and not q[3].any()
    # a ragged row equals the same row padded with zeros to a multiple of 128
    xp = np.zeros((8, 1536), dtype=np.float32)
    xp[:, :1500] = x
    qp, sp = oracle.quantize_act_dynamic_symmetric(xp)
    np.testing.assert_array_equal(qp[:, :1500], q)
    np.testing.assert_array_equal(sp, s)
    assert not qp[:, 1500:].any()


def test_act_sym_sign_symmetry():
    """Negating a row negates q and keeps s (the rule is odd-symmetric)."""
    x = wl.llama_activations(16, 512, seed=5).float().numpy()
    q, s = oracle.quantize_act_dynamic_symmetric(x)
    qn, sn = oracle.quantize_act_dynamic_symmetric(-x)
    np.testing.assert_array_equal(qn, -q)
    np.testing.assert_array_equal(sn, s)


# ------------------------------------------------------------------ S3

def test_act_static_worked_example():
    g = read_golden("act_static_worked_examples.txt")
    x = _floats(g["x"])
    sc = float(g["scale"][0][0])
    zp = int(g["zp"][0][0])
    np.testing.assert_array_equal(oracle.quantize_act_static_symmetric(x, sc),
                                  _ints(g["q_sym"]).astype(np.int8))
    np.testing.assert_array_equal(oracle.quantize_act_static_asymmetric(x, sc, zp),
                                  _ints(g["q_asym"]).astype(np.int8))


def test_act_static_bounds():
    x = wl.asym_activations(32, 1024, seed=6).float().numpy()
    sc, zp = oracle.static_scale_from_tensor(x)
    assert -128 <= zp <= 127
    q = oracle.quantize_act_static_asymmetric(x, sc, zp)
    s = np.full(x.shape[0], sc, dtype=np.float32)
    _half_step_check(x, q, s, lo=-128, hi=127, zp=np.full(x.shape[0], zp))
    # the tensor min/max land on the ends of the int8 range (one step of slack)
    assert q.min() <= -127 and q.max() >= 126
    qs = oracle.quantize_act_static_symmetric(x, sc)
    _half_step_check(x, qs, s)


# ------------------------------------------------------------------ S2

def test_act_asym_worked_example():
    g = read_golden("act_asym_worked_examples.txt")
    x = _floats(g["x"])
    q, s, zp = oracle.quantize_act_dynamic_asymmetric(x)
    np.testing.assert_array_equal(q, _ints(g["q"]).astype(np.int8))
    np.testing.assert_array_equal(zp, _ints(g["zp"])[0].astype(np.int32))
    assert s[0] == 0.125 and s[1] == 0.125 and s[3] == 1.0
    assert s[2] == np.float32(np.float32(2.0) / np.float32(127))


def test_act_asym_invariants():
    x = wl.asym_activations(64, 4096, seed=7).float().numpy()
    q, s, zp = oracle.quantize_act_dynamic_asymmetric(x)
    _half_step_check(x, q, s, lo=-128, hi=127, zp=zp)
    for m in range(x.shape[0]):
        jlo, jhi = int(np.argmin(x[m])), int(np.argmax(x[m]))
        assert q[m, jlo] in (-128, -127)
        assert q[m, jhi] in (126, 127)
    # the asymmetric map of a row with lo = -hi*128/127 is the symmetric one
    # shifted by nothing: with zp = 0 both reconstruct within a half step
    assert zp.dtype == np.int32


# ------------------------------------------------------------------ S4 / S6

def _brute_gemm(a, b):
    M, K = a.shape
    N = b.shape[0]
    out = [[0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = 0
            for k in range(K):
                acc += int(a[m, k]) * int(b[n, k])
            out[m][n] = acc
    return np.array(out, dtype=np.int64)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 9, 64), (8, 16, 48)])
def test_int8_gemm_bruteforce(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    a = rng.integers(-128, 128, size=(M, K), dtype=np.int64).astype(np.int8)
    b = rng.integers(-127, 128, size=(N, K), dtype=np.int64).astype(np.int8)
    a[0, :] = -128
    b[0, :] = -127
    np.testing.assert_array_equal(oracle.int8_gemm(a, b).astype(np.int64), _brute_gemm(a, b))


def test_int8_gemm_not_transposed():
    """A non-square case where acc = a @ b.T differs from any transposed reading."""
    a = np.array([[1, 2, 3]], dtype=np.int8)        # [1, 3]
    b = np.array([[1, 0, 0], [0, 0, 2]], dtype=np.int8)  # [2, 3]
    np.testing.assert_array_equal(oracle.int8_gemm(a, b), np.array([[1, 6]], dtype=np.int32))


def test_int8_gemm_extreme_k():
    """Largest magnitudes at K = 14336: -128 * 127 * K fits int32 and is exact."""
    K = 14336
    a = np.full((2, K), -128, dtype=np.int8)
    a[1] = 127
    b = np.full((2, K), 127, dtype=np.int8)
    b[1] = -127
    acc = oracle.int8_gemm(a, b)
    assert acc[0, 0] == -128 * 127 * K and acc[1, 1] == -127 * 127 * K
    assert acc[0, 1] == 128 * 127 * K


def test_azp_adj_bruteforce_and_identity():
    rng = np.random.default_rng(11)
    M, N, K = 5, 7, 33
    w = rng.integers(-127, 128, size=(N, K), dtype=np.int64).astype(np.int8)
    q = rng.integers(-128, 128, size=(M, K), dtype=np.int64).astype(np.int8)
    zp = rng.integers(-200, 200, size=M).astype(np.int32)
    adj = oracle.azp_adj(w)
    for n in range(N):
        assert int(adj[n]) == sum(int(v) for v in w[n])
    acc = oracle.int8_gemm(q, w).astype(np.int64)
    lhs = np.zeros((M, N), dtype=np.int64)
    for m in range(M):
        for n in range(N):
            lhs[m, n] = sum((int(q[m, k]) - int(zp[m])) * int(w[n, k]) for k in range(K))
    np.testing.assert_array_equal(lhs, acc - zp.astype(np.int64)[:, None] * adj.astype(np.int64)[None, :])
    # static form: premultiplied by the zero point
    np.testing.assert_array_equal(oracle.azp_adj(w, -7), (-7 * adj.astype(np.int64)).astype(np.int32))


# ------------------------------------------------------------------ S5

def test_epilogue_worked_example():
    g = read_golden("epilogue_worked_examples.txt")
    acc = _ints(g["acc"]).astype(np.int32)
    sx = _floats(g["s_x"])[0]
    sw = _floats(g["s_w"])[0]
    bias = oracle.f32_to_bf16_bits(_floats(g["bias"])[0])
    yb, y = oracle.scaled_mm_epilogue(acc, sx, sw, bias_bits=bias)
    np.testing.assert_array_equal(y, _floats(g["y_sym"]))
    np.testing.assert_array_equal(oracle.bf16_bits_to_f32(yb), _floats(g["y_sym"]))
    zp = _ints(g["zp"])[0].astype(np.int32)
    adj = _ints(g["azp_adj"])[0].astype(np.int32)
    yb2, y2 = oracle.scaled_mm_epilogue(acc, sx, sw, zp=zp, adj=adj, bias_bits=bias)
    np.testing.assert_array_equal(y2, _floats(g["y_asym"]))
    # premultiplied static form gives the same result
    yb3, _ = oracle.scaled_mm_epilogue(acc, sx, sw, adj=(zp[0] * adj).astype(np.int32),
                                       adj_premultiplied=True, bias_bits=bias)
    np.testing.assert_array_equal(yb3, yb2)


def test_bf16_rounding_definition():
    # ties to even at the bf16 LSB, against the library cast
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -3.14159, 65504.0, 1e-40, 3.0e38], dtype=np.float32)
    ours = oracle.f32_to_bf16_bits(vals)
    lib = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, lib)
    r = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 100
    lib = torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.f32_to_bf16_bits(r), lib)


def test_linear_closed_form_bound():
    """Whole pipeline against the unquantized fp64 product.

    With x_hat = s_x * q_x and w_hat = s_w * q_w the dequantized operands,
    |x.w - s_x*s_w*acc| <= sum_k (|x_hat_k| * s_w/2 + |w_hat_k| * s_x/2 + s_x*s_w/4),
    plus the float32/bf16 rounding of the output.
    """
    d = wl.tiny_linear(seed=0)
    xb, wb, bb = wl.bits(d["x"]), wl.bits(d["w"]), wl.bits(d["bias"])
    x = oracle.bf16_bits_to_f32(xb).astype(np.float64)
    w = oracle.bf16_bits_to_f32(wb).astype(np.float64)
    qw, sw = oracle.quantize_weight_per_channel(w.astype(np.float32))
    r = oracle.w8a8_linear(xb, qw, sw, bias_bits=bb)
    exact = x @ w.T + oracle.bf16_bits_to_f32(bb).astype(np.float64)[None, :]
    sx = r["s_x"].astype(np.float64)
    xh = np.abs(r["q"].astype(np.float64)) * sx[:, None]
    wh = np.abs(qw.astype(np.float64)) * sw.astype(np.float64)[:, None]
    bound = (xh.sum(1)[:, None] * sw[None, :] / 2 + sx[:, None] * wh.sum(1)[None, :] / 2
             + sx[:, None] * sw[None, :] * x.shape[1] / 4)
    got = oracle.bf16_bits_to_f32(r["y_bits"]).astype(np.float64)
    assert np.all(np.abs(got - exact) <= bound + np.abs(exact) * 2 ** -8 + 1e-6)
    # and the bound is not vacuous: the error is well below the output scale
    assert np.median(np.abs(got - exact)) < 0.05 * np.median(np.abs(exact))


def test_linear_asym_matches_sym_when_zero_point_vanishes():
    """Dynamic asymmetric with zp = 0 everywhere reduces to the symmetric epilogue."""
    rng = np.random.default_rng(5)
    acc = rng.integers(-10 ** 6, 10 ** 6, size=(4, 6)).astype(np.int32)
    sx = rng.random(4).astype(np.float32)
    sw = rng.random(6).astype(np.float32)
    adj = rng.integers(-1000, 1000, size=6).astype(np.int32)
    a, _ = oracle.scaled_mm_epilogue(acc, sx, sw)
    b, _ = oracle.scaled_mm_epilogue(acc, sx, sw, zp=np.zeros(4, np.int32), adj=adj)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------------ S8

def test_e4m3_decode_table_and_library():
    g = read_golden("e4m3_codes.txt")
    for code, val in g["codes"]:
        v = oracle.e4m3_to_f32(np.array([int(code, 16)], dtype=np.uint8))[0]
        if val == "nan":
            assert np.isnan(v)
        else:
            assert v == np.float32(float(val)) and (math.copysign(1, v) == math.copysign(1, float(val)))
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f32(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(ours)
    np.testing.assert_array_equal(ours[ok], lib[ok])


def test_fp8_requant_worked_example():
    g = read_golden("fp8_requant_worked_example.txt")
    codes = _ints(g["codes"]).astype(np.uint8)
    sinv = _floats(g["scale_inv"])
    q, s, bad = oracle.fp8_block_to_int8_rowwise(codes, sinv)
    np.testing.assert_array_equal(q, _ints(g["q"]).astype(np.int8))
    assert s[0] == float(g["s"][0][0]) and not bad.any()


def test_fp8_requant_half_step_zero_rows_ragged():
    codes, sinv, zero_rows = wl.fp8_block_matrix(300, 1500, seed=1, stream=7, zero_frac=0.01)
    c, si = codes.numpy(), sinv.numpy()
    assert si.shape == (3, 12)
    q, s, bad = oracle.fp8_block_to_int8_rowwise(c, si)
    assert not bad.any()
    zr = zero_rows.numpy()
    assert len(zr) == 3
    assert np.all(s[zr] == 1.0) and not q[zr].any()
    wf = oracle.e4m3_to_f32(c) * np.repeat(np.repeat(si, 128, 0), 128, 1)[:300, :1500]
    _half_step_check(wf.astype(np.float32), q, s)
    # the scale multiplies (a reading that inverted it would be off by ~1e4 here)
    nz = np.setdiff1d(np.arange(300), zr)
    a = np.max(np.abs(wf[nz]), axis=1)
    np.testing.assert_allclose(s[nz], a / 127, rtol=2 ** -23)
    # ragged == padded with zero codes to whole 128 blocks
    cp = np.zeros((384, 1536), dtype=np.uint8)
    cp[:300, :1500] = c
    qp, sp, _ = oracle.fp8_block_to_int8_rowwise(cp, si)
    np.testing.assert_array_equal(qp[:300, :1500], q)
    np.testing.assert_array_equal(sp[:300], s)


@pytest.mark.parametrize("bad_val", [0.0, -1.0, float("inf"), float("nan")])
def test_fp8_requant_illegal_scale(bad_val):
    codes, sinv, _ = wl.fp8_block_matrix(256, 384, seed=2, stream=9, zero_frac=0.0)
    c, si = codes.numpy().copy(), sinv.numpy().copy()
    si[1, 2] = bad_val          # rows 128..255 are affected
    c[5, 7] = 0x7F              # row 5 holds a NaN code
    q, s, bad = oracle.fp8_block_to_int8_rowwise(c, si)
    expect = np.zeros(256, dtype=bool)
    expect[128:] = True
    expect[5] = True
    np.testing.assert_array_equal(bad, expect)
    assert np.all(s[bad] == 1.0) and not q[bad].any()
    q2, s2, _ = oracle.fp8_block_to_int8_rowwise(codes.numpy(), sinv.numpy())
    np.testing.assert_array_equal(q[~bad], q2[~bad])


# ------------------------------------------------------------------ S9

def test_moe_segments_and_combine():
    d = wl.moe_workload(T=48, H=64, E=6, topk=2, inter=32, seed=3)
    xb = wl.bits(d["x"])
    w13 = oracle.bf16_bits_to_f32(wl.bits(d["w13"]))
    w2 = oracle.bf16_bits_to_f32(wl.bits(d["w2"]))
    E = d["E"]
    q13 = np.stack([oracle.quantize_weight_per_channel(w13[e])[0] for e in range(E)])
    s13 = np.stack([oracle.quantize_weight_per_channel(w13[e])[1] for e in range(E)])
    q2 = np.stack([oracle.quantize_weight_per_channel(w2[e])[0] for e in range(E)])
    s2 = np.stack([oracle.quantize_weight_per_channel(w2[e])[1] for e in range(E)])
    ids = d["topk_ids"].numpy()
    tw = d["topk_w"].numpy()
    # force one empty expert
    ids[ids == 4] = 5
    r = oracle.moe_forward(xb, ids, tw, q13, s13, q2, s2)
    seg = r["seg"]
    assert seg[-1] == 48 * 2 and seg[5] - seg[4] == 0
    # each segment equals a plain per-expert linear on that slice
    x = oracle.bf16_bits_to_f32(xb)
    for e in range(E):
        r0, r1 = seg[e], seg[e + 1]
        if r0 == r1:
            continue
        toks = r["tok"][r0:r1]
        assert np.all(ids[toks, r["slot"][r0:r1]] == e)
        lin = oracle.w8a8_linear(xb[toks], q13[e], s13[e])
        np.testing.assert_array_equal(r["h_bits"][r0:r1], lin["y_bits"])
    # combine: an independent per-token loop over the token's own slots
    row_of = {}
    for rr in range(seg[-1]):
        row_of[(int(r["tok"][rr]), int(r["slot"][rr]))] = rr
    for t in range(48):
        acc = np.zeros(64, dtype=np.float32)
        for j in range(2):
            acc = acc + np.float32(tw[t, j]) * oracle.bf16_bits_to_f32(r["out_bits"][row_of[(t, j)]])
        np.testing.assert_array_equal(r["y_bits"][t], oracle.f32_to_bf16_bits(acc))
    # the gated glue is silu(gate) * up: check one value by hand
    gb = oracle.silu_mul_bf16(oracle.f32_to_bf16_bits(np.array([2.0], np.float32)),
                              oracle.f32_to_bf16_bits(np.array([3.0], np.float32)))
    assert abs(oracle.bf16_bits_to_f32(gb)[0] - 3.0 * 2.0 / (1 + math.exp(-2.0))) < 0.02


def test_moe_combine_special_cases():
    """One slot of weight 1 is a gather of the rows (exact); weights 0.5 and 0.25 on two
    slots scale exactly, so the sum is the exact 0.5 a + 0.25 b rounded once to bf16."""
    rng = np.random.default_rng(4)
    out = oracle.f32_to_bf16_bits(rng.standard_normal((7, 40)).astype(np.float32))
    row_of = np.array([[3], [0], [6], [3]])
    yb, y32 = oracle.moe_combine(out, row_of, np.ones((4, 1), np.float32))
    np.testing.assert_array_equal(yb, out[[3, 0, 6, 3]])
    row_of2 = np.array([[1, 5], [2, 2]])
    w2 = np.array([[0.5, 0.25], [0.5, 0.25]], np.float32)
    yb2, y2 = oracle.moe_combine(out, row_of2, w2)
    a = oracle.bf16_bits_to_f32(out).astype(np.float64)
    exact = np.stack([0.5 * a[1] + 0.25 * a[5], 0.75 * a[2]])
    np.testing.assert_array_equal(y2.astype(np.float64), exact)     # no rounding below 2^-24 relative
    yb3, _ = oracle.moe_combine(out, row_of2, w2, rows=[1])
    assert not yb3[0].any() and np.array_equal(yb3[1], yb2[1])


def test_moe_routing_skew():
    d = wl.moe_workload(T=4096, H=8, E=32, topk=4, inter=8, seed=0, with_weights=False)
    ids = d["topk_ids"].numpy()
    counts = np.bincount(ids.reshape(-1), minlength=32)
    assert counts.sum() == 16384
    assert np.all((ids[:, :, None] == ids[:, None, :]).sum(-1) == 1)  # no repeats per token
    assert counts[0] > 10 * counts[-1]                                 # Zipf-like skew


# ---------------------------------------------------------------------------
# requantize_with_max_scale
# ---------------------------------------------------------------------------

def test_max_scale_partition_unchanged_and_bound():
    """The partition that already has the largest scale keeps every code (RN(RN(q*s)/s)
    is within 1e-5 of q); every other code lands within half a step of q * s_p / s_max."""
    rng = np.random.default_rng(11)
    codes = np.arange(-127, 128, dtype=np.int8)
    for _ in range(20):
        sc = np.float32(rng.uniform(1e-4, 1e-1, size=3)).astype(np.float32)
        widths = [2, 3, 4]
        q = np.stack([rng.permutation(codes) for _ in range(sum(widths))])
        out, s_max = oracle.requantize_with_max_scale(q, sc, widths)
        assert s_max == sc.max()
        row_scale = np.repeat(sc, widths)
        big = row_scale == s_max
        np.testing.assert_array_equal(out[big], q[big])
        exact = q.astype(np.float64) * row_scale[:, None].astype(np.float64) / float(s_max)
        assert np.all(np.abs(out - exact) <= 0.5 + 1e-5)


def test_max_scale_power_of_two_ratios_round_half_even():
    """s_p = s_max / 2 and s_max / 4: every step is exact, so w' = round(q / 2) and
    round(q / 4) with ties to even (Python's round), e.g. 3 -> 2, 5 -> 2, -3 -> -2."""
    codes = np.arange(-127, 128, dtype=np.int8)
    q = np.stack([codes, codes, codes])
    sc = np.array([2.0 ** -7, 2.0 ** -8, 2.0 ** -9], dtype=np.float32)
    out, s_max = oracle.requantize_with_max_scale(q, sc, [1, 1, 1])
    assert s_max == np.float32(2.0 ** -7)
    np.testing.assert_array_equal(out[0], codes)
    np.testing.assert_array_equal(out[1], [round(int(c) / 2) for c in codes])
    np.testing.assert_array_equal(out[2], [round(int(c) / 4) for c in codes])
    assert out[1][list(codes).index(3)] == 2 and out[1][list(codes).index(5)] == 2
    assert out[1][list(codes).index(-3)] == -2 and out[2][list(codes).index(6)] == 2


def test_max_scale_boundaries_and_errors():
    """Rows take the scale of the partition they fall in (a zero-width partition in the
    middle owns no row); mismatched widths and bad scales are rejected."""
    q = np.full((8, 4), 100, dtype=np.int8)
    sc = np.array([0.5, 8.0, 1.0], dtype=np.float32)  # the middle (max) partition is empty
    out, s_max = oracle.requantize_with_max_scale(q, sc, [3, 0, 5])
    assert s_max == np.float32(8.0)
    np.testing.assert_array_equal(out[:3], np.full((3, 4), 6, np.int8))    # 100*0.5/8 = 6.25
    np.testing.assert_array_equal(out[3:], np.full((5, 4), 12, np.int8))   # 100/8 = 12.5 -> 12
    with pytest.raises(ValueError):
        oracle.requantize_with_max_scale(q, sc, [3, 0, 4])
    with pytest.raises(ValueError):
        oracle.requantize_with_max_scale(q, np.array([0.5, 0.0, 1.0], np.float32), [3, 0, 5])


# ---------------------------------------------------------------------------
# moe_route
# ---------------------------------------------------------------------------

def test_moe_route_bruteforce_topk_and_ties():
    """Top-k by pairwise comparison: expert e ranks r(e) = #{e' : l[e'] > l[e], or equal
    with e' < e}; ids are the experts of rank 0..k-1 in rank order.  Logits drawn from a
    few values so that ties are frequent."""
    rng = np.random.default_rng(5)
    lg = rng.integers(-3, 3, size=(40, 9)).astype(np.float32) * np.float32(0.75)
    for k in (1, 2, 4, 9):
        ids, w = oracle.moe_route(lg, k)
        for t in range(lg.shape[0]):
            l = lg[t]
            rank = [sum(1 for f in range(9) if l[f] > l[e] or (l[f] == l[e] and f < e)) for e in range(9)]
            want = sorted(range(9), key=lambda e: rank[e])[:k]
            assert list(ids[t]) == want
        if k == 9:
            np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_moe_route_worked_example():
    """logits (0, ln 3, 0, 0): softmax = (1/6, 1/2, 1/6, 1/6); top-2 = expert 1 and, of the
    three equal ones, expert 0, with weights 1/2 and 1/6 (not renormalised to sum 1)."""
    lg = np.array([[0.0, math.log(3.0), 0.0, 0.0], [1.0, 3.0, 3.0, 0.0]], dtype=np.float32)
    ids, w = oracle.moe_route(lg, 2)
    assert list(ids[0]) == [1, 0] and list(ids[1]) == [1, 2]
    np.testing.assert_allclose(w[0], [0.5, 1 / 6], rtol=1e-6)
    e = np.exp(np.array([1.0, 3.0, 3.0, 0.0]) - 3.0)
    np.testing.assert_allclose(w[1], [e[1] / e.sum(), e[2] / e.sum()], rtol=1e-6)
