"""Pins of the oracle's expert math and FP8 quantisers.

The dense layer is checked against scalar pure-Python loops on tiny shapes
and against closed forms; the e4m3 encoder against the OCP FP8 E4M3
definition, exhaustively over its 256 codes, and against torch's own
float8_e4m3fn cast; the block-scaled GEMM against exact integer cases and its
error bound.
"""
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as om

F32 = np.float32


def _sig(z):
    return 1.0 / (1.0 + math.exp(-z))


def _py_layer(x, wr, w13, w2, ws13, ws2, b, G, K, M):
    """The layer with scalar loops only (tiny shapes)."""
    T, d = len(x), len(x[0])
    E = len(wr)
    I = len(w13[0]) // 2
    out = []
    for t in range(T):
        s = []
        for e in range(E):
            u = sum(float(x[t][i]) * float(wr[e][i]) for i in range(d))
            s.append(float(F32(_sig(float(F32(u))))))
        sp = [float(F32(F32(s[e]) + F32(b[e]))) for e in range(E)]
        gsz = E // G
        gs = []
        for g in range(G):
            v = sorted(sp[g * gsz:(g + 1) * gsz], reverse=True)
            gs.append(float(F32(F32(v[0]) + F32(v[1]))))
        groups = sorted(range(G), key=lambda g: (-gs[g], g))[:M]
        cand = [e for e in range(E) if e // gsz in groups]
        chosen = sorted(cand, key=lambda e: (-sp[e], e))[:K]
        tot = sum(s[e] for e in chosen)

        def ffn(w13e, w2e):
            h = []
            for j in range(I):
                a = sum(float(w13e[j][i]) * float(x[t][i]) for i in range(d))
                bb = sum(float(w13e[I + j][i]) * float(x[t][i]) for i in range(d))
                h.append(a * _sig(a) * bb)
            return [sum(float(w2e[o][j]) * h[j] for j in range(I)) for o in range(d)]

        y = [0.0] * d
        for sidx in range(len(ws13)):
            ys = ffn(ws13[sidx], ws2[sidx])
            y = [y[o] + ys[o] for o in range(d)]
        for e in chosen:
            ye = ffn(w13[e], w2[e])
            g = float(F32(s[e] / tot))  # gates are stored as fp32
            y = [y[o] + g * ye[o] for o in range(d)]
        out.append(y)
    return np.array(out)


def test_layer_against_scalar_loops():
    rng = np.random.default_rng(1)
    T, d, E, G, K, M, I, S = 5, 4, 8, 4, 2, 2, 3, 2
    x = rng.standard_normal((T, d)).astype(F32)
    wr = rng.standard_normal((E, d)).astype(F32)
    w13 = rng.standard_normal((E, 2 * I, d)).astype(F32)
    w2 = rng.standard_normal((E, d, I)).astype(F32)
    ws13 = rng.standard_normal((S, 2 * I, d)).astype(F32)
    ws2 = rng.standard_normal((S, d, I)).astype(F32)
    b = rng.uniform(-0.1, 0.1, E).astype(F32)
    got = om.layer_forward(x, wr, w13, w2, ws13, ws2, b, G, K, M)["out"]
    want = _py_layer(x, wr, w13, w2, ws13, ws2, b, G, K, M)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_swiglu_closed_form_scalar():
    for (a, b, c, x) in [(0.5, -2.0, 3.0, 1.5), (-1.0, 0.25, 2.0, -3.0), (0.0, 1.0, 1.0, 4.0)]:
        w13 = np.array([[a], [b]])
        w2 = np.array([[c]])
        got = om.swiglu_ffn(np.array([[x]]), w13, w2)[0, 0]
        z = a * x
        want = c * (z * _sig(z)) * (b * x)
        assert abs(got - want) <= 1e-15 * max(1.0, abs(want))


def test_zero_routed_weights_leave_shared_only():
    rng = np.random.default_rng(4)
    T, d, E, G, K, M, I, S = 16, 8, 8, 4, 2, 2, 4, 1
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((E, d))
    ws13 = rng.standard_normal((S, 2 * I, d))
    ws2 = rng.standard_normal((S, d, I))
    r = om.layer_forward(x, wr, np.zeros((E, 2 * I, d)), np.zeros((E, d, I)), ws13, ws2,
                         np.zeros(E, F32), G, K, M)
    np.testing.assert_array_equal(r["out"], om.shared_output(x, ws13, ws2))


def test_shared_experts_add():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 4))
    ws13 = rng.standard_normal((2, 6, 4))
    ws2 = rng.standard_normal((2, 4, 3))
    both = om.shared_output(x, ws13, ws2)
    sep = om.swiglu_ffn(x, ws13[0], ws2[0]) + om.swiglu_ffn(x, ws13[1], ws2[1])
    np.testing.assert_allclose(both, sep, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# e4m3
# --------------------------------------------------------------------------

def _ocp_e4m3(code):
    """OCP FP8 E4M3: bias 7, subnormals at exponent field 0, S.1111.111 NaN."""
    s = -1.0 if code & 0x80 else 1.0
    ef, mf = (code >> 3) & 0xF, code & 0x7
    if ef == 0xF and mf == 0x7:
        return float("nan")
    if ef == 0:
        return s * (mf / 8.0) * 2.0 ** -6
    return s * (1 + mf / 8.0) * 2.0 ** (ef - 7)


def test_e4m3_all_codes():
    for code in range(256):
        want = _ocp_e4m3(code)
        got = om.e4m3_decode(np.array([code], np.uint8))[0]
        if math.isnan(want):
            assert math.isnan(got)
            continue
        assert got == want
        # every finite code is a fixed point of the rounding and re-encodes to itself
        assert om.e4m3_value(np.array([want], F32))[0] == want
        assert om.e4m3_code(np.array([want], F32))[0] == code
    assert max(_ocp_e4m3(c) for c in range(256) if not math.isnan(_ocp_e4m3(c))) == 448.0


def test_e4m3_rounding_vs_torch_cast():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.uniform(-460, 460, 200000),
        rng.standard_normal(200000) * 0.01,
        rng.standard_normal(100000) * 2.0 ** -8,
        np.linspace(-463.9, 463.9, 100001),
    ]).astype(F32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = om.e4m3_value(v)
    np.testing.assert_array_equal(got, want)
    # codes agree bit for bit too (signed zeros included)
    want_code = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(om.e4m3_code(v), want_code)


def test_e4m3_special_values():
    v = np.array([1e6, -1e6, 464.0, 448.0, 447.0, 2.0 ** -9, 2.0 ** -10,
                  3 * 2.0 ** -10, 2.0 ** -11, np.inf], F32)
    want = [448.0, -448.0, 448.0, 448.0, 448.0, 2.0 ** -9, 0.0, 2.0 ** -8, 0.0, 448.0]
    np.testing.assert_array_equal(om.e4m3_value(v), want)


def test_quantize_rows_scale_and_bound():
    rng = np.random.default_rng(8)
    v = rng.standard_normal((16, 384)).astype(F32)
    v[3, 128:256] = 0.0
    q, sc = om.quantize_rows_1x128(v)
    assert sc.shape == (16, 3) and sc[3, 1] == 1.0
    for r in range(16):
        for b in range(3):
            blk = v[r, b * 128:(b + 1) * 128]
            amax = np.abs(blk).max()
            if amax > 0:
                assert sc[r, b] == F32(F32(amax) / F32(448.0))
    deq = q * np.repeat(sc.astype(np.float64), 128, axis=1)
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normals, plus the
    # absolute subnormal step (2^-10 * scale)
    err = np.abs(deq - v)
    bound = np.abs(v) * 2.0 ** -4 + np.repeat(sc.astype(np.float64), 128, axis=1) * 2.0 ** -10
    assert np.all(err <= bound * 1.0001)


def test_quantize_power_of_two_invariance():
    rng = np.random.default_rng(9)
    v = rng.standard_normal((4, 256)).astype(F32)
    q1, s1 = om.quantize_rows_1x128(v)
    q2, s2 = om.quantize_rows_1x128((v * F32(8.0)).astype(F32))
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s2, s1 * F32(8.0))


def test_fp8_gemm_exact_integers():
    rng = np.random.default_rng(10)
    # small integers are exact in e4m3; with unit scales the blocked GEMM is
    # an ordinary integer matmul
    a = rng.integers(-8, 9, (6, 256)).astype(np.float64)
    w = rng.integers(-8, 9, (130, 256)).astype(np.float64)
    got = om.fp8_gemm(a, np.ones((6, 2), F32), w, np.ones((2, 2), F32))
    np.testing.assert_array_equal(got, a @ w.T)
    # block scales apply per (row, K block) and per (128-row block, K block)
    sa = np.array([[2.0, 0.5]] * 6, F32)
    sw = np.array([[4.0, 1.0], [0.25, 8.0]], F32)
    got = om.fp8_gemm(a, sa, w, sw)
    want = np.zeros((6, 130))
    for i in range(6):
        for j in range(130):
            for k in range(256):
                want[i, j] += a[i, k] * w[j, k] * sa[i, k // 128] * sw[j // 128, k // 128]
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-12)


def test_fp8_gemm_error_bound():
    rng = np.random.default_rng(12)
    a = rng.standard_normal((32, 512)).astype(F32)
    w = (rng.standard_normal((256, 512)) * 0.006).astype(F32)
    qa, sa = om.quantize_rows_1x128(a)
    qw, sw = om.quantize_blocks_128x128(w)
    got = om.fp8_gemm(qa, sa, qw, sw)
    exact = a.astype(np.float64) @ w.astype(np.float64).T
    # each operand carries <= 2^-4 relative rounding error: the product error
    # is bounded by sum |a||w| * (2 * 2^-4 + 2^-8) plus subnormal terms
    bound = np.abs(a).astype(np.float64) @ np.abs(w).astype(np.float64).T * (2 * 2.0 ** -4 + 2.0 ** -8)
    assert np.all(np.abs(got - exact) <= bound + 1e-6)
    rel = np.abs(got - exact).max() / np.abs(exact).max()
    assert rel < 0.05


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (130, 200)])
def test_quantize_blocks_layout(shape):
    rng = np.random.default_rng(13)
    w = rng.standard_normal(shape).astype(F32)
    q, sc = om.quantize_blocks_128x128(w)
    nbn, nbk = (shape[0] + 127) // 128, (shape[1] + 127) // 128
    assert sc.shape == (nbn, nbk)
    for i in range(nbn):
        for j in range(nbk):
            blk = w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            assert sc[i, j] == F32(F32(np.abs(blk).max()) / F32(448.0))
            np.testing.assert_array_equal(
                q[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128],
                om.e4m3_value((blk / sc[i, j]).astype(F32)))


def test_fp8_layer_without_shared_experts():
    """S = 0: the FP8 layer is the gate-weighted routed sum alone."""
    rng = np.random.default_rng(14)
    T, d, I = 4, 128, 128
    x = rng.standard_normal((T, d)).astype(F32)
    w13 = (rng.standard_normal((2, 2 * I, d)) * 0.05).astype(F32)
    w2 = (rng.standard_normal((2, d, I)) * 0.05).astype(F32)
    idx = np.array([[0, 1]] * T, np.int32)
    gate = np.full((T, 2), 0.5, F32)
    wq = {e: om.quantize_expert_weights(w13[e], w2[e]) for e in range(2)}
    out = om.layer_forward_fp8(x, idx, gate, wq, [])
    qx, sx = om.quantize_rows_1x128(x)
    want = sum(0.5 * om.swiglu_ffn_fp8(qx, sx, *wq[e]) for e in range(2))
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# power-of-two (UE8M0) scale rule
# --------------------------------------------------------------------------

def _powers_448():
    return (448.0 * 2.0 ** np.arange(-20, 21)).astype(F32)


def test_ue8m0_scale_brute_force():
    """The scale is the smallest 2^e (e >= -127) with 448 * 2^e >= amax,
    found here by walking the exponents (exact float64 comparisons)."""
    rng = np.random.default_rng(21)
    p = _powers_448()
    amax = np.concatenate([p, np.nextafter(p, F32(np.inf)), np.nextafter(p, F32(0)),
                           (rng.uniform(0, 1, 1500) * 10.0 ** rng.integers(-6, 7, 1500)).astype(F32),
                           np.array([0.0, 1e-40, 3e38], F32)]).astype(F32)
    sc = om.tile_scale_ue8m0(amax)
    assert sc.dtype == F32
    for a, s in zip(amax.tolist(), sc.tolist()):
        if a == 0.0:
            assert s == 1.0
            continue
        e = next(e for e in range(-127, 128) if 448.0 * 2.0 ** e >= a)
        assert s == 2.0 ** e, (a, s, e)


def _check_pow2_tiles(v_tiles, sc, q_tiles):
    """Every tile: scale a power of two, amax / scale in (224, 448] (no
    saturation, no smaller power would do), codes = torch's e4m3 cast of the
    exact quotient."""
    import torch
    for blk, s, q in zip(v_tiles, sc, q_tiles):
        amax = float(np.abs(blk).max())
        if amax == 0.0:
            assert s == 1.0 and not np.any(q)
            continue
        m, _ = np.frexp(float(s))
        assert m == 0.5
        assert 224.0 < amax / float(s) <= 448.0
        quot = (blk / s).astype(F32)
        assert np.array_equal(quot.astype(np.float64) * float(s), blk.astype(np.float64))  # exact division
        want = torch.from_numpy(quot.copy()).to(torch.float8_e4m3fn).float().numpy()
        np.testing.assert_array_equal(q, want.astype(np.float64))


def test_ue8m0_rows():
    rng = np.random.default_rng(22)
    v = (rng.standard_normal((16, 384)) * 10.0 ** rng.uniform(-3, 3, (16, 1))).astype(F32)
    v[5, 256:] = 0.0
    q, sc = om.quantize_rows_1x128(v, ue8m0=True)
    assert sc.shape == (16, 3)
    tiles = [v[r, b * 128:(b + 1) * 128] for r in range(16) for b in range(3)]
    qt = [q[r, b * 128:(b + 1) * 128] for r in range(16) for b in range(3)]
    _check_pow2_tiles(tiles, [sc[r, b] for r in range(16) for b in range(3)], qt)


def test_ue8m0_blocks():
    rng = np.random.default_rng(23)
    w = (rng.standard_normal((130, 200)) * 0.02).astype(F32)
    w[:128, 128:] = 0.0
    q, sc = om.quantize_blocks_128x128(w, ue8m0=True)
    assert sc.shape == (2, 2)
    tiles, scs, qt = [], [], []
    for i in range(2):
        for j in range(2):
            tiles.append(w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128])
            qt.append(q[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128])
            scs.append(sc[i, j])
    _check_pow2_tiles(tiles, scs, qt)


def test_ue8m0_coincides_with_fp32_rule_on_exact_powers():
    """When every tile's amax is 448 * 2^k, both scale rules give 2^k, so the
    two modes quantise identically."""
    rng = np.random.default_rng(24)
    v = rng.uniform(-1, 1, (8, 256)).astype(F32)
    for r in range(8):
        for b in range(2):
            v[r, b * 128:(b + 1) * 128] *= F32(2.0 ** (r - b - 3))
            v[r, b * 128 + (r * 7 + b) % 128] = F32(448.0 * 2.0 ** (r - b - 3)) * (1 if r % 2 else -1)
    q1, s1 = om.quantize_rows_1x128(v)
    q2, s2 = om.quantize_rows_1x128(v, ue8m0=True)
    np.testing.assert_array_equal(s1, s2)
    np.testing.assert_array_equal(q1, q2)


def test_ue8m0_power_of_two_invariance():
    rng = np.random.default_rng(25)
    v = rng.standard_normal((4, 256)).astype(F32)
    q1, s1 = om.quantize_rows_1x128(v, ue8m0=True)
    q2, s2 = om.quantize_rows_1x128((v * F32(2.0 ** -5)).astype(F32), ue8m0=True)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s2, s1 * F32(2.0 ** -5))


def test_ue8m0_gemm_error_bound():
    rng = np.random.default_rng(26)
    a = rng.standard_normal((32, 512)).astype(F32)
    w = (rng.standard_normal((256, 512)) * 0.006).astype(F32)
    qa, sa = om.quantize_rows_1x128(a, ue8m0=True)
    qw, sw = om.quantize_blocks_128x128(w, ue8m0=True)
    got = om.fp8_gemm(qa, sa, qw, sw)
    exact = a.astype(np.float64) @ w.astype(np.float64).T
    # quotients lie in (224, 448] at the tile maximum, so the same 2^-4
    # relative rounding bound holds, plus the subnormal step of each tile
    bound = np.abs(a).astype(np.float64) @ np.abs(w).astype(np.float64).T * (2 * 2.0 ** -4 + 2.0 ** -8)
    assert np.all(np.abs(got - exact) <= bound + 1e-6)
    assert np.abs(got - exact).max() / np.abs(exact).max() < 0.05


def test_ue8m0_layer_differs_only_by_scale_rule():
    """The UE8M0 FP8 layer stays within the quantisation bound of the exact
    layer, and its h scales really are the power-of-two ones."""
    rng = np.random.default_rng(27)
    T, d, I = 6, 256, 128
    x = rng.standard_normal((T, d)).astype(F32)
    w13 = (rng.standard_normal((2, 2 * I, d)) * 0.05).astype(F32)
    w2 = (rng.standard_normal((2, d, I)) * 0.05).astype(F32)
    idx = np.array([[0, 1]] * T, np.int32)
    gate = np.full((T, 2), 0.5, F32)
    wq = {e: om.quantize_expert_weights(w13[e], w2[e], ue8m0=True) for e in range(2)}
    for e in range(2):
        for s in (wq[e][1], wq[e][3]):
            assert np.all(np.frexp(s.astype(np.float64))[0] == 0.5)
    out = om.layer_forward_fp8(x, idx, gate, wq, [], ue8m0=True)
    exact = sum(0.5 * om.swiglu_ffn(x.astype(np.float64), w13[e].astype(np.float64),
                                    w2[e].astype(np.float64)) for e in range(2))
    rel = np.abs(out - exact).max() / np.abs(exact).max()
    assert rel < 0.08
    out32 = om.layer_forward_fp8(x, idx, gate,
                                 {e: om.quantize_expert_weights(w13[e], w2[e]) for e in range(2)}, [])
    assert not np.array_equal(out, out32)
