"""Pins of the C++ CPU oracle (oracle/moe_oracle.cpp).

The C++ oracle is checked against what the pages and the mathematics fix --
the hand-worked examples under tests/golden/, brute-force enumeration of the
group-limited selection, closed forms, the OCP E4M3 definition and torch's
e4m3 cast -- and against the independent NumPy oracle: routing, counts,
permutation and bias trajectories bit for bit, dense outputs to 1e-12
("DeepSeek-V3技术报告" digest, mpbf.cn, sections 2.2 and 3.1;
"DeepSeek-V3架构深度解析", blog.resmic.cn, 核心架构二).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from mixture_experts_layer_100_b300 import synth
from oracle import cpp
from oracle import moe_oracle as om
from tests.test_oracle_routing import _brute_route_token

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# hand-worked examples
# --------------------------------------------------------------------------

def test_two_token_example():
    g = _golden("two_token_example.json")
    s = np.array(g["scores"], F32)
    b = np.array(g["bias"], F32)
    np.testing.assert_array_equal(cpp.group_scores(s, b, g["G"], g["group_topk"]),
                                  np.array(g["group_scores"], F32))
    idx, gate = cpp.select_experts(s, b, g["G"], g["K"], g["M"], g["group_topk"])
    np.testing.assert_array_equal(idx, np.array(g["topk_idx"]))
    want_gate = np.array([[n / d for n, d in row] for row in g["topk_gate_num_den"]])
    np.testing.assert_array_equal(gate, want_gate.astype(F32))
    counts = cpp.expert_counts(idx, g["E"])
    np.testing.assert_array_equal(counts, g["counts"])
    np.testing.assert_array_equal(cpp.exclusive_offsets(counts), g["offsets"])
    st, sp = cpp.permutation(idx, g["E"])
    np.testing.assert_array_equal(st, g["sorted_tok"])
    np.testing.assert_array_equal(sp, g["slot_pos"])
    b1 = cpp.bias_update(counts, b, g["gamma"], g["T"], g["K"])
    want = np.array([F32(b[e] + np.sign(d) * F32(g["gamma"])) for e, d in enumerate(g["bias_delta_sign"])], F32)
    np.testing.assert_array_equal(b1, want)


def test_sequence_balance_hand_example():
    g = _golden("seq_balance_example.json")
    loss, f, P = cpp.sequence_balance(np.array(g["scores"], F32), np.array(g["topk_idx"], np.int32),
                                      g["seq_len"], g["alpha"])
    np.testing.assert_allclose(f, np.array(g["f"], np.float64), rtol=0, atol=1e-15)
    np.testing.assert_allclose(P, [[n / d for n, d in row] for row in g["P_num_den"]], rtol=1e-15)
    np.testing.assert_allclose(loss, [n / d for n, d in g["loss_num_den"]], rtol=1e-15)


# --------------------------------------------------------------------------
# routing: brute force, special cases, and the NumPy oracle bit for bit
# --------------------------------------------------------------------------

@pytest.mark.parametrize("E,G,K,M,gk", [(8, 4, 2, 2, 2), (12, 3, 3, 2, 2), (16, 4, 4, 2, 2), (16, 8, 3, 3, 2),
                                        (12, 4, 2, 1, 1), (16, 4, 5, 3, 3), (16, 4, 4, 2, 4), (12, 2, 3, 1, 6)])
@pytest.mark.parametrize("kind", ["uniform", "dyadic"])
def test_brute_force_selection(E, G, K, M, gk, kind):
    rng = np.random.default_rng(E * 1000 + K * 10 + M + (7 if kind == "dyadic" else 0))
    T = 24
    if kind == "uniform":
        s = rng.uniform(0.05, 0.95, (T, E)).astype(F32)
        b = rng.uniform(-0.05, 0.05, E).astype(F32)
    else:
        s = (rng.integers(1, 8, (T, E)) / 8.0).astype(F32)
        b = (rng.integers(-2, 3, E) / 16.0).astype(F32)
    idx, gate = cpp.select_experts(s, b, G, K, M, gk)
    sp = (s + b[None, :]).astype(F32)
    for t in range(T):
        want = _brute_route_token(sp[t], G, K, M, gk)
        assert list(idx[t]) == want, (t, list(idx[t]), want)
        chosen = s[t, want].astype(np.float64)
        np.testing.assert_array_equal(gate[t], (chosen / chosen.sum()).astype(F32))


def test_all_groups_allowed_is_plain_topk():
    rng = np.random.default_rng(3)
    T, E, G, K = 64, 32, 4, 6
    s = (rng.integers(1, 16, (T, E)) / 16.0).astype(F32)
    idx, _ = cpp.select_experts(s, np.zeros(E, F32), G, K, G)
    for t in range(T):
        assert list(idx[t]) == sorted(range(E), key=lambda e: (-float(s[t, e]), e))[:K]


def test_zero_router_everything_ties():
    T, d, E, G, K, M = 8, 16, 16, 4, 4, 2
    x = np.random.default_rng(0).standard_normal((T, d)).astype(F32)
    s = cpp.router_scores(x, np.zeros((E, d), F32))
    assert np.all(s == F32(0.5))
    idx, gate = cpp.select_experts(s, np.zeros(E, F32), G, K, M)
    assert np.all(idx == np.arange(4)[None, :]) and np.all(gate == F32(0.25))


def test_router_scores_closed_form():
    x = np.array([[2.0, 0.0], [0.0, -1.0], [0.0, 0.0]], F32)
    w = np.array([[0.5, 3.0], [0.25, -2.0]], F32)
    s = cpp.router_scores(x, w)
    u = [[1.0, 0.5], [-3.0, 2.0], [0.0, 0.0]]
    for t in range(3):
        for e in range(2):
            assert s[t, e] == F32(1.0 / (1.0 + math.exp(-u[t][e])))


@pytest.mark.parametrize("T,E,G,K,M,gk", [(512, 16, 4, 4, 2, 2), (512, 64, 8, 6, 3, 2), (1024, 256, 8, 8, 4, 2),
                                          (300, 256, 8, 8, 4, 32), (200, 64, 4, 16, 2, 2), (90, 64, 2, 32, 1, 2),
                                          (257, 128, 8, 6, 3, 3)])
@pytest.mark.parametrize("kind", ["uniform", "dyadic", "const", "skewed"])
def test_routing_matches_numpy_oracle(T, E, G, K, M, gk, kind):
    s = synth.make_scores(T, E, seed=T + E + K, kind=kind).numpy()
    b = (np.random.default_rng(E).integers(-4, 5, E) / 256.0).astype(F32)
    idx_c, gate_c = cpp.select_experts(s, b, G, K, M, gk)
    idx_n, gate_n = om.select_experts(s, b, G, K, M, gk)
    np.testing.assert_array_equal(idx_c, idx_n)
    np.testing.assert_allclose(gate_c, gate_n, rtol=2 ** -23, atol=0)
    np.testing.assert_array_equal(cpp.group_scores(s, b, G, gk), om.group_scores(om.biased_scores(s, b), G, gk))


def test_selection_invariants():
    rng = np.random.default_rng(7)
    T, E, G, K, M = 512, 64, 8, 6, 3
    s = rng.uniform(0, 1, (T, E)).astype(F32)
    b = rng.uniform(-0.05, 0.05, E).astype(F32)
    idx, gate = cpp.select_experts(s, b, G, K, M)
    sp = (s + b[None, :]).astype(F32)
    gsz = E // G
    for t in range(T):
        assert len(set(idx[t])) == K
        groups = set(int(e) // gsz for e in idx[t])
        assert len(groups) <= M
        w = int(idx[t, K - 1])
        for g in groups:
            for e in range(g * gsz, (g + 1) * gsz):
                if e not in idx[t]:
                    assert sp[t, e] < sp[t, w] or (sp[t, e] == sp[t, w] and e > w)
    np.testing.assert_allclose(gate.astype(np.float64).sum(1), 1.0, atol=1e-6)
    assert cpp.expert_counts(idx, E).sum() == T * K


def test_router_scores_match_numpy_oracle():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((200, 384)).astype(F32)
    w = (rng.standard_normal((64, 384)) * 0.05).astype(F32)
    sc, sn = cpp.router_scores(x, w), om.router_scores(x, w)
    # the two exp implementations may round a last float64 bit differently
    assert np.abs(sc.view(np.int32) - sn.view(np.int32)).max() <= 1
    assert (sc == sn).mean() > 0.999


# --------------------------------------------------------------------------
# counts, permutation, bias update
# --------------------------------------------------------------------------

def test_permutation_against_sort_and_numpy():
    rng = np.random.default_rng(5)
    T, E, K = 300, 16, 4
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    counts = cpp.expert_counts(idx, E)
    off = cpp.exclusive_offsets(counts)
    st, sp = cpp.permutation(idx, E)
    pairs = sorted((int(idx[t, k]), t, k) for t in range(T) for k in range(K))
    for p, (e, t, k) in enumerate(pairs):
        assert st[p] == t and sp[t, k] == p and off[e] <= p < off[e + 1]
    st_n, sp_n = om.permutation(idx, E)
    np.testing.assert_array_equal(st, st_n)
    np.testing.assert_array_equal(sp, sp_n)
    np.testing.assert_array_equal(counts, om.expert_counts(idx, E))


def test_bias_update_moves_toward_balance():
    counts = np.array([0, 1, 2, 3, 4, 5, 6, 7], np.int32)  # T*K/E = 28/8 = 3.5
    b = np.zeros(8, F32)
    b1 = cpp.bias_update(counts, b, 1e-3, 7, 4)
    g = F32(1e-3)
    np.testing.assert_array_equal(b1, np.array([g, g, g, g, -g, -g, -g, -g], F32))
    even = np.full(8, 4, np.int32)  # T*K/E = 4 exactly: unchanged
    np.testing.assert_array_equal(cpp.bias_update(even, b1, 1e-3, 8, 4), b1)
    assert cpp.load_max_over_mean(counts, 7, 4) == float(F32(7 / 3.5))


@pytest.mark.parametrize("T,E,G,K,M", [(256, 16, 4, 4, 2), (2048, 256, 8, 8, 4)])
def test_bias_balancing_loop_matches_numpy_oracle(T, E, G, K, M):
    s = synth.make_scores(T, E, seed=42, kind="skewed").numpy()
    b0 = np.zeros(E, F32)
    bc, ic, lc = cpp.bias_balancing_loop(s, b0, 12, 1e-3, G, K, M)
    bn, in_, ln = om.bias_balancing_loop(s, b0, 12, 1e-3, G, K, M)
    for k in range(12):
        np.testing.assert_array_equal(ic[k], in_[k])
        np.testing.assert_array_equal(bc[k], bn[k])
        assert lc[k] == F32(ln[k])
    assert lc[-1] < lc[0]


# --------------------------------------------------------------------------
# dense layer
# --------------------------------------------------------------------------

def _layer_inputs(p):
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    b = synth.make_bias(p)
    return w, x.float().numpy(), b.numpy()


@pytest.mark.parametrize("over", [{}, dict(S=0), dict(S=2), dict(group_topk=4)])
def test_layer_matches_numpy_oracle(over):
    p = synth.PRESETS["tiny_t256_d512_e16_fp32"].replace(**over)
    w, x, b = _layer_inputs(p)
    a = [w.w_router.float().numpy(), w.w13.float().numpy(), w.w2.float().numpy(), w.ws13.float().numpy(),
         w.ws2.float().numpy()]
    rc = cpp.layer_forward(x, *a, b, p.G, p.K, p.M, p.group_topk)
    rn = om.layer_forward(x.astype(np.float64), *[v.astype(np.float64) for v in a], b, p.G, p.K, p.M, p.group_topk,
                          scores=rc["scores"])
    np.testing.assert_array_equal(rc["topk_idx"], rn["topk_idx"])
    err = np.abs(rc["out"] - rn["out"]).max() / np.abs(rn["out"]).max()
    assert err <= 1e-12, err


def test_swiglu_closed_form_scalar():
    # one expert, d = I = 1: y = c * silu(a x) * (b x)
    a_, b_, c_, x_ = 0.75, -1.5, 2.0, 0.5
    y = cpp.swiglu_ffn(np.array([[x_]], F32), np.array([[a_], [b_]], F32), np.array([[c_]], F32))
    z = a_ * x_
    assert y[0, 0] == c_ * (z / (1.0 + math.exp(-z))) * (b_ * x_)


def test_expert_accumulate_is_the_layer():
    """Streaming the experts one at a time (the form the full-size parity
    tests use) gives the same bits as the whole-layer call."""
    p = synth.PRESETS["tiny_t256_d512_e16_fp32"].replace(T=64, S=2)
    w, x, b = _layer_inputs(p)
    full = cpp.layer_forward(x, w.w_router.numpy(), w.w13.numpy(), w.w2.numpy(), w.ws13.numpy(), w.ws2.numpy(), b,
                             p.G, p.K, p.M)
    acc = np.zeros_like(full["out"])
    for s in range(p.S):
        cpp.expert_accumulate(x, np.arange(p.T), w.ws13[s].numpy(), w.ws2[s].numpy(), None, acc)
    idx, gate = full["topk_idx"], full["topk_gate"]
    for e in np.unique(idx):
        rows, slots = np.nonzero(idx == e)
        cpp.expert_accumulate(x, rows, w.w13[e].numpy(), w.w2[e].numpy(), gate[rows, slots], acc)
    # the whole-layer call adds the routed terms slot by slot, the streamed
    # form expert by expert: equal up to the order of a few double adds
    np.testing.assert_allclose(acc, full["out"], rtol=1e-13, atol=1e-15)


def test_zero_routed_weights_leave_shared_only():
    p = synth.PRESETS["tiny_t256_d512_e16_fp32"].replace(T=32)
    w = synth.make_weights(p, zero_routed=True)
    x = synth.make_x(p, w.w_router).numpy()
    r = cpp.layer_forward(x, w.w_router.numpy(), w.w13.numpy(), w.w2.numpy(), w.ws13.numpy(), w.ws2.numpy(),
                          np.zeros(p.E, F32), p.G, p.K, p.M)
    shared = cpp.swiglu_ffn(x, w.ws13[0].numpy(), w.ws2[0].numpy())
    np.testing.assert_array_equal(r["out"], shared)


# --------------------------------------------------------------------------
# e4m3 and the FP8 path
# --------------------------------------------------------------------------

def _ocp_e4m3(code):
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
        got = cpp.e4m3_decode(code)
        if math.isnan(want):
            assert math.isnan(got)
            continue
        assert got == want
        assert cpp.e4m3_value(want) == want
        assert cpp.e4m3_code(want) == code


def test_e4m3_rounding_vs_torch_cast():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(-460, 460, 20000), rng.standard_normal(20000) * 0.01,
                        rng.standard_normal(10000) * 2.0 ** -8, np.linspace(-463.9, 463.9, 10001)]).astype(F32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn)
    got_v = np.array([cpp.e4m3_value(a) for a in v.tolist()])
    np.testing.assert_array_equal(got_v, want.float().numpy().astype(np.float64))
    got_c = np.array([cpp.e4m3_code(a) for a in v.tolist()], np.uint8)
    np.testing.assert_array_equal(got_c, want.view(torch.uint8).numpy())


def test_e4m3_special_values():
    v = [1e6, -1e6, 464.0, 448.0, 447.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -11]
    want = [448.0, -448.0, 448.0, 448.0, 448.0, 2.0 ** -9, 0.0, 2.0 ** -8, 0.0]
    assert [cpp.e4m3_value(a) for a in v] == want


def test_tile_scales_against_definitions():
    rng = np.random.default_rng(21)
    p = (448.0 * 2.0 ** np.arange(-20, 21)).astype(F32)
    amax = np.concatenate([p, np.nextafter(p, F32(np.inf)), np.nextafter(p, F32(0)),
                           (rng.uniform(0, 1, 500) * 10.0 ** rng.integers(-6, 7, 500)).astype(F32),
                           np.array([0.0, 1e-40, 3e38], F32)]).astype(F32)
    for a in amax.tolist():
        # fp32 rule: one IEEE division; power-of-two rule: the exponent walk
        assert cpp.tile_scale(a, False) == (1.0 if a == 0 else float(F32(a) / F32(448.0)))
        e = next(e for e in range(-127, 128) if 448.0 * 2.0 ** e >= a) if a > 0 else None
        assert cpp.tile_scale(a, True) == (1.0 if a == 0 else 2.0 ** e)


@pytest.mark.parametrize("ue8m0", [False, True])
def test_quantizers_match_numpy_oracle(ue8m0):
    rng = np.random.default_rng(9)
    v = (rng.standard_normal((40, 300)) * 10.0 ** rng.uniform(-3, 3, (40, 1))).astype(F32)
    v[3, 128:256] = 0.0
    qc, sc = cpp.quantize_rows_1x128(v, ue8m0)
    qn, sn = om.quantize_rows_1x128(v, ue8m0)
    np.testing.assert_array_equal(qc, qn)
    np.testing.assert_array_equal(sc, sn)
    w = (rng.standard_normal((300, 260)) * 0.01).astype(F32)
    qc, sc = cpp.quantize_blocks_128x128(w, ue8m0)
    qn, sn = om.quantize_blocks_128x128(w, ue8m0)
    np.testing.assert_array_equal(qc, qn)
    np.testing.assert_array_equal(sc, sn)


def test_fp8_gemm_exact_integers_and_numpy():
    rng = np.random.default_rng(2)
    qa = rng.integers(-8, 9, (5, 256)).astype(np.float64)
    qw = rng.integers(-8, 9, (130, 256)).astype(np.float64)
    sa = np.full((5, 2), 0.5, F32)
    sw = np.full((2, 2), 4.0, F32)
    np.testing.assert_array_equal(cpp.fp8_gemm(qa, sa, qw, sw), 2.0 * (qa @ qw.T))
    sa = rng.uniform(0.1, 2, (5, 2)).astype(F32)
    sw = rng.uniform(0.1, 2, (2, 2)).astype(F32)
    np.testing.assert_allclose(cpp.fp8_gemm(qa, sa, qw, sw), om.fp8_gemm(qa, sa, qw, sw), rtol=1e-13)


@pytest.mark.parametrize("ue8m0", [False, True])
def test_fp8_layer_matches_numpy_oracle(ue8m0):
    p = synth.PRESETS["tiny_t256_d512_e16_fp32"].replace(T=48, S=2, dtype="bf16")
    w, x, b = _layer_inputs(p)
    a = [w.w_router.float().numpy(), w.w13.float().numpy(), w.w2.float().numpy(), w.ws13.float().numpy(),
         w.ws2.float().numpy()]
    rc = cpp.layer_forward_fp8(x, *a, b, p.G, p.K, p.M, ue8m0=ue8m0)
    rn = om.layer_forward_fp8_full(x.astype(np.float64), *a, b, p.G, p.K, p.M, ue8m0=ue8m0)
    np.testing.assert_array_equal(rc["topk_idx"], rn["topk_idx"])
    err = np.abs(rc["out"] - rn["out"]).max() / np.abs(rn["out"]).max()
    assert err <= 1e-12, err


def test_fp8_accumulate_is_the_layer():
    p = synth.PRESETS["tiny_t256_d512_e16_fp32"].replace(T=20, S=1, dtype="bf16")
    w, x, b = _layer_inputs(p)
    full = cpp.layer_forward_fp8(x, w.w_router.float().numpy(), w.w13.float().numpy(), w.w2.float().numpy(),
                                 w.ws13.float().numpy(), w.ws2.float().numpy(), b, p.G, p.K, p.M, ue8m0=True)
    acc = np.zeros_like(full["out"])
    cpp.expert_accumulate(x, np.arange(p.T), w.ws13[0].float().numpy(), w.ws2[0].float().numpy(), None, acc,
                          fp8=True, ue8m0=True)
    for e in np.unique(full["topk_idx"]):
        rows, slots = np.nonzero(full["topk_idx"] == e)
        cpp.expert_accumulate(x, rows, w.w13[e].float().numpy(), w.w2[e].float().numpy(),
                              full["topk_gate"][rows, slots], acc, fp8=True, ue8m0=True)
    np.testing.assert_allclose(acc, full["out"], rtol=1e-13, atol=1e-15)


def test_sequence_balance_matches_numpy_oracle():
    s = synth.make_scores(1000, 64, seed=5, kind="skewed").numpy()
    idx, _ = om.select_experts(s, np.zeros(64, F32), 8, 6, 3)
    lc, fc, pc = cpp.sequence_balance(s, idx, 300, 0.01)
    ln, fn, pn = om.sequence_balance(s, idx, 300, 0.01)
    np.testing.assert_allclose(lc, ln, rtol=1e-13)
    np.testing.assert_allclose(fc, fn, rtol=1e-15)
    np.testing.assert_allclose(pc, pn, rtol=1e-13)


def test_thread_count_does_not_change_results():
    p = synth.PRESETS["tiny_t256_d512_e16_fp32"].replace(T=40)
    w, x, b = _layer_inputs(p)
    a = [w.w_router.numpy(), w.w13.numpy(), w.w2.numpy(), w.ws13.numpy(), w.ws2.numpy()]
    r1 = cpp.layer_forward(x, *a, b, p.G, p.K, p.M, threads=1)
    r7 = cpp.layer_forward(x, *a, b, p.G, p.K, p.M, threads=7)
    for k in ("scores", "topk_idx", "topk_gate", "out"):
        np.testing.assert_array_equal(r1[k], r7[k])
