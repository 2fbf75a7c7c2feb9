"""Pins of the oracle's routing, load count, permutation and bias update.

Each check ties the oracle to something other than itself: a hand-worked
example, a brute-force enumeration of the selection rule on tiny inputs, the
plain top-K it must reduce to, or an invariant the method guarantees
("DeepSeek-V3技术报告" digest, mpbf.cn, section 2.2).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# hand-worked example
# --------------------------------------------------------------------------

def test_two_token_example():
    g = _golden("two_token_example.json")
    s = np.array(g["scores"], F32)
    b = np.array(g["bias"], F32)
    sp = om.biased_scores(s, b)
    np.testing.assert_array_equal(om.group_scores(sp, g["G"], g["group_topk"]),
                                  np.array(g["group_scores"], F32))
    idx, gate = om.select_experts(s, b, g["G"], g["K"], g["M"], g["group_topk"])
    np.testing.assert_array_equal(idx, np.array(g["topk_idx"]))
    want_gate = np.array([[n / d for n, d in row] for row in g["topk_gate_num_den"]])
    np.testing.assert_array_equal(gate, want_gate.astype(F32))
    counts = om.expert_counts(idx, g["E"])
    np.testing.assert_array_equal(counts, g["counts"])
    np.testing.assert_array_equal(om.exclusive_offsets(counts), g["offsets"])
    st, sp_ = om.permutation(idx, g["E"])
    np.testing.assert_array_equal(st, g["sorted_tok"])
    np.testing.assert_array_equal(sp_, g["slot_pos"])
    b1 = om.bias_update(counts, b, g["gamma"], g["T"], g["K"])
    want = np.array([F32(b[e] + np.sign(d) * F32(g["gamma"])) for e, d in
                     enumerate(g["bias_delta_sign"])], F32)
    np.testing.assert_array_equal(b1, want)


# --------------------------------------------------------------------------
# brute force
# --------------------------------------------------------------------------

def _brute_route_token(sp, G, K, M, gk):
    """The selection rule by exhaustive enumeration (pure Python)."""
    E = len(sp)
    gsz = E // G
    # group score: best sum over all gk-subsets of the group, added largest first
    gscore = []
    for g in range(G):
        best = None
        for sub in itertools.combinations(range(g * gsz, (g + 1) * gsz), gk):
            vals = sorted((float(sp[e]) for e in sub), reverse=True)
            acc = F32(vals[0])
            for v in vals[1:]:
                acc = F32(acc + F32(v))
            best = acc if best is None or acc > best else best
        gscore.append(best)
    # group subset: the M-subset whose (score desc, index asc) list is smallest
    # under the order (-score, index)
    best_groups = min(itertools.combinations(range(G), M),
                      key=lambda c: sorted((-float(gscore[g]), g) for g in c))
    cand = [e for g in best_groups for e in range(g * gsz, (g + 1) * gsz)]
    best_experts = min(itertools.combinations(cand, K),
                       key=lambda c: sorted((-float(sp[e]), e) for e in c))
    return sorted(best_experts, key=lambda e: (-float(sp[e]), e))


@pytest.mark.parametrize("E,G,K,M,gk", [(8, 4, 2, 2, 2), (12, 3, 3, 2, 2),
                                        (16, 4, 4, 2, 2), (16, 8, 3, 3, 2),
                                        (12, 4, 2, 1, 1), (16, 4, 5, 3, 3),
                                        (16, 4, 4, 2, 4), (12, 2, 3, 1, 6)])  # full group sums
@pytest.mark.parametrize("kind", ["uniform", "dyadic"])
def test_brute_force_selection(E, G, K, M, gk, kind):
    rng = np.random.default_rng(E * 100 + K * 10 + M)
    T = 24
    if kind == "uniform":
        s = rng.uniform(0.05, 0.95, (T, E)).astype(F32)
        b = rng.uniform(-0.05, 0.05, E).astype(F32)
    else:  # many exact ties
        s = (rng.integers(1, 8, (T, E)) / 8.0).astype(F32)
        b = (rng.integers(-2, 3, E) / 16.0).astype(F32)
    idx, gate = om.select_experts(s, b, G, K, M, gk)
    sp = om.biased_scores(s, b)
    for t in range(T):
        want = _brute_route_token(sp[t], G, K, M, gk)
        assert list(idx[t]) == want, (t, list(idx[t]), want)
        chosen = s[t, want].astype(np.float64)
        np.testing.assert_allclose(gate[t], chosen / chosen.sum(), rtol=1e-7)


def test_all_groups_allowed_is_plain_topk():
    rng = np.random.default_rng(3)
    T, E, G, K = 64, 32, 4, 6
    s = (rng.integers(1, 16, (T, E)) / 16.0).astype(F32)
    b = np.zeros(E, F32)
    idx, _ = om.select_experts(s, b, G, K, G)
    for t in range(T):
        want = sorted(range(E), key=lambda e: (-float(s[t, e]), e))[:K]
        assert list(idx[t]) == want


def test_all_scores_tie_small_preset():
    """W_r = 0 and b = 0: every affinity is 0.5, so groups 0,1 and experts
    0..3 win every tie, each with gate 1/4."""
    T, d, E, G, K, M = 8, 16, 16, 4, 4, 2
    x = np.random.default_rng(0).standard_normal((T, d)).astype(F32)
    s = om.router_scores(x, np.zeros((E, d), F32))
    assert np.all(s == F32(0.5))
    idx, gate = om.select_experts(s, np.zeros(E, F32), G, K, M)
    assert np.all(idx == np.arange(4)[None, :])
    assert np.all(gate == F32(0.25))


def test_selection_invariants():
    rng = np.random.default_rng(7)
    T, E, G, K, M = 512, 64, 8, 6, 3
    s = rng.uniform(0, 1, (T, E)).astype(F32)
    b = rng.uniform(-0.05, 0.05, E).astype(F32)
    idx, gate = om.select_experts(s, b, G, K, M)
    sp = om.biased_scores(s, b)
    gsz = E // G
    for t in range(T):
        assert len(set(idx[t])) == K
        groups = set(int(e) // gsz for e in idx[t])
        assert len(groups) <= M
        # no unchosen expert of a chosen group beats the weakest chosen one
        w = int(idx[t, K - 1])
        for g in groups:
            for e in range(g * gsz, (g + 1) * gsz):
                if e not in idx[t]:
                    assert sp[t, e] < sp[t, w] or (sp[t, e] == sp[t, w] and e > w)
    np.testing.assert_allclose(gate.astype(np.float64).sum(1), 1.0, atol=1e-6)
    # outputs ordered by (s' desc, index asc)
    key = np.take_along_axis(sp, idx, 1)
    assert np.all(key[:, :-1] >= key[:, 1:])
    counts = om.expert_counts(idx, E)
    assert counts.sum() == T * K


def test_bias_moves_selection_not_gates():
    """The gates of a chosen set are the same whatever bias chose it."""
    rng = np.random.default_rng(11)
    T, E, G, K, M = 256, 32, 4, 4, 2
    s = rng.uniform(0, 1, (T, E)).astype(F32)
    b = rng.uniform(-0.3, 0.3, E).astype(F32)
    idx_b, gate_b = om.select_experts(s, b, G, K, M)
    idx_0, gate_0 = om.select_experts(s, np.zeros(E, F32), G, K, M)
    assert (idx_b != idx_0).any()  # the bias does steer routing
    for t in range(T):
        chosen = s[t, idx_b[t]].astype(np.float64)
        np.testing.assert_array_equal(gate_b[t], (chosen / chosen.sum()).astype(F32))
        if set(idx_b[t]) == set(idx_0[t]):
            np.testing.assert_array_equal(np.sort(gate_b[t]), np.sort(gate_0[t]))


# --------------------------------------------------------------------------
# scores
# --------------------------------------------------------------------------

def test_router_scores_closed_form():
    x = np.array([[2.0, 0.0], [0.0, -1.0], [0.0, 0.0]], F32)
    w = np.array([[0.5, 3.0], [0.25, -2.0]], F32)
    s = om.router_scores(x, w)
    u = [[1.0, 0.5], [-3.0, 2.0], [0.0, 0.0]]
    for t in range(3):
        for e in range(2):
            assert s[t, e] == F32(1.0 / (1.0 + math.exp(-u[t][e])))


# --------------------------------------------------------------------------
# count, scan, permutation
# --------------------------------------------------------------------------

def test_permutation_against_sort():
    rng = np.random.default_rng(5)
    T, E, K = 300, 16, 4
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    counts = om.expert_counts(idx, E)
    off = om.exclusive_offsets(counts)
    st, sp = om.permutation(idx, E)
    pairs = sorted((int(idx[t, k]), t, k) for t in range(T) for k in range(K))
    for p, (e, t, k) in enumerate(pairs):
        assert st[p] == t and sp[t, k] == p
        assert off[e] <= p < off[e + 1]
    assert off[-1] == T * K
    assert sorted(sp.ravel().tolist()) == list(range(T * K))


# --------------------------------------------------------------------------
# bias update
# --------------------------------------------------------------------------

def test_bias_update_moves_toward_balance():
    rng = np.random.default_rng(2)
    T, E, G, K, M, gamma = 256, 16, 4, 4, 2, 1e-3
    s = (rng.uniform(0.2, 0.6, (T, E)) + np.linspace(0.2, 0, E)).astype(F32)
    biases, idxs, loads = om.bias_balancing_loop(s, np.zeros(E, F32), 10, gamma, G, K, M)
    prev = np.zeros(E, F32)
    target = T * K / E
    for b, idx in zip(biases, idxs):
        counts = om.expert_counts(idx, E)
        for e in range(E):
            if counts[e] > target:
                assert b[e] == F32(prev[e] - F32(gamma))
            elif counts[e] < target:
                assert b[e] == F32(prev[e] + F32(gamma))
            else:
                assert b[e] == prev[e]
        prev = b
    assert loads[-1] < loads[0]  # balancing reduces the peak load here


def test_load_max_over_mean():
    counts = np.array([4, 0, 2, 2], np.int32)  # T*K = 8, E = 4, mean 2
    assert om.load_max_over_mean(counts, 4, 2) == 2.0


def test_bias_checkpoint_round_trip():
    import torch
    from mixture_experts_layer_100_b300 import state
    b = torch.tensor([1e-3, -2e-3, 0.0, -0.0, 3.4e38, 1.17549435e-38], dtype=torch.float32)
    blob = state.save_bias(b, step=42)
    b2, step = state.load_bias(blob)
    assert step == 42 and torch.equal(b2.view(torch.int32), b.view(torch.int32))
    with pytest.raises(ValueError):
        state.load_bias(b"XXXX" + blob[4:])
    with pytest.raises(ValueError):
        state.load_bias(blob[:-4])


# --------------------------------------------------------------------------
# sequence-wise balance statistic
# --------------------------------------------------------------------------

def test_sequence_balance_hand_example():
    g = _golden("seq_balance_example.json")
    loss, f, P = om.sequence_balance(np.array(g["scores"], F32), np.array(g["topk_idx"]), g["seq_len"], g["alpha"])
    np.testing.assert_array_equal(f, np.array(g["f"], float))
    np.testing.assert_allclose(P, [[n / d for n, d in row] for row in g["P_num_den"]], rtol=1e-15)
    np.testing.assert_allclose(loss, [n / d for n, d in g["loss_num_den"]], rtol=1e-15)


def test_sequence_balance_uniform_is_alpha():
    """Equal affinities and perfectly even choices: f_i = 1, P_i = 1/E, so
    the statistic is alpha exactly."""
    T, E, K = 64, 16, 4
    s = np.full((T, E), 0.3, F32)
    idx = np.array([[(4 * t + k) % E for k in range(K)] for t in range(T)])  # every expert 16 times
    loss, f, P = om.sequence_balance(s, idx, T, 0.01)
    np.testing.assert_allclose(f, 1.0, rtol=1e-15)
    np.testing.assert_allclose(P, 1.0 / E, rtol=1e-12)
    np.testing.assert_allclose(loss, [0.01], rtol=1e-12)


def test_sequence_balance_invariants_and_loops():
    rng = np.random.default_rng(31)
    T, E, K, L = 300, 32, 6, 128          # runs of 128, 128, 44
    s = rng.uniform(0.01, 1.0, (T, E)).astype(F32)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    loss, f, P = om.sequence_balance(s, idx, L, 1e-3)
    assert loss.shape == (3,)
    np.testing.assert_allclose(f.sum(axis=1), E, rtol=1e-12)    # sum_i f_i = E
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=1e-12)  # sum_i P_i = 1
    # plain loops over the definition
    for q, (a, b) in enumerate([(0, 128), (128, 256), (256, 300)]):
        n = b - a
        want = 0.0
        for i in range(E):
            c = sum(1 for t in range(a, b) for k in range(K) if idx[t, k] == i)
            p = sum(float(s[t, i]) / sum(float(v) for v in s[t]) for t in range(a, b)) / n
            want += (E / (K * n)) * c * p
        assert abs(loss[q] - 1e-3 * want) <= 1e-12 * abs(want)


def test_sequence_balance_concentrated():
    """Every token chooses experts 0..K-1 and puts all its affinity mass
    there: f_i = E/K and P_i = 1/K on those, so the statistic is alpha * E / K."""
    T, E, K = 40, 16, 4
    s = np.zeros((T, E), F32)
    s[:, :K] = 0.25
    idx = np.tile(np.arange(K), (T, 1))
    loss, _, _ = om.sequence_balance(s, idx, T, 0.5)
    np.testing.assert_allclose(loss, [0.5 * E / K], rtol=1e-12)
