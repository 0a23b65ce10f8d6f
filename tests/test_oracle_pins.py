"""Pins for the CPU oracle: worked examples printed on the pages, closed forms,
library routines and brute force. CPU only (no GPU marker).

A mistake anywhere in the oracle (a dropped term, a wrong sign or index, a
transposed operand, an overwrite instead of an add) fails at least one test
here; the mutation tests at the end plant such mistakes in the oracle and
check that the pins catch them.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

from conftest import load_golden
from oracle import moe_oracle as O


# ---------------------------------------------------------------- router ---
def test_router_logits_vs_library_linear():
    rng = np.random.default_rng(1)
    h = rng.standard_normal((7, 5))
    W = rng.standard_normal((3, 5))
    b = rng.standard_normal(3)
    ref = Fnn.linear(torch.from_numpy(h), torch.from_numpy(W), torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(O.router_logits(h, W, b), ref, rtol=0, atol=1e-12)
    ref0 = Fnn.linear(torch.from_numpy(h), torch.from_numpy(W)).numpy()
    np.testing.assert_allclose(O.router_logits(h, W), ref0, rtol=0, atol=1e-12)
    # orientation: logit i is row i of W_r dotted with h (not a column)
    h1 = np.array([[1.0, 0.0, 0.0, 0.0, 0.0]])
    np.testing.assert_array_equal(O.router_logits(h1, W)[0], W[:, 0])


# ----------------------------------------------------------------- scores ---
def test_page1_softmax_example():
    g = load_golden("page1_softmax_example.json")
    z = np.array([g["logits"]])
    tol = g["printed_abs_tol"]
    p = O.softmax(z)
    np.testing.assert_allclose(p[0], g["softmax_printed"], atol=tol, rtol=0)
    S, gates, _, _ = O.route(z, g["k"], O.SOFTMAX, O.NORM_SELECTED)
    assert S[0].tolist() == g["selected"]
    np.testing.assert_allclose(gates[0], g["gates_printed"], atol=tol, rtol=0)
    np.testing.assert_allclose(O.gates_from_selected_logits(z, S)[0],
                               g["gates_printed"], atol=tol, rtol=0)


def test_page2_selected_renorm_example():
    g = load_golden("page2_selected_renorm_example.json")
    z = np.array([g["scores"]])
    S, gates, _, _ = O.route(z, g["k"], O.SOFTMAX, O.NORM_SELECTED)
    assert S[0].tolist() == g["selected"]
    np.testing.assert_allclose(gates[0], g["gates_printed"], atol=g["printed_abs_tol"], rtol=0)
    # closed form: e^2 / (e^2 + e^1) = 1 / (1 + e^-1)
    assert abs(gates[0, 0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15


def test_softmax_vs_library_and_closed_forms():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((11, 9)) * 3
    np.testing.assert_allclose(O.softmax(z), torch.softmax(torch.from_numpy(z), -1).numpy(),
                               atol=1e-15, rtol=0)
    np.testing.assert_allclose(O.softmax(np.zeros((1, 8))), np.full((1, 8), 1 / 8), atol=1e-15)
    a = 0.7
    p = O.softmax(np.array([[a, 0.0]]))
    assert abs(p[0, 0] - 1 / (1 + math.exp(-a))) < 1e-15
    # large logits do not overflow
    assert np.isfinite(O.softmax(np.array([[1000.0, 999.0]]))).all()


def test_sigmoid_vs_library_and_closed_forms():
    rng = np.random.default_rng(3)
    z = rng.standard_normal((5, 6)) * 4
    np.testing.assert_allclose(O.sigmoid(z), torch.sigmoid(torch.from_numpy(z)).numpy(),
                               atol=1e-15, rtol=0)
    assert O.sigmoid(np.array([0.0]))[0] == 0.5
    assert abs(O.sigmoid(np.array([math.log(3.0)]))[0] - 0.75) < 1e-15
    assert O.sigmoid(np.array([-800.0]))[0] == 0.0


def test_renorm_identity_softmax_then_renorm_equals_topk_then_softmax():
    rng = np.random.default_rng(4)
    for k in (1, 2, 3, 8):
        z = rng.standard_normal((50, 16)) * 2
        S = O.select_topk(z, k)
        a = O.gates_from_scores(O.softmax(z), S, O.NORM_SELECTED)
        b = O.gates_from_selected_logits(z, S)
        np.testing.assert_allclose(a, b, atol=1e-12, rtol=0)
        np.testing.assert_allclose(a.sum(-1), 1.0, atol=1e-12)


# -------------------------------------------------------------- selection ---
def test_topk_ties_go_to_lower_index():
    q = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]])
    assert O.select_topk(q, 1)[0].tolist() == [1]
    assert O.select_topk(q, 2)[0].tolist() == [1, 2]
    assert O.select_topk(q, 3)[0].tolist() == [1, 2, 4]
    assert O.select_topk(q, 5)[0].tolist() == [1, 2, 4, 3, 0]
    q0 = np.zeros((1, 6))
    assert O.select_topk(q0, 3)[0].tolist() == [0, 1, 2]


def test_topk_vs_rank_counting_brute_force():
    rng = np.random.default_rng(5)
    for _ in range(300):
        N = int(rng.integers(1, 9))
        k = int(rng.integers(1, N + 1))
        q = np.round(rng.standard_normal(N) * 2) / 2   # many exact ties
        assert O.select_topk(q[None], k)[0].tolist() == O.topk_by_rank_count(q, k)


def test_topk_vs_subset_brute_force_and_library():
    rng = np.random.default_rng(6)
    for _ in range(200):
        N = int(rng.integers(1, 8))
        k = int(rng.integers(1, N + 1))
        q = rng.standard_normal(N)          # continuous: no ties
        S = O.select_topk(q[None], k)[0]
        assert set(S.tolist()) == O.topk_by_subsets(q, k)
        tv, ti = torch.topk(torch.from_numpy(q), k)
        assert S.tolist() == ti.tolist()


def test_switch_top1_keeps_full_softmax_probability():
    rng = np.random.default_rng(7)
    z = rng.standard_normal((20, 6))
    S, g, p, _ = O.route(z, 1, O.SOFTMAX, O.NORM_NONE)
    np.testing.assert_allclose(g[:, 0], p.max(-1), atol=0)
    assert (g[:, 0] >= 1 / 6 - 1e-15).all() and (g[:, 0] < 1).all()
    # with renormalisation a top-1 gate would be exactly 1
    _, g1, _, _ = O.route(z, 1, O.SOFTMAX, O.NORM_SELECTED)
    np.testing.assert_array_equal(g1, 1.0)
    # one expert: the gate is 1 either way
    _, gN1, _, _ = O.route(z[:, :1], 1, O.SOFTMAX, O.NORM_NONE)
    np.testing.assert_array_equal(gN1, 1.0)


def test_k_equals_N_gates_are_the_probabilities():
    rng = np.random.default_rng(8)
    z = rng.standard_normal((10, 5))
    S, g, p, _ = O.route(z, 5, O.SOFTMAX, O.NORM_SELECTED)
    np.testing.assert_allclose(g, np.take_along_axis(p, S, -1), atol=1e-15)
    np.testing.assert_allclose(g.sum(-1), 1.0, atol=1e-15)


def test_sigmoid_bias_steers_selection_not_gates():
    z = np.array([[2.0, 0.0, -1.0]])
    bias = np.array([0.0, 0.0, 10.0])
    S, g, p, q = O.route(z, 2, O.SIGMOID, O.NORM_SELECTED, bias)
    assert S[0].tolist() == [2, 0]
    s2, s0 = 1 / (1 + math.exp(1.0)), 1 / (1 + math.exp(-2.0))
    np.testing.assert_allclose(g[0], [s2 / (s2 + s0), s0 / (s2 + s0)], atol=1e-15)
    # without the bias expert 1 (sigma(0) = 0.5) beats expert 2
    S0, _, _, _ = O.route(z, 2, O.SIGMOID, O.NORM_SELECTED)
    assert S0[0].tolist() == [0, 1]
    # NORM_NONE keeps the raw sigmoid scores
    _, gn, _, _ = O.route(z, 2, O.SIGMOID, O.NORM_NONE, bias)
    np.testing.assert_allclose(gn[0], [s2, s0], atol=1e-15)


def test_sigmoid_bias_brute_force():
    rng = np.random.default_rng(9)
    for _ in range(200):
        N = int(rng.integers(2, 9))
        k = int(rng.integers(1, N + 1))
        z = rng.standard_normal(N) * 2
        b = rng.standard_normal(N) * 0.3
        S, g, _, _ = O.route(z[None], k, O.SIGMOID, O.NORM_SELECTED, b)
        sig = [1 / (1 + math.exp(-v)) for v in z]
        q = [sig[i] + b[i] for i in range(N)]
        assert S[0].tolist() == O.topk_by_rank_count(q, k)
        tot = sum(sig[i] for i in S[0])
        np.testing.assert_allclose(g[0], [sig[i] / tot for i in S[0]], atol=1e-14)


def test_gate_matrix_matches_scatter():
    rng = np.random.default_rng(10)
    z = rng.standard_normal((6, 5))
    S, g, _, _ = O.route(z, 2)
    G = O.gate_matrix(S, g, 5)
    ref = torch.zeros(6, 5, dtype=torch.float64).scatter_(
        -1, torch.from_numpy(S), torch.from_numpy(g)).numpy()
    np.testing.assert_array_equal(G, ref)


# --------------------------------------------------------------- dispatch ---
def _choices(golden):
    S = np.array([[e for e, _ in row] for row in golden["choices"]])
    g = np.array([[w for _, w in row] for row in golden["choices"]])
    return S, g


def test_page1_dispatch_table():
    gd = load_golden("page1_dispatch_table.json")
    S, _ = _choices(gd)
    counts, offsets, row_token, inv = O.dispatch(S, gd["N"])
    assert counts.tolist() == gd["counts"]
    assert offsets.tolist() == gd["offsets"]
    for e, toks in gd["buckets"].items():
        e = int(e)
        assert row_token[offsets[e]:offsets[e + 1]].tolist() == toks
    for t in range(S.shape[0]):
        for j in range(S.shape[1]):
            r = inv[t, j]
            assert row_token[r] == t and offsets[S[t, j]] <= r < offsets[S[t, j] + 1]


def test_dispatch_brute_force():
    rng = np.random.default_rng(11)
    for _ in range(50):
        N = int(rng.integers(1, 10))
        k = int(rng.integers(1, N + 1))
        T = int(rng.integers(0, 40))
        S = np.array([rng.permutation(N)[:k] for _ in range(T)]).reshape(T, k)
        counts, offsets, row_token, inv = O.dispatch(S, N)
        pairs = sorted((int(S[t, j]), t, j) for t in range(T) for j in range(k))
        assert row_token.tolist() == [t for _, t, _ in pairs]
        for r, (e, t, j) in enumerate(pairs):
            assert inv[t, j] == r
        assert counts.sum() == T * k
        assert counts.tolist() == [sum(1 for p in pairs if p[0] == e) for e in range(N)]


# ------------------------------------------------------------- expert FFN ---
def test_swiglu_vs_library():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((9, 6))
    Wg, Wu, Wd = rng.standard_normal((5, 6)), rng.standard_normal((5, 6)), rng.standard_normal((6, 5))
    tx, tg, tu, td = map(torch.from_numpy, (x, Wg, Wu, Wd))
    ref = Fnn.linear(Fnn.silu(Fnn.linear(tx, tg)) * Fnn.linear(tx, tu), td).numpy()
    np.testing.assert_allclose(O.swiglu_expert(x, Wg, Wu, Wd), ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(O.silu(x), Fnn.silu(tx).numpy(), atol=1e-15, rtol=0)


def test_swiglu_scalar_closed_form():
    a, b, c = 1.3, -0.4, 2.5
    y = O.swiglu_expert(np.array([[1.0]]), np.array([[a]]), np.array([[b]]), np.array([[c]]))
    assert abs(y[0, 0] - c * (a / (1 + math.exp(-a))) * b) < 1e-15
    # gate branch is the SiLU one: swapping W_gate and W_up changes the result
    y2 = O.swiglu_expert(np.array([[1.0]]), np.array([[b]]), np.array([[a]]), np.array([[c]]))
    assert abs(y2[0, 0] - y[0, 0]) > 1e-3


# ---------------------------------------------------------------- combine ---
def test_page2_combine_example():
    gd = load_golden("page2_combine_example.json")
    S, g = _choices(gd)
    counts, offsets, row_token, inv = O.dispatch(S, gd["N"])
    y_rows = np.zeros((S.size, 2))
    for t in range(S.shape[0]):
        for j in range(S.shape[1]):
            y_rows[inv[t, j]] = gd["expert_outputs"][f"{t}:{S[t, j]}"]
    # dispatch regrouping of the page: expert 2 receives both tokens
    assert counts.tolist() == [1, 1, 2]
    out = O.combine(y_rows, inv, g)
    np.testing.assert_allclose(out, gd["y_printed"], atol=1e-12, rtol=0)


def test_combine_with_shared_and_zero_gates():
    rng = np.random.default_rng(13)
    y_rows = rng.standard_normal((6, 4))
    inv = np.array([[0, 3], [1, 4], [2, 5]])
    ysh = rng.standard_normal((3, 4))
    g = np.zeros((3, 2))
    np.testing.assert_array_equal(O.combine(y_rows, inv, g, ysh), ysh)
    g1 = np.array([[1.0, 0.0], [0.0, 1.0], [0.5, 0.5]])
    out = O.combine(y_rows, inv, g1)
    np.testing.assert_allclose(out[0], y_rows[0]); np.testing.assert_allclose(out[1], y_rows[4])
    np.testing.assert_allclose(out[2], 0.5 * (y_rows[2] + y_rows[5]))


# ------------------------------------------------------------ whole layer ---
def _tiny(rng, T, d, N, F, shared=False, F_sh=3):
    h = rng.standard_normal((T, d))
    W_r = rng.standard_normal((N, d))
    Wg = rng.standard_normal((N, F, d)); Wu = rng.standard_normal((N, F, d))
    Wd = rng.standard_normal((N, d, F))
    sh = None
    if shared:
        sh = (rng.standard_normal((F_sh, d)), rng.standard_normal((F_sh, d)),
              rng.standard_normal((d, F_sh)))
    return h, W_r, Wg, Wu, Wd, sh


@pytest.mark.parametrize("score", [O.SOFTMAX, O.SIGMOID])
@pytest.mark.parametrize("norm", [O.NORM_SELECTED, O.NORM_NONE])
@pytest.mark.parametrize("use_bias", [False, True])
@pytest.mark.parametrize("shared", [False, True])
def test_sparse_equals_dense_masked(score, norm, use_bias, shared):
    rng = np.random.default_rng(14)
    for _ in range(4):
        T, d, N, F = int(rng.integers(1, 17)), int(rng.integers(1, 9)), int(rng.integers(1, 7)), int(rng.integers(1, 6))
        k = int(rng.integers(1, N + 1))
        h, W_r, Wg, Wu, Wd, sh = _tiny(rng, T, d, N, F, shared)
        bias = rng.standard_normal(N) * 0.2 if use_bias else None
        ys, z, S, g = O.moe_forward(h, W_r, Wg, Wu, Wd, k, score, norm, bias, shared=sh)
        yd, _, _, _ = O.moe_forward_dense(h, W_r, Wg, Wu, Wd, k, score, norm, bias, shared=sh)
        np.testing.assert_allclose(ys, yd, atol=1e-12, rtol=1e-12)


def test_single_expert_is_dense_swiglu_ffn():
    rng = np.random.default_rng(15)
    h, W_r, Wg, Wu, Wd, _ = _tiny(rng, 12, 6, 1, 5)
    y, _, S, g = O.moe_forward(h, W_r, Wg, Wu, Wd, 1)
    th = torch.from_numpy(h)
    ref = Fnn.linear(Fnn.silu(Fnn.linear(th, torch.from_numpy(Wg[0]))) *
                     Fnn.linear(th, torch.from_numpy(Wu[0])), torch.from_numpy(Wd[0])).numpy()
    np.testing.assert_allclose(y, ref, atol=1e-12, rtol=0)
    assert (S == 0).all() and (g == 1).all()


def test_shared_expert_alone_when_routed_outputs_vanish():
    rng = np.random.default_rng(16)
    h, W_r, Wg, Wu, Wd, sh = _tiny(rng, 10, 6, 4, 5, shared=True, F_sh=7)
    Wd0 = np.zeros_like(Wd)
    y, _, _, _ = O.moe_forward(h, W_r, Wg, Wu, Wd0, 2, shared=sh)
    th = torch.from_numpy(h)
    ref = Fnn.linear(Fnn.silu(Fnn.linear(th, torch.from_numpy(sh[0]))) *
                     Fnn.linear(th, torch.from_numpy(sh[1])), torch.from_numpy(sh[2])).numpy()
    np.testing.assert_allclose(y, ref, atol=1e-12, rtol=0)


def test_stagewise_composition_equals_layer():
    """route -> dispatch -> expert_rows -> combine equals moe_forward."""
    rng = np.random.default_rng(17)
    h, W_r, Wg, Wu, Wd, sh = _tiny(rng, 15, 6, 5, 4, shared=True)
    bias = rng.standard_normal(5) * 0.1
    y, z, S, g = O.moe_forward(h, W_r, Wg, Wu, Wd, 3, O.SIGMOID, O.NORM_SELECTED, bias, shared=sh)
    counts, offsets, row_token, inv = O.dispatch(S, 5)
    y_rows = O.expert_rows(h[row_token], offsets, Wg, Wu, Wd)
    out = O.combine(y_rows, inv, g, O.swiglu_expert(h, *sh))
    np.testing.assert_allclose(out, y, atol=1e-12, rtol=0)


def test_page1_worked_output_weights():
    """The page's y_t = 0.599 E0 + 0.401 E2 with E_i replaced by unit vectors."""
    g = load_golden("page1_softmax_example.json")
    z = np.array([g["logits"]])
    S, gates, _, _ = O.route(z, 2)
    counts, offsets, row_token, inv = O.dispatch(S, 4)
    y_rows = np.zeros((2, 4))
    for j in range(2):
        y_rows[inv[0, j], S[0, j]] = 1.0        # E_i(h) = e_i
    out = O.combine(y_rows, inv, gates)
    np.testing.assert_allclose(out[0], [0.599, 0, 0.401, 0], atol=5e-4)


# ------------------------------------------------- mutation: pins catch bugs ---
def _run_pins_expect_failure(monkeypatch, name, bad, pins):
    monkeypatch.setattr(O, name, bad)
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, f"a planted mistake in {name} went unnoticed"


def test_mutation_overwrite_instead_of_add(monkeypatch):
    def bad_combine(y_rows, inv, g, y_shared=None):
        out = np.zeros((inv.shape[0], y_rows.shape[1]))
        for j in range(inv.shape[1]):
            out = g[:, j:j + 1] * y_rows[inv[:, j]]          # overwrite
        return out
    _run_pins_expect_failure(monkeypatch, "combine", bad_combine, [test_page2_combine_example])


def test_mutation_transposed_gate_up(monkeypatch):
    def bad_swiglu(x, Wg, Wu, Wd):
        return (O.silu(x @ np.asarray(Wu).T) * (x @ np.asarray(Wg).T)) @ np.asarray(Wd).T
    _run_pins_expect_failure(monkeypatch, "swiglu_expert", bad_swiglu,
                             [test_swiglu_vs_library, test_swiglu_scalar_closed_form])


def test_mutation_tie_break_to_higher_index(monkeypatch):
    def bad_topk(q, k):
        q = np.asarray(q, dtype=np.float64)
        order = np.argsort(-q[:, ::-1], axis=-1, kind="stable")
        return (q.shape[-1] - 1 - order)[:, :k]
    _run_pins_expect_failure(monkeypatch, "select_topk", bad_topk,
                             [test_topk_ties_go_to_lower_index])


def test_mutation_bias_in_gates(monkeypatch):
    orig = O.gates_from_scores
    def bad_route(z, k, score_kind=O.SOFTMAX, norm=O.NORM_SELECTED, sel_bias=None):
        p = O.scores(z, score_kind)
        q = p if sel_bias is None else p + np.asarray(sel_bias)[None, :]
        S = O.select_topk(q, k)
        return S, orig(q, S, norm), p, q                      # gates from q
    _run_pins_expect_failure(monkeypatch, "route", bad_route,
                             [test_sigmoid_bias_steers_selection_not_gates])


def test_mutation_dispatch_unstable_order(monkeypatch):
    def bad_dispatch(S, N):
        T, k = S.shape
        e_flat = S.reshape(-1); t_flat = np.repeat(np.arange(T), k)
        counts = np.bincount(e_flat, minlength=N)
        offsets = np.concatenate([[0], np.cumsum(counts)])
        order = np.lexsort((-t_flat, e_flat))                  # tokens descending
        inv = np.empty(T * k, dtype=np.int64); inv[order] = np.arange(T * k)
        return counts, offsets, t_flat[order], inv.reshape(T, k)
    _run_pins_expect_failure(monkeypatch, "dispatch", bad_dispatch, [test_page1_dispatch_table])


# -------------------------------------------------------- routing statistics ---
def test_stats_uniform_closed_forms():
    """Equal logits and perfectly balanced assignments: L_bal = 1,
    entropy = log N, z-loss = (z0 + log N)^2."""
    T, N, k = 8, 4, 2
    z0 = 0.7
    z = np.full((T, N), z0)
    S = np.array([[(t + j) % N for j in range(k)] for t in range(T)])
    for score in (O.SOFTMAX, O.SIGMOID):
        st = O.routing_stats(z, S, score, N)
        assert abs(st["L_bal"] - 1.0) < 1e-12
        assert abs(st["entropy"] - math.log(N)) < 1e-12
        assert abs(st["L_z"] - (z0 + math.log(N)) ** 2) < 1e-12
        np.testing.assert_allclose(st["P"], 1 / N, atol=1e-15)
        np.testing.assert_allclose(st["f"], 1 / N, atol=1e-15)


def test_stats_collapse_limit():
    """Every token sent to expert 0 with probability -> 1: L_bal -> N, entropy -> 0."""
    T, N = 5, 6
    z = np.zeros((T, N)); z[:, 0] = 60.0
    S = np.zeros((T, 1), dtype=np.int64)
    st = O.routing_stats(z, S, O.SOFTMAX, N)
    assert abs(st["L_bal"] - N) < 1e-12
    assert st["entropy"] < 1e-20
    assert abs(st["L_z"] - 60.0 ** 2) < 1e-9


def test_stats_brute_force_and_library():
    rng = np.random.default_rng(21)
    T, N, k = 13, 5, 2
    z = rng.standard_normal((T, N)) * 2
    S, _, _, _ = O.route(z, k)
    st = O.routing_stats(z, S, O.SOFTMAX, N)
    # brute force, token by token with math
    P = [0.0] * N; cnt = [0] * N; lz = 0.0; H = 0.0
    for t in range(T):
        ex = [math.exp(v) for v in z[t]]
        tot = sum(ex)
        lz += math.log(tot) ** 2
        for i in range(N):
            P[i] += ex[i] / tot / T
            H -= ex[i] / tot * math.log(ex[i] / tot) / T
        for j in range(k):
            cnt[S[t, j]] += 1
    f = [c / (T * k) for c in cnt]
    assert abs(st["L_bal"] - N * sum(a * b for a, b in zip(f, P))) < 1e-12
    assert abs(st["L_z"] - lz / T) < 1e-12
    assert abs(st["entropy"] - H) < 1e-12
    tz = torch.from_numpy(z)
    np.testing.assert_allclose(O.logsumexp(z), torch.logsumexp(tz, -1).numpy(), atol=1e-13)
    np.testing.assert_allclose(st["entropy"], torch.distributions.Categorical(logits=tz).entropy().mean().item(), atol=1e-12)


# ------------------------------------------------------- group-limited top-k ---
def test_page2_group_limited_example():
    g = load_golden("page2_group_limited_example.json")
    q = np.array([g["scores"]])
    k = g["k"]
    assert sorted(q[0, O.select_topk(q, k)[0]].tolist()) == sorted(g["unrestricted"])
    Sm = O.select_topk_grouped(q, k, 2, 1, O.GROUP_MAX)
    assert q[0, Sm[0]].tolist() == g["group_max_keep1"]
    Ss = O.select_topk_grouped(q, k, 2, 1, O.GROUP_TOPM_SUM, top_m=2)
    assert q[0, Ss[0]].tolist() == g["group_top2sum_keep1"]


def test_grouped_special_cases_reduce_to_plain_topk():
    rng = np.random.default_rng(31)
    q = np.round(rng.standard_normal((40, 12)) * 2) / 2
    for k in (1, 3, 5):
        plain = O.select_topk(q, k)
        # every group kept
        np.testing.assert_array_equal(O.select_topk_grouped(q, k, 4, 4), plain)
        # one expert per group, keep the k best groups
        np.testing.assert_array_equal(O.select_topk_grouped(q, k, 12, k), plain)


def test_grouped_masks_with_minus_infinity_not_zero():
    q = np.array([[-5.0, -6.0, -1.0, -2.0]])
    # group B (max -1) kept; group A must not win through a zero mask
    assert O.select_topk_grouped(q, 2, 2, 1).tolist() == [[2, 3]]


def test_grouped_brute_force_and_errors():
    rng = np.random.default_rng(32)
    for _ in range(100):
        G = int(rng.integers(1, 5)); gs = int(rng.integers(1, 4)); N = G * gs
        kg = int(rng.integers(1, G + 1))
        k = int(rng.integers(1, kg * gs + 1))
        m = int(rng.integers(1, gs + 1))
        q = np.round(rng.standard_normal(N) * 2) / 2
        for rule in (O.GROUP_MAX, O.GROUP_TOPM_SUM):
            got = O.select_topk_grouped(q[None], k, G, kg, rule, m)[0].tolist()
            # brute force: group scores, rank-count the groups, then rank-count experts
            def gscore(gi):
                vals = sorted(q[gi * gs:(gi + 1) * gs], reverse=True)
                return vals[0] if rule == O.GROUP_MAX else sum(vals[:m])
            kept = set(O.topk_by_rank_count([gscore(gi) for gi in range(G)], kg))
            cand = [float(q[i]) if i // gs in kept else -np.inf for i in range(N)]
            assert got == O.topk_by_rank_count(cand, k)
    with pytest.raises(ValueError):
        O.select_topk_grouped(np.zeros((1, 8)), 5, 4, 2)      # 2 groups x 2 = 4 < 5
    with pytest.raises(ValueError):
        O.select_topk_grouped(np.zeros((1, 9)), 2, 4, 2)      # 9 experts, 4 groups


# ------------------------------------------------------------ capacity ---
def test_capacity_formula():
    assert O.expert_capacity(4, 2, 4, 1.0) == 2
    assert O.expert_capacity(4, 2, 4, 1.25) == 3          # ceil(2.5)
    assert O.expert_capacity(4096, 2, 8, 1.0) == 1024
    assert O.expert_capacity(10, 1, 3, 1.0) == 4          # ceil(10/3)


def test_page1_dispatch_table_with_capacity_two():
    gd = load_golden("page1_dispatch_table.json")
    S, _ = _choices(gd)
    counts, offsets, row_token, inv = O.dispatch_capacity(S, gd["N"], 2)
    # E2 receives T0, T1, T3 in token order; with C = 2 the pair of T3 is dropped
    assert counts.tolist() == [2, 2, 2, 1]
    assert row_token.tolist() == [0, 2, 1, 3, 0, 1, 2]
    assert inv[3].tolist() == [-1, 3]                     # T3: (E2 dropped, E1 kept)
    assert (inv >= 0).sum() == 7


def test_capacity_large_is_dropless_and_zero_drops_all():
    rng = np.random.default_rng(41)
    S = np.array([rng.permutation(6)[:2] for _ in range(30)])
    c0, o0, r0, i0 = O.dispatch(S, 6)
    c1, o1, r1, i1 = O.dispatch_capacity(S, 6, 10 ** 6)
    assert c0.tolist() == c1.tolist() and r0.tolist() == r1.tolist() and (i0 == i1).all()
    c2, o2, r2, i2 = O.dispatch_capacity(S, 6, 0)
    assert c2.sum() == 0 and (i2 == -1).all() and r2.size == 0


def test_capacity_layer_brute_force_and_limits():
    rng = np.random.default_rng(42)
    h, W_r, Wg, Wu, Wd, sh = _tiny(rng, 14, 5, 4, 3, shared=True)
    y_full, _, _, _ = O.moe_forward(h, W_r, Wg, Wu, Wd, 2, shared=sh)
    y_big, _, _, inv_big = O.moe_forward_capacity(h, W_r, Wg, Wu, Wd, 2, 100, shared=sh)
    np.testing.assert_allclose(y_big, y_full, atol=1e-12)
    y0, _, _, _ = O.moe_forward_capacity(h, W_r, Wg, Wu, Wd, 2, 0, shared=sh)
    np.testing.assert_allclose(y0, O.swiglu_expert(h, *sh), atol=1e-12)
    # brute force for C = 3: per expert keep the 3 lowest-index tokens
    C = 3
    y3, S, g, inv = O.moe_forward_capacity(h, W_r, Wg, Wu, Wd, 2, C, shared=sh)
    ref = O.swiglu_expert(h, *sh)
    for e in range(4):
        toks = [t for t in range(14) for j in range(2) if S[t, j] == e][:C]
        for t in toks:
            j = list(S[t]).index(e)
            ref[t] += g[t, j] * O.swiglu_expert(h[t:t + 1], Wg[e], Wu[e], Wd[e])[0]
    np.testing.assert_allclose(y3, ref, atol=1e-12)


# ---------------------------------------------------------- expert choice ---
def test_expert_choice_hand_example():
    # 3 tokens, 2 experts, each expert picks 2 tokens by its column of p
    z = np.log(np.array([[0.7, 0.3], [0.2, 0.8], [0.6, 0.4]]))
    tokens, gates, p = O.expert_choice(z, 2)
    assert tokens.tolist() == [[0, 2], [1, 2]]          # E0: 0.7, 0.6; E1: 0.8, 0.4
    np.testing.assert_allclose(gates, [[0.7, 0.6], [0.8, 0.4]], atol=1e-15)
    # token 2 is picked by both experts; no token is left out here, none picked thrice


def test_expert_choice_ties_lower_token_and_loads_fixed():
    z = np.zeros((6, 3))                                 # every score equal
    tokens, _, _ = O.expert_choice(z, 4)
    assert tokens.tolist() == [[0, 1, 2, 3]] * 3
    rng = np.random.default_rng(51)
    z = rng.standard_normal((40, 5))
    tokens, gates, p = O.expert_choice(z, 7)
    assert tokens.shape == (5, 7)                        # every expert exactly C tokens
    for e in range(5):
        # brute force: the 7 largest p[:, e] with lower index first on ties
        assert set(tokens[e].tolist()) == set(O.topk_by_rank_count(p[:, e], 7))


def test_expert_choice_layer_vs_dense_mask():
    rng = np.random.default_rng(52)
    h, W_r, Wg, Wu, Wd, sh = _tiny(rng, 12, 5, 4, 3, shared=True)
    y, tokens, gates = O.moe_forward_expert_choice(h, W_r, Wg, Wu, Wd, 5, shared=sh)
    z = O.router_logits(h, W_r)
    p = O.softmax(z)
    G = np.zeros((12, 4))
    for e in range(4):
        G[tokens[e], e] = p[tokens[e], e]
    ref = O.swiglu_expert(h, *sh)
    for e in range(4):
        ref += G[:, e:e + 1] * O.swiglu_expert(h, Wg[e], Wu[e], Wd[e])
    np.testing.assert_allclose(y, ref, atol=1e-12)
    y0, _, _ = O.moe_forward_expert_choice(h, W_r, Wg, Wu, Wd, 0, shared=sh)
    np.testing.assert_allclose(y0, O.swiglu_expert(h, *sh), atol=1e-12)


# ------------------------------------ pins added for the remaining functions ---
def test_swiglu_act_vs_library_and_closed_form():
    """SiLU(x W_gate^T) ⊙ (x W_up^T) against torch in fp64, a scalar closed
    form, and the identity E(x) = act(x) W_down^T ("MOE 专家选择与路由机制" §一)."""
    rng = np.random.default_rng(61)
    x = rng.standard_normal((11, 7))
    Wg, Wu, Wd = rng.standard_normal((6, 7)), rng.standard_normal((6, 7)), rng.standard_normal((7, 6))
    tx, tg, tu = map(torch.from_numpy, (x, Wg, Wu))
    ref = (Fnn.silu(Fnn.linear(tx, tg)) * Fnn.linear(tx, tu)).numpy()
    np.testing.assert_allclose(O.swiglu_act(x, Wg, Wu), ref, atol=1e-13, rtol=0)
    np.testing.assert_allclose(O.swiglu_act(x, Wg, Wu) @ Wd.T, O.swiglu_expert(x, Wg, Wu, Wd),
                               atol=1e-12, rtol=0)
    # scalar: x = 2, W_gate = a, W_up = b -> silu(2a) * 2b
    a, b = 0.7, -1.9
    got = O.swiglu_act(np.array([[2.0]]), np.array([[a]]), np.array([[b]]))[0, 0]
    assert abs(got - (2 * a / (1 + math.exp(-2 * a))) * (2 * b)) < 1e-15
    # the SiLU is on the gate branch only: act(x; a, b) != act(x; b, a)
    got_sw = O.swiglu_act(np.array([[2.0]]), np.array([[b]]), np.array([[a]]))[0, 0]
    assert abs(got_sw - got) > 1e-2
    # SiLU(0) = 0 kills the row whatever the up branch holds
    assert O.swiglu_act(np.array([[0.0, 1.0]]), np.array([[1.0, 0.0]]), np.array([[0.0, 5.0]]))[0, 0] == 0.0


def _group_brute_force(q_row, p_row, k, n_group, topk_group, rule, top_m, norm):
    """Group-limited routing of one token by enumeration ("MoE：router 怎样选
    expert" §跨设备时，为什么还要先选组): group scores from sorted lists,
    the kept groups as the topk_group-subset with the largest score sum
    (distinct group scores make it unique), then the k-subset of the kept
    groups' experts with the largest selection-score sum; slots by descending
    q; gates from the un-biased scores p. Valid only without ties."""
    N = len(q_row)
    gs = N // n_group
    gsc = []
    for gi in range(n_group):
        vals = sorted((float(v) for v in q_row[gi * gs:(gi + 1) * gs]), reverse=True)
        gsc.append(vals[0] if rule == O.GROUP_MAX else sum(vals[:top_m]))
    kept = max(itertools.combinations(range(n_group), topk_group),
               key=lambda c: sum(gsc[i] for i in c))
    cand = [i for gi in kept for i in range(gi * gs, (gi + 1) * gs)]
    best = max(itertools.combinations(cand, k), key=lambda c: sum(float(q_row[i]) for i in c))
    S = sorted(best, key=lambda i: -float(q_row[i]))
    if norm == O.NORM_SELECTED:
        tot = sum(float(p_row[i]) for i in S)
        g = [float(p_row[i]) / tot for i in S]
    else:
        g = [float(p_row[i]) for i in S]
    return S, g


@pytest.mark.parametrize("score", [O.SOFTMAX, O.SIGMOID])
@pytest.mark.parametrize("norm", [O.NORM_SELECTED, O.NORM_NONE])
def test_route_grouped_brute_force_gates_from_unbiased_scores(score, norm):
    rng = np.random.default_rng(62)
    for _ in range(150):
        n_group = int(rng.integers(1, 5)); gs = int(rng.integers(1, 4)); N = n_group * gs
        kg = int(rng.integers(1, n_group + 1))
        k = int(rng.integers(1, kg * gs + 1))
        m = int(rng.integers(1, gs + 1))
        z = rng.standard_normal((1, N)) * 1.5
        bias = rng.standard_normal(N) * 0.3
        for rule in (O.GROUP_MAX, O.GROUP_TOPM_SUM):
            S, g, p, q = O.route_grouped(z, k, n_group, kg, rule, m, score, norm, bias)
            # p straight from the definitions, token by token with math
            if score == O.SOFTMAX:
                ex = [math.exp(v) for v in z[0]]
                p_ref = [v / sum(ex) for v in ex]
            else:
                p_ref = [1 / (1 + math.exp(-v)) for v in z[0]]
            q_ref = [p_ref[i] + bias[i] for i in range(N)]
            S_bf, g_bf = _group_brute_force(q_ref, p_ref, k, n_group, kg, rule, m, norm)
            assert S[0].tolist() == S_bf
            np.testing.assert_allclose(g[0], g_bf, atol=1e-14, rtol=0)


def test_route_grouped_page2_example_through_route():
    """The page's two groups [0.90, 0.10 | 0.80, 0.79], top-2, one group kept,
    through route_grouped: sigmoid scores with logits chosen so that
    sigma(z) reproduces the printed scores, no bias. Group max keeps group A
    (gates 0.90/1.00, 0.10/1.00); the top-2 sum keeps group B (0.80/1.59,
    0.79/1.59)."""
    gd = load_golden("page2_group_limited_example.json")
    s = np.array(gd["scores"])
    z = np.log(s / (1 - s))[None]
    S, g, p, _ = O.route_grouped(z, gd["k"], 2, 1, O.GROUP_MAX, 2, O.SIGMOID, O.NORM_SELECTED)
    np.testing.assert_allclose(p[0], s, atol=1e-15)
    assert S[0].tolist() == [0, 1]
    np.testing.assert_allclose(g[0], [0.90, 0.10], atol=1e-12)
    S, g, _, _ = O.route_grouped(z, gd["k"], 2, 1, O.GROUP_TOPM_SUM, 2, O.SIGMOID, O.NORM_SELECTED)
    assert S[0].tolist() == [2, 3]
    np.testing.assert_allclose(g[0], [0.80 / 1.59, 0.79 / 1.59], atol=1e-12)
    # with a bias that lifts expert 3 above expert 2, slot order follows q
    # but the gates still come from the un-biased p
    S, g, _, q = O.route_grouped(z, gd["k"], 2, 1, O.GROUP_TOPM_SUM, 2, O.SIGMOID,
                                 O.NORM_SELECTED, np.array([0.0, 0.0, 0.0, 0.05]))
    assert S[0].tolist() == [3, 2]
    np.testing.assert_allclose(g[0], [0.79 / 1.59, 0.80 / 1.59], atol=1e-12)


def test_stats_sigmoid_brute_force_nonuniform():
    """Routing statistics of a sigmoid router on non-uniform logits against a
    token-by-token computation with math: P_i from sigma(z) divided by its
    per-token sum (the reading taken for a sigmoid router), f_i the share of
    the T*k pairs, L_bal = N sum f_i P_i ("MOE 专家选择与路由机制" §五),
    z-loss from the raw logits, entropy of the normalised scores."""
    rng = np.random.default_rng(63)
    T, N, k = 17, 6, 3
    z = rng.standard_normal((T, N)) * 1.7 + rng.standard_normal(N)[None] * 0.8
    bias = rng.standard_normal(N) * 0.2
    S, _, _, _ = O.route(z, k, O.SIGMOID, O.NORM_SELECTED, bias)
    st = O.routing_stats(z, S, O.SIGMOID, N)
    P = [0.0] * N; cnt = [0] * N; lz = 0.0; H = 0.0
    for t in range(T):
        sig = [1 / (1 + math.exp(-v)) for v in z[t]]
        tot = sum(sig)
        lz += math.log(sum(math.exp(v) for v in z[t])) ** 2
        for i in range(N):
            pi = sig[i] / tot
            P[i] += pi / T
            H -= pi * math.log(pi) / T
        for j in range(k):
            cnt[S[t, j]] += 1
    f = [c / (T * k) for c in cnt]
    np.testing.assert_allclose(st["P"], P, atol=1e-14)
    np.testing.assert_allclose(st["f"], f, atol=0)
    assert abs(st["L_bal"] - N * sum(a * b for a, b in zip(f, P))) < 1e-12
    assert abs(st["L_z"] - lz / T) < 1e-12
    assert abs(st["entropy"] - H) < 1e-12
    assert abs(sum(st["P"]) - 1.0) < 1e-12 and abs(sum(st["f"]) - 1.0) < 1e-15


# --------------------------------------- planted mistakes in the new pins ---
def test_mutation_swiglu_act_branches_swapped(monkeypatch):
    def bad_act(x, Wg, Wu):
        x = np.asarray(x, np.float64)
        return O.silu(x @ np.asarray(Wu).T) * (x @ np.asarray(Wg).T)
    _run_pins_expect_failure(monkeypatch, "swiglu_act", bad_act,
                             [test_swiglu_act_vs_library_and_closed_form])


def test_mutation_route_grouped_gates_from_biased_scores(monkeypatch):
    def bad_route_grouped(z, k, n_group, topk_group, group_score=O.GROUP_MAX, top_m=2,
                          score_kind=O.SOFTMAX, norm=O.NORM_SELECTED, sel_bias=None):
        p = O.scores(z, score_kind)
        q = p if sel_bias is None else p + np.asarray(sel_bias, dtype=np.float64)[None, :]
        S = O.select_topk_grouped(q, k, n_group, topk_group, group_score, top_m)
        return S, O.gates_from_scores(q, S, norm), p, q          # gates from q
    _run_pins_expect_failure(
        monkeypatch, "route_grouped", bad_route_grouped,
        [lambda: test_route_grouped_brute_force_gates_from_unbiased_scores(O.SIGMOID, O.NORM_SELECTED),
         test_route_grouped_page2_example_through_route])


def test_mutation_group_mask_zero_instead_of_minus_inf(monkeypatch):
    orig = O.select_topk
    def bad_grouped(q, k, n_group, topk_group, group_score=O.GROUP_MAX, top_m=2):
        q = np.asarray(q, dtype=np.float64)
        T, N = q.shape
        gs = N // n_group
        qg = q.reshape(T, n_group, gs)
        sg = qg.max(axis=-1) if group_score == O.GROUP_MAX else \
            -np.sort(-qg, axis=-1)[..., :top_m].sum(axis=-1)
        kept = orig(sg, topk_group)
        keep = np.zeros((T, n_group)); np.put_along_axis(keep, kept, 1.0, axis=-1)
        return orig((qg * keep[..., None]).reshape(T, N), k)     # masked to 0
    _run_pins_expect_failure(
        monkeypatch, "select_topk_grouped", bad_grouped,
        [test_grouped_masks_with_minus_infinity_not_zero,
         lambda: test_route_grouped_brute_force_gates_from_unbiased_scores(O.SIGMOID, O.NORM_SELECTED)])


def test_mutation_group_score_sum_of_all_instead_of_top_m(monkeypatch):
    orig = O.select_topk
    def bad_grouped(q, k, n_group, topk_group, group_score=O.GROUP_MAX, top_m=2):
        q = np.asarray(q, dtype=np.float64)
        T, N = q.shape
        gs = N // n_group
        qg = q.reshape(T, n_group, gs)
        sg = qg.max(axis=-1) if group_score == O.GROUP_MAX else qg.sum(axis=-1)   # all, not top-m
        kept = orig(sg, topk_group)
        mask = np.full((T, n_group), -np.inf); np.put_along_axis(mask, kept, 0.0, axis=-1)
        return orig((qg + mask[..., None]).reshape(T, N), k)
    _run_pins_expect_failure(
        monkeypatch, "select_topk_grouped", bad_grouped,
        [lambda: test_route_grouped_brute_force_gates_from_unbiased_scores(O.SOFTMAX, O.NORM_NONE)])


def test_mutation_sigmoid_stats_unnormalised(monkeypatch):
    def bad_probs(z, score_kind):
        return O.softmax(z) if score_kind == O.SOFTMAX else O.sigmoid(z)   # not divided by the sum
    _run_pins_expect_failure(monkeypatch, "router_probabilities", bad_probs,
                             [test_stats_sigmoid_brute_force_nonuniform])
