"""Parity at the five named workloads' full sizes, in the launch configuration
the benchmark times (one moe_forward). Routing, gates and dispatch are checked
on every token; expert rows on every expert that received rows (its first,
last and random rows); the combine on 512 sampled tokens; the layer output on
512 tokens (all of them on the smaller batches) stratified so that every
expert with a nonzero count appears, the oracle batching the sampled tokens
expert by expert. Inputs are drawn on the device from a seeded generator and
copied to the host for the oracle."""
import gc

import numpy as np
import pytest
import torch

from gpu_helpers import (U32, assert_close_tol, check_selection, e2e_selection_check,
                         logit_bound, max_ambiguous, np_f, np_i, oracle_gates_from_logits,
                         out_tol, run_forward, run_staged, selection_scores)
from oracle import moe_oracle as O
from top_routing_grouped_bias_b300 import api, synth
from top_routing_grouped_bias_b300.synth import to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

FULL = ["tiny_fp32", "mixtral_prefill", "mixtral_decode", "fine_grained_shared", "switch_top1"]


def stratified_tokens(row_token, offsets, T, n, rng):
    """Up to n tokens: one random token from every expert's bucket (so that
    every expert with a nonzero count appears), then random further tokens;
    all T tokens when T <= n. Sorted."""
    if T <= n:
        return np.arange(T)
    pick = set()
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0 and len(pick) < n:
            pick.add(int(row_token[rng.integers(r0, r1)]))
    rest = rng.permutation(T)
    i = 0
    while len(pick) < n:
        pick.add(int(rest[i]))
        i += 1
    return np.array(sorted(pick))


def expert_weights(inp, e):
    return to_f64(inp["W_gate"][e]), to_f64(inp["W_up"][e]), to_f64(inp["W_down"][e])


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(cuda_lib, name):
    w = synth.WORKLOADS[name]
    cfg = api.config_for(w)
    rng = np.random.default_rng(0)
    inp = synth.make_inputs(w, seed=0, device="cuda")
    r = run_forward(cfg, inp)
    s = run_staged(cfg, inp)
    for key in ("idx", "gate", "logits", "counts"):
        assert torch.equal(r[key], s[key]), f"{key}: forward differs from the stages"
    if w.k == 1 and w.F_sh == 0:
        # moe_forward fuses the top-1 combine into the down pass: it scales the
        # fp32 accumulator before the single rounding, the stages round y
        # first; the two differ by at most that extra rounding
        a, b = np_f(r["out"]), np_f(s["out"])
        assert (np.abs(a - b) <= 2.0 ** -7 * np.abs(b) + 1e-6).all(), "fused top-1 combine"
    else:
        assert torch.equal(r["out"], s["out"]), "out: forward differs from the stages"

    # ---- routing on every token ----
    h64 = to_f64(inp["h"])
    Wr64 = to_f64(inp["W_r"])
    bias = to_f64(inp["sel_bias"])
    z_ref = O.router_logits(h64, Wr64)
    z_gpu = np_f(r["logits"])
    bound = logit_bound(h64, Wr64)
    assert (np.abs(z_gpu - z_ref) <= bound).all(), "logits beyond the fp32 summation bound"
    idx = np_i(r["idx"])
    delta_given = 0.0 if bias is None else 4e-6
    check_selection(idx, selection_scores(z_gpu, w.score, bias), w.k, delta_given, "given logits")
    n_amb = e2e_selection_check(idx, z_ref, z_gpu, w.score, bias, w.k, "end to end")
    print(f"{name}: {n_amb} of {w.T} tokens within the logit-error margin of a tie")
    assert n_amb <= max_ambiguous(w.T)
    g_ref = oracle_gates_from_logits(z_gpu, idx, w.score, w.norm)
    np.testing.assert_allclose(np_f(r["gate"]), g_ref, atol=1e-6, rtol=0)
    del z_ref, bound

    # ---- dispatch on every pair ----
    counts, offsets, row_token, inv = O.dispatch(idx, w.N)
    assert np_i(s["counts"]).tolist() == counts.tolist()
    assert np_i(s["offsets"]).tolist() == offsets.tolist()
    assert np_i(s["row_token"]).tolist() == row_token.tolist()
    assert (np_i(s["inv"]) == inv).all()
    rt_dev = s["row_token"].long()
    assert torch.equal(s["x_disp"], inp["h"].index_select(0, rt_dev))
    if w.bias_zipf_s is not None:
        print(f"{name}: {int((counts == 0).sum())} experts with no tokens, max load {counts.max()}")
        assert (counts == 0).sum() >= 1

    if w.F_sh > 0:
        toks = rng.choice(w.T, size=64, replace=False)
        sh = (to_f64(inp["Ws_gate"]), to_f64(inp["Ws_up"]), to_f64(inp["Ws_down"]))
        assert_close_tol(np_f(s["y_sh"][torch.from_numpy(toks).cuda()]),
                         O.swiglu_expert(h64[toks], *sh), out_tol(w), f"{name} y_shared")

    # ---- combine on sampled tokens: one rounding of the GPU's own terms ----
    toks = np.sort(rng.choice(w.T, size=min(w.T, 512), replace=False))
    inv_s = inv[toks]
    flat = np.unique(inv_s.reshape(-1))
    remap = {int(v): i for i, v in enumerate(flat)}
    y_s = np_f(s["y_rows"][torch.from_numpy(flat).cuda()])
    inv_local = np.vectorize(remap.get)(inv_s)
    g_s = np_f(s["gate"])[toks]
    ysh_s = None if w.F_sh == 0 else np_f(s["y_sh"][torch.from_numpy(toks).cuda()])
    ref = O.combine(y_s, inv_local, g_s, ysh_s)
    mag = O.combine(np.abs(y_s), inv_local, np.abs(g_s), None if ysh_s is None else np.abs(ysh_s))
    E = (w.k + 1) * U32 * mag
    rnd = 2 * U32 if w.dtype == "f32" else 2.0 ** -8
    got = np_f(s["out"][torch.from_numpy(toks).cuda()])
    assert (np.abs(got - ref) <= rnd * (np.abs(ref) + E) + E).all(), "combine beyond one rounding"

    # ---- every touched expert's rows, and the whole layer on 512 stratified
    # tokens: oracle in fp64 with the GPU's (validated) selection, the
    # sampled tokens batched expert by expert with each expert's weights
    # copied once ----
    toks = stratified_tokens(row_token, offsets, w.T, 512, rng)
    assert set(np.unique(idx[toks]).tolist()) == set(np.nonzero(counts)[0].tolist())
    z_t = O.router_logits(h64[toks], Wr64)
    g_t = O.gates_from_scores(O.scores(z_t, w.score), idx[toks], w.norm)
    y_ref = np.zeros((len(toks), w.d))
    if w.F_sh > 0:
        y_ref += O.swiglu_expert(h64[toks], to_f64(inp["Ws_gate"]), to_f64(inp["Ws_up"]),
                                 to_f64(inp["Ws_down"]))
    worst_rows = 0.0
    for e in np.nonzero(counts)[0]:
        e = int(e)
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        rows = np.unique(np.concatenate([np.arange(r0, min(r1, r0 + 4)),
                                         np.arange(max(r0, r1 - 4), r1),
                                         rng.integers(r0, r1, size=min(8, r1 - r0))]))
        ti, sj = np.nonzero(idx[toks] == e)
        Wg, Wu, Wd = expert_weights(inp, e)
        y_e = O.swiglu_expert(np.concatenate([h64[row_token[rows]], h64[toks][ti]]), Wg, Wu, Wd)
        mx, _ = assert_close_tol(np_f(s["y_rows"][torch.from_numpy(rows).cuda()]), y_e[:len(rows)],
                                 out_tol(w), f"{name} y_rows expert {e}")
        worst_rows = max(worst_rows, mx)
        y_ref[ti] += g_t[ti, sj][:, None] * y_e[len(rows):]
        del Wg, Wu, Wd
    got = np_f(r["out"][torch.from_numpy(toks).cuda()])
    mx, rl = assert_close_tol(got, y_ref, out_tol(w), f"{name} layer output")
    print(f"{name}: expert rows of {int((counts > 0).sum())} experts, max-abs {worst_rows:.3e}; "
          f"layer output max-abs {mx:.3e} rel-L2 {rl:.3e} on {len(toks)} tokens")
    del inp, r, s
    gc.collect()
    torch.cuda.empty_cache()


def test_timeout_status_path(cuda_lib):
    """A bounded wait that nothing satisfies reports MOE_ERR_TIMEOUT and the
    context stays usable."""
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    api.selftest_wait_timeout(20_000_000, ws)       # 20 ms budget
    assert api.read_status(ws) == api.MOE_ERR_TIMEOUT
    assert api.read_status(ws) == api.MOE_OK        # cleared by the read
    w = synth.Workload("after_timeout", T=64, d=64, N=4, F=64, k=2)
    r = run_forward(api.config_for(w), {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
                                        for k, v in synth.make_inputs(w).items()})
    assert torch.isfinite(r["out"].float()).all()
