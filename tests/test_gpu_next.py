"""GPU parity of the rows beyond the core layer: routing side statistics,
group-limited top-k, capacity with token dropping and expert-choice routing,
each against the CPU oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import np_f, np_i
from oracle import moe_oracle as O
from top_routing_grouped_bias_b300 import api, synth
from top_routing_grouped_bias_b300.synth import Workload, to_f64

pytestmark = pytest.mark.gpu


def _route_logits(cfg, z, bias=None):
    dev = "cuda"
    ws = api.alloc_workspace(cfg, dev)
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    gate = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    api.moe_route(cfg, None, None, None, None if bias is None else bias.to(dev), z.to(dev), None,
                  idx, gate, ws)
    return idx, gate, ws


def _stats(cfg, z, idx, ws):
    out = torch.empty(3 + 2 * cfg.N, dtype=torch.float32, device="cuda")
    api.moe_route_stats(cfg, z, idx, out, ws)
    torch.cuda.synchronize()
    return out.cpu().double().numpy()


def _check_stats(got, ref, N):
    scal = np.array([ref["L_bal"], ref["L_z"], ref["entropy"]])
    np.testing.assert_allclose(got[:3], scal, rtol=5e-5, atol=1e-6)
    np.testing.assert_allclose(got[3:3 + N], ref["P"], rtol=5e-5, atol=1e-7)
    np.testing.assert_allclose(got[3 + N:], ref["f"], rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("T,N,k,score", [(3000, 8, 2, "softmax"), (1001, 256, 8, "sigmoid"),
                                         (257, 1024, 16, "softmax"), (64, 4, 1, "sigmoid")])
def test_route_stats_vs_oracle(cuda_lib, T, N, k, score):
    z = synth.random_logits(T, N, seed=T + N, std=2.0)
    cfg = api.make_config(T, 8, N, k, 8, score=score)
    idx, _, ws = _route_logits(cfg, z)
    got = _stats(cfg, z.cuda(), idx, ws)
    ref = O.routing_stats(to_f64(z), np_i(idx), score, N)
    _check_stats(got, ref, N)


def test_route_stats_deterministic(cuda_lib):
    """Fixed summation order: two calls give the same bits (T spans 40 blocks)."""
    T, N, k = 10000, 96, 4
    z = synth.random_logits(T, N, seed=7, std=2.0)
    cfg = api.make_config(T, 8, N, k, 8, score="softmax")
    idx, _, ws = _route_logits(cfg, z)
    a = _stats(cfg, z.cuda(), idx, ws)
    b = _stats(cfg, z.cuda(), idx, ws)
    assert (a == b).all()


def test_route_stats_uniform_closed_form(cuda_lib):
    T, N, k = 512, 16, 2
    z = torch.zeros((T, N), dtype=torch.float32)
    cfg = api.make_config(T, 8, N, k, 8)
    # balanced assignments: token t takes experts (2t, 2t+1) mod N
    idx = torch.tensor([[(2 * t) % N, (2 * t + 1) % N] for t in range(T)], dtype=torch.int32)
    ws = api.alloc_workspace(cfg, "cuda")
    got = _stats(cfg, z.cuda(), idx.cuda(), ws)
    assert abs(got[0] - 1.0) < 1e-5
    assert abs(got[1] - np.log(N) ** 2) < 1e-5
    assert abs(got[2] - np.log(N)) < 1e-5


@pytest.mark.parametrize("name", ["fine_grained_shared", "switch_top1"])
def test_route_stats_full_size(cuda_lib, name):
    w = synth.WORKLOADS[name]
    cfg = api.config_for(w)
    inp = synth.make_inputs(w, seed=0, device="cuda")
    ws = api.alloc_workspace(cfg, "cuda")
    logits = torch.empty((w.T, w.N), dtype=torch.float32, device="cuda")
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    api.moe_route(cfg, inp["h"], inp["W_r"], None, inp["sel_bias"], None, logits, idx, gate, ws)
    got = _stats(cfg, logits, idx, ws)
    ref = O.routing_stats(np_f(logits), np_i(idx), w.score, w.N)
    _check_stats(got, ref, w.N)
    print(f"{name}: L_bal {got[0]:.4f} L_z {got[1]:.4f} entropy {got[2]:.4f}")


# ------------------------------------------------------- group-limited top-k ---
def _route_grouped(cfg, grp, z=None, h=None, W_r=None, bias=None):
    dev = "cuda"
    ws = api.alloc_workspace(cfg, dev)
    logits = torch.empty((cfg.T, cfg.N), dtype=torch.float32, device=dev)
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    gate = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    api.moe_route_grouped(cfg, grp, h, W_r, None, None if bias is None else bias.to(dev),
                          None if z is None else z.to(dev), logits, idx, gate, ws)
    torch.cuda.synchronize()
    assert api.read_status(ws) == api.MOE_OK
    return logits, idx, gate


def test_grouped_page2_example(cuda_lib):
    """Scores [0.90, 0.10 | 0.80, 0.79] as sigmoid scores: group max keeps A,
    the top-2 sum keeps B (1.59 > 1.00)."""
    from conftest import load_golden
    g = load_golden("page2_group_limited_example.json")
    q = torch.tensor([g["scores"]], dtype=torch.float64)
    z = torch.log(q / (1 - q)).to(torch.float32)
    cfg = api.make_config(1, 8, 4, 2, 8, score="sigmoid")
    _, idx, _ = _route_grouped(cfg, api.make_group_config(2, 1, "max"), z=z)
    assert np_i(idx)[0].tolist() == [0, 1]
    _, idx, _ = _route_grouped(cfg, api.make_group_config(2, 1, "topm_sum", 2), z=z)
    assert np_i(idx)[0].tolist() == [2, 3]
    _, idx, _ = _route_grouped(cfg, api.make_group_config(2, 2, "max"), z=z)
    assert np_i(idx)[0].tolist() == [0, 2]


@pytest.mark.parametrize("N,k,G,kg,rule,m,score", [
    (64, 8, 8, 4, "topm_sum", 2, "sigmoid"), (64, 6, 8, 3, "max", 1, "softmax"),
    (256, 8, 8, 4, "topm_sum", 2, "sigmoid"), (32, 4, 32, 4, "max", 1, "softmax"),
    (60, 5, 6, 2, "topm_sum", 3, "softmax"),
    # every register-slot count of the selection kernel (1, 2, 4, 8, 16, 32
    # experts per lane), groups that are lane segments (size dividing 32, at
    # most top-2 summed) and groups that are not, expert counts that leave a
    # partial 32-expert chunk
    (24, 4, 3, 2, "topm_sum", 2, "softmax"), (48, 5, 6, 3, "max", 1, "sigmoid"),
    (96, 6, 8, 4, "topm_sum", 2, "sigmoid"), (128, 4, 16, 4, "topm_sum", 1, "softmax"),
    (200, 8, 8, 2, "max", 1, "softmax"), (256, 8, 32, 4, "topm_sum", 2, "softmax"),
    (512, 8, 16, 4, "topm_sum", 2, "sigmoid"), (768, 12, 8, 3, "topm_sum", 2, "softmax"),
    (1024, 16, 32, 8, "max", 1, "sigmoid")])
def test_grouped_given_logits_exact(cuda_lib, N, k, G, kg, rule, m, score):
    T = 700
    z = synth.random_logits(T, N, seed=N * G + k, std=1.5, ties=True)
    cfg = api.make_config(T, 8, N, k, 8, score=score)
    _, idx, gate = _route_grouped(cfg, api.make_group_config(G, kg, rule, m), z=z)
    rule_o = O.GROUP_MAX if rule == "max" else O.GROUP_TOPM_SUM
    S, g, _, _ = O.route_grouped(to_f64(z), k, G, kg, rule_o, m, score, "selected")
    assert (np_i(idx) == S).all()
    np.testing.assert_allclose(np_f(gate), g, atol=1e-6, rtol=0)


def test_grouped_from_hidden_states_with_bias(cuda_lib):
    """bf16 routing from h: logits on the tensor cores, then the grouped
    selection (DeepSeek-V3-like: 8 groups, keep 4, top-2 sums, sigmoid + bias)."""
    w = Workload("grouped", T=500, d=256, N=64, F=64, k=8, score="sigmoid", bias_zipf_s=1.1,
                 bias_beta=0.3)
    cfg = api.config_for(w)
    inp = synth.make_inputs(w, seed=2, device="cuda")
    logits, idx, gate = _route_grouped(cfg, api.make_group_config(8, 4, "topm_sum", 2),
                                       h=inp["h"], W_r=inp["W_r"], bias=inp["sel_bias"])
    z = np_f(logits)
    from gpu_helpers import logit_bound
    assert (np.abs(z - O.router_logits(to_f64(inp["h"]), to_f64(inp["W_r"])))
            <= logit_bound(to_f64(inp["h"]), to_f64(inp["W_r"]))).all()
    S, g, _, _ = O.route_grouped(z, w.k, 8, 4, O.GROUP_TOPM_SUM, 2, w.score, w.norm,
                                 to_f64(inp["sel_bias"]))
    same = (np_i(idx) == S).all(axis=1)
    # fp32 group sums and scores may flip near-ties; everything else is exact
    assert same.mean() >= 0.99, same.mean()
    np.testing.assert_allclose(np_f(gate)[same], g[same], atol=1e-6, rtol=0)


@pytest.mark.parametrize("N,k,G,kg,rule,m", [(1024, 8, 32, 8, "max", 1),
                                               (96, 6, 8, 4, "topm_sum", 2),
                                               (256, 8, 8, 4, "topm_sum", 2),
                                               (40, 4, 5, 2, "topm_sum", 2)])
def test_grouped_given_logits_with_bias(cuda_lib, N, k, G, kg, rule, m):
    """Sigmoid + selection bias with groups, from given logits: the group
    pass and the selection run on q = p + bias."""
    T = 600
    z = synth.random_logits(T, N, seed=N + G, std=1.5)
    bias = synth.zipf_bias(torch.Generator().manual_seed(N), N, 1.1, 0.3, "cpu")
    cfg = api.make_config(T, 8, N, k, 8, score="sigmoid")
    _, idx, gate = _route_grouped(cfg, api.make_group_config(G, kg, rule, m), z=z, bias=bias)
    rule_o = O.GROUP_MAX if rule == "max" else O.GROUP_TOPM_SUM
    S, g, _, _ = O.route_grouped(to_f64(z), k, G, kg, rule_o, m, "sigmoid", "selected",
                                 to_f64(bias))
    same = (np_i(idx) == S).all(axis=1)
    # fp32 scores and group sums may flip near-ties; everything else is exact
    assert same.mean() >= 0.99, same.mean()
    np.testing.assert_allclose(np_f(gate)[same], g[same], atol=1e-6, rtol=0)


def test_grouped_rejects_too_few_candidates(cuda_lib):
    import ctypes
    lib = api.load()
    fake = ctypes.c_void_p(1 << 20)
    cfg = api.make_config(16, 8, 8, 5, 8)
    grp = api.make_group_config(4, 2, "max")          # 2 groups x 2 experts = 4 < 5
    assert lib.moe_route_grouped(ctypes.byref(cfg), ctypes.byref(grp), None, None, None, None,
                                 fake, None, fake, fake, None, 0, None) == api.MOE_ERR_INVALID_ARG


# ------------------------------------------------------------- capacity ---
def _dispatch_cap(cfg, C, idx, h):
    dev = "cuda"
    R = cfg.T * cfg.k
    ws = api.alloc_workspace(cfg, dev)
    out = dict(counts=torch.empty(cfg.N, dtype=torch.int32, device=dev),
               offsets=torch.empty(cfg.N + 1, dtype=torch.int32, device=dev),
               row_token=torch.full((R,), -7, dtype=torch.int32, device=dev),
               inv=torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev),
               x_disp=torch.zeros((R, cfg.d), dtype=h.dtype, device=dev))
    api.moe_dispatch_capacity(cfg, C, h.to(dev), idx.to(dev), out["counts"], out["offsets"],
                              out["row_token"], out["inv"], out["x_disp"], ws)
    torch.cuda.synchronize()
    assert api.read_status(ws) == api.MOE_OK
    return out


def test_capacity_page1_table(cuda_lib):
    from conftest import load_golden
    gd = load_golden("page1_dispatch_table.json")
    idx = torch.tensor([[e for e, _ in row] for row in gd["choices"]], dtype=torch.int32)
    h = torch.arange(32, dtype=torch.float32).reshape(4, 8).to(torch.bfloat16)
    r = _dispatch_cap(api.make_config(4, 8, 4, 2, 8), 2, idx, h)
    assert np_i(r["counts"]).tolist() == [2, 2, 2, 1]
    kept = int(np_i(r["offsets"])[-1])
    assert np_i(r["row_token"])[:kept].tolist() == [0, 2, 1, 3, 0, 1, 2]
    assert np_i(r["inv"])[3].tolist() == [-1, 3]


@pytest.mark.parametrize("T,N,k,C", [(3000, 8, 2, 0), (3000, 8, 2, 700), (3000, 8, 2, 10 ** 6),
                                     (1000, 128, 8, 50), (513, 64, 1, 6),
                                     # the multi-block scan and the warp-per-token gather
                                     (9000, 16, 3, 1200), (20000, 64, 2, 500)])
def test_capacity_dispatch_random_exact(cuda_lib, T, N, k, C):
    gen = torch.Generator().manual_seed(T + C)
    # skewed routing so that some experts overflow
    w = torch.arange(N, 0, -1, dtype=torch.float64) ** 2
    idx = torch.stack([torch.multinomial(w, k, replacement=False, generator=gen)
                       for _ in range(T)]).to(torch.int32)
    h = torch.randn((T, 16), generator=gen).to(torch.bfloat16)
    r = _dispatch_cap(api.make_config(T, 16, N, k, 8), C, idx, h)
    counts, offsets, row_token, inv = O.dispatch_capacity(idx.numpy(), N, C)
    assert np_i(r["counts"]).tolist() == counts.tolist()
    assert np_i(r["offsets"]).tolist() == offsets.tolist()
    kept = int(offsets[-1])
    assert np_i(r["row_token"])[:kept].tolist() == row_token.tolist()
    assert (np_i(r["inv"]) == inv).all()
    assert torch.equal(r["x_disp"][:kept].cpu(), h[torch.from_numpy(row_token)])


@pytest.mark.parametrize("cf", [0.5, 1.0, 1.25])
def test_capacity_layer_vs_oracle(cuda_lib, cf):
    # W_down at half the named workloads' deviation keeps outputs of order one,
    # where the stated 2e-2 absolute bound is reachable after bf16 roundings
    w = Workload("cap", T=700, d=128, N=8, F=128, k=2, F_sh=128, score="sigmoid",
                 bias_zipf_s=1.1, bias_beta=0.5, wd_scale=0.5)
    cfg = api.config_for(w)
    C = api.expert_capacity(w.T, w.k, w.N, cf)
    inp = synth.make_inputs(w, seed=6, device="cpu")
    gin = {k_: (v.cuda() if isinstance(v, torch.Tensor) else v) for k_, v in inp.items()}
    ws = api.alloc_workspace(cfg, "cuda")
    outs = api.alloc_outputs(cfg, "cuda", torch.bfloat16)
    api.forward_capacity(cfg, C, gin, outs, ws)
    torch.cuda.synchronize()
    assert api.read_status(ws) == api.MOE_OK
    o = {k_: to_f64(v) for k_, v in inp.items()}
    idx = np_i(outs["idx"])
    z = O.router_logits(o["h"], o["W_r"])
    g = O.gates_from_scores(O.scores(z, w.score), idx, w.norm)
    counts, offsets, row_token, inv = O.dispatch_capacity(idx, w.N, C)
    assert np_i(outs["counts"]).tolist() == counts.tolist()
    y_rows = O.expert_rows(o["h"][row_token], offsets, o["W_gate"], o["W_up"], o["W_down"])
    ysh = O.swiglu_expert(o["h"], o["Ws_gate"], o["Ws_up"], o["Ws_down"])
    ref = ysh.copy()
    for t in range(w.T):
        for j in range(w.k):
            if inv[t, j] >= 0:
                ref[t] += g[t, j] * y_rows[inv[t, j]]
    from gpu_helpers import BF16_TOL, assert_close_tol
    assert_close_tol(np_f(outs["out"]), ref, BF16_TOL, f"capacity cf={cf}")
    dropped = int((inv < 0).sum())
    print(f"cf={cf}: C={C}, dropped {dropped} of {w.T * w.k} pairs")
    if cf < 1:
        assert dropped > 0


def test_capacity_unlimited_equals_dropless_forward(cuda_lib):
    w = Workload("cap2", T=400, d=128, N=8, F=128, k=2)
    cfg = api.config_for(w)
    inp = {k_: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k_, v in synth.make_inputs(w, seed=7).items()}
    ws = api.alloc_workspace(cfg, "cuda")
    a = api.alloc_outputs(cfg, "cuda", torch.bfloat16)
    b = api.alloc_outputs(cfg, "cuda", torch.bfloat16)
    api.forward(cfg, inp, a, ws)
    api.forward_capacity(cfg, w.T * w.k, inp, b, ws)
    torch.cuda.synchronize()
    for key in ("out", "idx", "gate", "counts"):
        assert torch.equal(a[key], b[key])


# --------------------------------------------------------- expert choice ---
def _ec_run(cfg, C, inp):
    dev = "cuda"
    ws = api.alloc_workspace(cfg, dev)
    tdt = torch.float32 if cfg.dtype == api.DTYPES["f32"] else torch.bfloat16
    out = torch.empty((cfg.T, cfg.d), dtype=tdt, device=dev)
    logits = torch.empty((cfg.T, cfg.N), dtype=torch.float32, device=dev)
    tokens = torch.full((cfg.N, max(C, 1)), -1, dtype=torch.int32, device=dev)
    gates = torch.zeros((cfg.N, max(C, 1)), dtype=torch.float32, device=dev)
    gin = {k_: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k_, v in inp.items()}
    api.forward_expert_choice(cfg, C, gin, out, ws, logits, tokens, gates)
    torch.cuda.synchronize()
    assert api.read_status(ws) == api.MOE_OK
    return out, logits, tokens[:, :C], gates[:, :C]


def _ec_check_selection(z64, score, C, tokens, gates):
    """Each expert's picked set equals the oracle's, except where the oracle's
    C-th and (C+1)-th scores are within what fp32 scoring can move."""
    p = O.scores(z64, score)
    ref_tokens, _, _ = O.expert_choice(z64, C, score)
    amb = 0
    for e in range(p.shape[1]):
        got = np_i(tokens)[e]
        assert (np.diff(got) > 0).all(), "picked tokens must be ascending and distinct"
        col = -np.sort(-p[:, e])
        gap = col[C - 1] - col[C] if C < p.shape[0] else np.inf
        if gap > 4e-6:
            assert set(got.tolist()) == set(ref_tokens[e].tolist()), f"expert {e}"
        else:
            amb += 1
            assert (p[got, e] >= col[C - 1] - 4e-6).all()
        np.testing.assert_allclose(np_f(gates)[e], p[got, e], atol=1e-6, rtol=0)
    return amb


@pytest.mark.parametrize("score,shared,T,N,k,dtype", [
    ("softmax", False, 700, 8, 2, "bf16"), ("sigmoid", True, 700, 8, 2, "bf16"),
    # fp32 with a ragged expert count; 1024 experts (the combine's largest
    # per-warp choice list)
    ("sigmoid", True, 600, 300, 4, "f32"), ("sigmoid", False, 512, 1024, 8, "bf16")])
def test_expert_choice_layer_vs_oracle(cuda_lib, score, shared, T, N, k, dtype):
    w = Workload("ec", T=T, d=128, N=N, F=128, k=k, F_sh=128 if shared else 0, score=score,
                 dtype=dtype, wd_scale=0.5 if dtype == "bf16" else 1.0)
    cfg = api.config_for(w)
    C = w.T * w.k // w.N
    inp = synth.make_inputs(w, seed=8, device="cpu")
    out, logits, tokens, gates = _ec_run(cfg, C, inp)
    z = np_f(logits)
    o = {k_: to_f64(v) for k_, v in inp.items()}
    amb = _ec_check_selection(z, score, C, tokens, gates)
    assert amb <= max(1, N // 100)   # boundaries within fp32 reach, validated above
    # layer output with the GPU's (validated) picks, oracle fp64 scores and experts
    p = O.scores(O.router_logits(o["h"], o["W_r"]), score)
    ref = np.zeros((w.T, w.d)) if not shared else O.swiglu_expert(o["h"], o["Ws_gate"],
                                                                  o["Ws_up"], o["Ws_down"])
    tk = np_i(tokens)
    for e in range(w.N):
        ye = O.swiglu_expert(o["h"][tk[e]], o["W_gate"][e], o["W_up"][e], o["W_down"][e])
        ref[tk[e]] += p[tk[e], e][:, None] * ye
    from gpu_helpers import assert_close_tol, out_tol
    assert_close_tol(np_f(out), ref, out_tol(w), "expert choice")


def test_expert_choice_ties_and_empty(cuda_lib):
    """Duplicated hidden rows give bitwise-equal scores: the lower token index
    is picked first. C = 0 leaves only the shared expert."""
    w = Workload("ec_ties", T=64, d=64, N=4, F=64, k=1, F_sh=64)
    cfg = api.config_for(w)
    inp = synth.make_inputs(w, seed=9, device="cpu")
    inp["h"][1::2] = inp["h"][0::2]                 # tokens 2i and 2i+1 identical
    C = 16
    out, logits, tokens, gates = _ec_run(cfg, C, inp)
    z = np_f(logits)
    ref_tokens, _, _ = O.expert_choice(z, C, w.score)
    assert (np_i(tokens) == ref_tokens).all()
    out0, _, _, _ = _ec_run(cfg, 0, inp)
    o = {k_: to_f64(v) for k_, v in inp.items()}
    from gpu_helpers import BF16_TOL, assert_close_tol
    assert_close_tol(np_f(out0), O.swiglu_expert(o["h"], o["Ws_gate"], o["Ws_up"], o["Ws_down"]),
                     BF16_TOL, "C = 0")


def test_expert_choice_switch_sized(cuda_lib):
    """Switch-sized batch (T = 65536, N = 128, d = 2048): every expert takes
    exactly T/N tokens; picks and gates checked on every expert."""
    w = synth.WORKLOADS["switch_top1"]
    cfg = api.config_for(w)
    C = w.T * w.k // w.N
    inp = synth.make_inputs(w, seed=0, device="cuda")
    out, logits, tokens, gates = _ec_run(cfg, C, inp)
    amb = _ec_check_selection(np_f(logits), w.score, C, tokens, gates)
    print(f"expert choice switch-sized: {amb} experts with a boundary within fp32 reach")
    assert torch.isfinite(out.float()).all()
