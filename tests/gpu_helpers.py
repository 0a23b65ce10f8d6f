"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
(stage by stage or as one moe_forward), and compare with the CPU oracle.

Tolerances (derived in the design notes):
* indices, counts, offsets, permutation: bit-exact; routing decisions within
  a stated margin of a tie are "ambiguous" and checked for validity instead;
* gates: 1e-6 absolute against the oracle fed the GPU's own logits;
* logits: |z_gpu - z| <= d * 2^-24 * sum_i |h_i W_i| + 1e-6 (fp32 summation of
  exact bf16 products, any order);
* combine: one rounding to the output dtype of an fp32 sum with error E:
  |out - ref| <= 2^-8 (|ref| + E) + E (bf16), ref = the oracle's combine of
  the GPU's own y_rows and gates;
* layer output and expert rows: bf16 max-abs <= 2e-2 and rel-L2 <= 5e-3;
  fp32 (tf32 tensor cores) max-abs <= 1e-2 and rel-L2 <= 2e-3, on every case;
* end-to-end selection: at most max_ambiguous(T) tokens may sit within the
  logit-error margin of a tie (each still checked for validity).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O
from top_routing_grouped_bias_b300 import api
from top_routing_grouped_bias_b300.synth import to_f64

U32 = 2.0 ** -24
BF16_TOL = dict(max_abs=2e-2, rel_l2=5e-3)
F32_TOL = dict(max_abs=1e-2, rel_l2=2e-3)


def max_ambiguous(T: int) -> int:
    """Cap on tokens with a top-(k+1) gap inside its per-gap margin (twice what
    the two experts' own logit errors can move it): 3, or one token in 500.
    Measured with the per-gap margins: 0 of 4096 (Mixtral-shaped prefill),
    4 of 65536 (Switch top-1), 13 of 8192 (fine-grained: sigmoid scores plus a
    selection bias put many of 256 experts in a narrow band around the 8th).
    Every such token is still checked for a valid choice within its margin."""
    return max(3, T // 500)


def out_tol(w):
    return F32_TOL if w.dtype == "f32" else BF16_TOL


def assert_close_tol(got, ref, tol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if got.size == 0:
        return 0.0, 0.0
    err = np.abs(got - ref)
    max_abs = float(err.max())
    rel_l2 = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    assert max_abs <= tol["max_abs"], f"{what}: max-abs {max_abs:.3e} > {tol['max_abs']}"
    assert rel_l2 <= tol["rel_l2"], f"{what}: rel-L2 {rel_l2:.3e} > {tol['rel_l2']}"
    return max_abs, rel_l2


def np_i(t):
    return t.detach().cpu().numpy().astype(np.int64)


def np_f(t):
    return to_f64(t)


# ------------------------------------------------------------- GPU runs ---
def gpu_inputs(inp: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_staged(cfg, inp: dict, logits_in=None, stream=None) -> dict:
    """route -> dispatch -> expert FFN -> combine, each through its entry point."""
    dev = inp["h"].device if inp.get("h") is not None else logits_in.device
    T, d, N, k, F, Fs = cfg.T, cfg.d, cfg.N, cfg.k, cfg.ffn, cfg.ffn_shared
    tdt = torch.float32 if cfg.dtype == api.DTYPES["f32"] else torch.bfloat16
    R = T * k
    ws = api.alloc_workspace(cfg, dev)
    r = {}
    r["logits"] = torch.empty((T, N), dtype=torch.float32, device=dev)
    r["idx"] = torch.empty((T, k), dtype=torch.int32, device=dev)
    r["gate"] = torch.empty((T, k), dtype=torch.float32, device=dev)
    h = inp.get("h") if logits_in is None else None
    api.moe_route(cfg, h, inp.get("W_r"), inp.get("b_r"), inp.get("sel_bias"), logits_in,
                  r["logits"], r["idx"], r["gate"], ws, stream)
    if logits_in is not None:
        torch.cuda.synchronize()
        return r
    r["counts"] = torch.empty((N,), dtype=torch.int32, device=dev)
    r["offsets"] = torch.empty((N + 1,), dtype=torch.int32, device=dev)
    r["row_token"] = torch.empty((R,), dtype=torch.int32, device=dev)
    r["inv"] = torch.empty((T, k), dtype=torch.int32, device=dev)
    r["x_disp"] = torch.empty((R, d), dtype=tdt, device=dev)
    api.moe_dispatch(cfg, inp["h"], r["idx"], r["counts"], r["offsets"], r["row_token"], r["inv"],
                     r["x_disp"], ws, stream)
    r["y_rows"] = torch.empty((R, d), dtype=tdt, device=dev)
    r["y_sh"] = torch.empty((T, d), dtype=tdt, device=dev) if Fs > 0 else None
    api.moe_expert_ffn(cfg, r["x_disp"], r["offsets"], inp["W_gate"], inp["W_up"], inp["W_down"],
                       r["y_rows"], inp["h"], inp.get("Ws_gate"), inp.get("Ws_up"),
                       inp.get("Ws_down"), r["y_sh"], ws, stream)
    r["out"] = torch.empty((T, d), dtype=tdt, device=dev)
    api.moe_combine(cfg, r["y_rows"], r["inv"], r["gate"], r["y_sh"], r["out"], stream)
    torch.cuda.synchronize()
    assert api.read_status(ws) == api.MOE_OK
    return r


def run_forward(cfg, inp: dict, stream=None) -> dict:
    dev = inp["h"].device
    tdt = torch.float32 if cfg.dtype == api.DTYPES["f32"] else torch.bfloat16
    ws = api.alloc_workspace(cfg, dev)
    outs = api.alloc_outputs(cfg, dev, tdt)
    api.forward(cfg, inp, outs, ws, stream)
    torch.cuda.synchronize()
    assert api.read_status(ws) == api.MOE_OK
    return dict(outs)


# ---------------------------------------------------------- comparisons ---
def logit_bound(h64, W64):
    """Per-(token, expert) bound on |z_fp32 - z_exact| for fp32 summation."""
    d = h64.shape[1]
    return d * U32 * (np.abs(h64) @ np.abs(W64).T) + 1e-6


def selection_scores(z, w_score, bias):
    p = O.scores(z, w_score)
    return p if bias is None else p + bias[None, :]


def check_selection(idx_gpu, q_ref, k, delta, what=""):
    """GPU indices vs the oracle's selection on scores q_ref [T,N].

    Tokens whose adjacent gaps among the k+1 best scores are all >= delta
    must match exactly (set and slot order). Tokens whose set boundary
    (k-th vs (k+1)-th) gap is >= delta must match as a set. The rest must be a
    valid choice within delta. Returns the number of ambiguous tokens."""
    T, N = q_ref.shape
    delta = np.broadcast_to(np.asarray(delta, dtype=np.float64), (T,))
    S_ref = O.select_topk(q_ref, k)
    qs = -np.sort(-q_ref, axis=1)
    top = qs[:, :min(k + 1, N)]
    gaps = top[:, :-1] - top[:, 1:] if top.shape[1] > 1 else np.full((T, 1), np.inf)
    order_amb = (gaps[:, :k].min(axis=1) < delta) if gaps.shape[1] else np.zeros(T, bool)
    set_amb = (gaps[:, k - 1] < delta) if k < N else np.zeros(T, bool)
    if not delta.any():
        order_amb[:] = False
        set_amb[:] = False
    exact = ~order_amb
    bad = np.nonzero((idx_gpu[exact] != S_ref[exact]).any(axis=1))[0]
    assert bad.size == 0, f"{what}: {bad.size} tokens differ, e.g. t={np.nonzero(exact)[0][bad[0]]}"
    for t in np.nonzero(order_amb)[0]:
        sel = idx_gpu[t]
        assert len(set(sel.tolist())) == k and (sel >= 0).all() and (sel < N).all()
        if not set_amb[t]:
            assert set(sel.tolist()) == set(S_ref[t].tolist()), f"{what}: set differs at t={t}"
        # each chosen expert is at least as good as the k-th best, up to delta
        assert (q_ref[t, sel] >= qs[t, k - 1] - delta[t]).all(), f"{what}: invalid choice at t={t}"
        # slots descend up to delta
        assert (np.diff(q_ref[t, sel]) <= delta[t]).all(), f"{what}: slot order at t={t}"
    return int(order_amb.sum())


def check_selection_gaps(idx_gpu, q_ref, k, err, what=""):
    """GPU indices vs the oracle's selection on scores q_ref [T,N], with a
    per-expert bound err [T,N] on how far the GPU's selection score of that
    expert can lie from q_ref. A gap between the oracle's adjacent i-th and
    (i+1)-th best experts a, b is ambiguous when it is below twice
    err[a] + err[b] (only there can the GPU's order differ). Tokens with no
    ambiguous gap among the k+1 best must match exactly (set and slot order);
    tokens whose k-th gap is clear must match as a set; the rest must be a
    valid choice within their largest margin. Returns the ambiguous count."""
    T, N = q_ref.shape
    S_ref = O.select_topk(q_ref, min(k + 1, N))
    qs = np.take_along_axis(q_ref, S_ref, axis=1)
    es = np.take_along_axis(err, S_ref, axis=1)
    if S_ref.shape[1] > 1:
        gaps = qs[:, :-1] - qs[:, 1:]
        margins = 2.0 * (es[:, :-1] + es[:, 1:]) + 1e-12
        amb_gap = gaps < margins
        order_amb = amb_gap[:, :k].any(axis=1)
        set_amb = amb_gap[:, k - 1] if k < N else np.zeros(T, bool)
        delta = margins[:, :k].max(axis=1)
    else:
        order_amb = set_amb = np.zeros(T, bool)
        delta = np.zeros(T)
    S_k = S_ref[:, :k]
    exact = ~order_amb
    bad = np.nonzero((idx_gpu[exact] != S_k[exact]).any(axis=1))[0]
    assert bad.size == 0, f"{what}: {bad.size} tokens differ, e.g. t={np.nonzero(exact)[0][bad[0]]}"
    for t in np.nonzero(order_amb)[0]:
        sel = idx_gpu[t]
        assert len(set(sel.tolist())) == k and (sel >= 0).all() and (sel < N).all()
        if not set_amb[t]:
            assert set(sel.tolist()) == set(S_k[t].tolist()), f"{what}: set differs at t={t}"
        assert (q_ref[t, sel] >= qs[t, k - 1] - delta[t]).all(), f"{what}: invalid choice at t={t}"
        assert (np.diff(q_ref[t, sel]) <= delta[t]).all(), f"{what}: slot order at t={t}"
    return int(order_amb.sum())


def e2e_selection_check(idx_gpu, z_ref, z_gpu, w_score, bias, k, what=""):
    """End-to-end selection: GPU indices against the oracle's selection from
    exact logits.

    The GPU selects exactly on its own fp32 logits (checked separately), so a
    decision can differ from the oracle's only where the logit error (z_gpu -
    z_ref, itself checked against the fp32 summation bound) moves a gap among
    the k+1 best scores across zero. Per expert e, the GPU's selection score
    lies within err_e of the oracle's:
      no bias    selection on z itself (softmax and sigmoid are monotone):
                 err_e = |dz_e|;
      sigmoid    q = sigma(z) + bias: slope <= 1/4, so 0.25 |dz_e|, plus the
                 fp32 evaluation of sigma (a few ulp: 2^-20 p_e) and of the
                 add (2^-22 |q_e|);
      softmax    q = p + bias: |dp_e| <= p_e (|dz_e| + max |dz|) <= 2 p_e max|dz|
                 (2.5 p_e max|dz| kept), plus the same fp32 terms."""
    dz = np.abs(z_gpu - z_ref)
    if bias is None:
        return check_selection_gaps(idx_gpu, z_ref, k, dz, what)
    p = O.scores(z_ref, w_score)
    q = p + bias[None, :]
    rnd = 2.0 ** -20 * p + 2.0 ** -22 * np.abs(q)
    if w_score == O.SIGMOID:
        err = 0.25 * dz + rnd
    else:
        err = 2.5 * p * dz.max(axis=1, keepdims=True) + rnd
    return check_selection_gaps(idx_gpu, q, k, err, what)


def oracle_gates_from_logits(z_gpu64, idx_gpu, w_score, w_norm):
    p = O.scores(z_gpu64, w_score)
    return O.gates_from_scores(p, idx_gpu, w_norm)


def check_combine(r, cfg, what="combine"):
    """GPU out vs the oracle combine of the GPU's own y_rows, inv, gates."""
    y_rows, inv, g = np_f(r["y_rows"]), np_i(r["inv"]), np_f(r["gate"])
    ysh = None if r.get("y_sh") is None else np_f(r["y_sh"])
    ref = O.combine(y_rows, inv, g, ysh)
    got = np_f(r["out"])
    # fp32 accumulation error E (k+1 fused steps), then one rounding to dtype
    mag = O.combine(np.abs(y_rows), inv, np.abs(g), None if ysh is None else np.abs(ysh))
    E = (inv.shape[1] + 1) * U32 * mag + 1e-30
    if cfg.dtype == api.DTYPES["f32"]:
        bound = U32 * 2 * (np.abs(ref) + E) + E
    else:
        bound = 2.0 ** -8 * (np.abs(ref) + E) + E
    viol = np.abs(got - ref) > bound
    assert not viol.any(), f"{what}: {int(viol.sum())} elements beyond one rounding"
