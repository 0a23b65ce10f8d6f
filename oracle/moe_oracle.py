"""CPU oracle for the forward pass of a token-choice top-k MoE SwiGLU layer.

TEST INFRASTRUCTURE ONLY. This module is the slow, plain reference that the
CUDA library is checked against. Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it. The library's product path never calls it, and it shares no code with the
CUDA sources.

Everything here works in float64 on numpy arrays built from the exact values
of the (possibly bf16-rounded) inputs. Each function restates one step of the
method as the pages define it; the citation names the page title and the
section or formula.

Pages cited
-----------
[P1] "MOE 专家选择与路由机制" (wuhy-notes)
[P2] "MoE：router 怎样选 expert" (cooking-agi, router page)
[P3] pwwt.cn blog on MoE routing, §2.1 "Top-K取法的工作细节"
[P4] "拆解 MoE：单个 Token 如何经过专家层"
[P5] "【大模型】MoE（专家混合模型）简介"

Readings taken where the pages leave a step open (each is listed with its
reason in the design notes of the repository):
* ties in top-k go to the lower expert index; selected slots are ordered by
  descending selection score, then ascending index;
* the per-expert bias enters the selection score only; gates use the
  un-biased scores;
* sigmoid + renormalise divides each selected sigmoid score by the sum over
  the selected experts, with no further scale;
* rows of the dispatched layout are ordered by (expert ascending, token
  ascending);
* no capacity limit, nothing dropped.

Pinned by ``tests/test_oracle_pins.py`` against the worked examples the pages
print, closed forms, library routines and brute force. Every function below
has at least one pin.
"""
from __future__ import annotations

import itertools

import numpy as np

SOFTMAX = "softmax"
SIGMOID = "sigmoid"
NORM_SELECTED = "selected"
NORM_NONE = "none"


# --------------------------------------------------------------------------
# Stage 1: router logits
# --------------------------------------------------------------------------
def router_logits(h, W_r, b_r=None):
    """z_t = W_r h_t + b_r for every token.

    [P1] §二 第一步: the router is a small linear layer, W_r in R^{N x d};
    [P4] "router_logits = x @ W_router^T".
    h: [T, d], W_r: [N, d], b_r: [N] or None. Returns z: [T, N].
    """
    h = np.asarray(h, dtype=np.float64)
    W_r = np.asarray(W_r, dtype=np.float64)
    z = h @ W_r.T
    if b_r is not None:
        z = z + np.asarray(b_r, dtype=np.float64)[None, :]
    return z


# --------------------------------------------------------------------------
# Stage 2: scores, selection, gates
# --------------------------------------------------------------------------
def softmax(z):
    """p_{t,i} = exp(z_{t,i}) / sum_j exp(z_{t,j}) over all N experts.

    [P1] §二 第二步. The row maximum is subtracted first; in exact
    arithmetic this changes nothing.
    """
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def sigmoid(z):
    """sigma(z) = 1 / (1 + exp(-z)), per expert.

    [P2] "最常见的 router": DeepSeek-V3 scores with a sigmoid and then
    normalises over the selected experts; [P5] §8 lists sigmoid routers.
    """
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def scores(z, score_kind):
    if score_kind == SOFTMAX:
        return softmax(z)
    if score_kind == SIGMOID:
        return sigmoid(z)
    raise ValueError(f"unknown score kind {score_kind!r}")


def select_topk(q, k):
    """S_t = TopK(q_t, k): the k experts with the largest selection score.

    [P1] §二 第三步. Order: descending q; equal q go to the lower index
    first (the pages only warn that torch.topk is not stable on ties, [P2]
    "怎么知道实现没把梯度弄丢"). A stable sort of -q gives exactly this order.
    q: [T, N]. Returns int64 [T, k].
    """
    q = np.asarray(q, dtype=np.float64)
    if not 1 <= k <= q.shape[-1]:
        raise ValueError("need 1 <= k <= N")
    order = np.argsort(-q, axis=-1, kind="stable")
    return order[:, :k]


def gates_from_scores(p, S, norm):
    """Gate weights of the selected experts, in slot order.

    NORM_SELECTED: g_{t,i} = p_{t,i} / sum_{j in S_t} p_{t,j}  ([P1] §二
    第三步 formula for g; [P2] sigmoid-then-renormalise).
    NORM_NONE: g_{t,i} = p_{t,i}, the full-softmax probability of the chosen
    expert (Switch top-1, [P2] "例如分数为 [2, 1, 0]" paragraph; [P3] §2.1
    scatter of top_probs with no renormalisation).
    """
    ps = np.take_along_axis(np.asarray(p, dtype=np.float64), S, axis=-1)
    if norm == NORM_SELECTED:
        return ps / ps.sum(axis=-1, keepdims=True)
    if norm == NORM_NONE:
        return ps
    raise ValueError(f"unknown norm {norm!r}")


def gates_from_selected_logits(z, S):
    """g_i = exp(s_i) / sum_{j in TopK} exp(s_j): softmax over the selected logits.

    [P2] "最常见的 router" formula; the page states it equals a full softmax
    followed by renormalisation over the selected experts.
    """
    zs = np.take_along_axis(np.asarray(z, dtype=np.float64), S, axis=-1)
    m = zs.max(axis=-1, keepdims=True)
    e = np.exp(zs - m)
    return e / e.sum(axis=-1, keepdims=True)


def route(z, k, score_kind=SOFTMAX, norm=NORM_SELECTED, sel_bias=None):
    """Scores, selection and gates for every token.

    p = score(z); q = p + bias (bias steers selection only: [P1] §五
    "动态调整专家选择偏置", [P4] overloaded experts become harder to select,
    [P5] §7 bias added to router scores); S = TopK(q, k); g from p.
    Returns (S [T,k] int64, g [T,k], p [T,N], q [T,N]).
    """
    p = scores(z, score_kind)
    q = p if sel_bias is None else p + np.asarray(sel_bias, dtype=np.float64)[None, :]
    S = select_topk(q, k)
    g = gates_from_scores(p, S, norm)
    return S, g, p, q


def gate_matrix(S, g, N):
    """Dense [T, N] gate matrix: g at the selected experts, zero elsewhere.

    [P3] §2.1: gates = zeros_like(probs); gates.scatter_(-1, top_indices, w).
    """
    T = S.shape[0]
    G = np.zeros((T, N), dtype=np.float64)
    np.put_along_axis(G, S, g, axis=-1)
    return G


# --------------------------------------------------------------------------
# Stage 3/4: dispatch (regroup (token, slot) pairs by expert)
# --------------------------------------------------------------------------
def dispatch(S, N):
    """Per-expert buckets of the (token, slot) pairs.

    [P1] §三 Token Dispatch: pairs sent to the same expert are gathered
    together, tokens listed in ascending order (E0 <- T0, T2 ...); [P5] §3
    stage ② regroups tokens by expert so that each expert runs one GEMM.
    Returns
      counts    [N]    tokens per expert,
      offsets   [N+1]  exclusive prefix sum of counts,
      row_token [T*k]  token of each dispatched row,
      inv       [T,k]  dispatched row of (token t, slot j).
    """
    S = np.asarray(S)
    T, k = S.shape
    e_flat = S.reshape(-1)
    t_flat = np.repeat(np.arange(T), k)
    counts = np.bincount(e_flat, minlength=N).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    order = np.lexsort((t_flat, e_flat))      # by expert, then by token
    row_token = t_flat[order]
    inv_flat = np.empty(T * k, dtype=np.int64)
    inv_flat[order] = np.arange(T * k)
    return counts, offsets, row_token, inv_flat.reshape(T, k)


# --------------------------------------------------------------------------
# Stage 5/6: the expert FFN
# --------------------------------------------------------------------------
def silu(a):
    """SiLU(a) = a * sigma(a)."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def swiglu_expert(x, W_gate, W_up, W_down):
    """E(x) = W_down (SiLU(W_gate x) ⊙ W_up x), row by row.

    [P1] §一: FFN(h) = W_down (SiLU(W_gate h) ⊙ W_up h) and the per-expert
    form E_i(h). x: [R, d], W_gate/W_up: [F, d], W_down: [d, F].
    """
    x = np.asarray(x, dtype=np.float64)
    a = silu(x @ np.asarray(W_gate, np.float64).T) * (x @ np.asarray(W_up, np.float64).T)
    return a @ np.asarray(W_down, np.float64).T


def swiglu_act(x, W_gate, W_up):
    """The expert's hidden activation SiLU(W_gate x) ⊙ W_up x, [R, F]."""
    x = np.asarray(x, dtype=np.float64)
    return silu(x @ np.asarray(W_gate, np.float64).T) * (x @ np.asarray(W_up, np.float64).T)


def expert_rows(x_disp, offsets, W_gate, W_up, W_down):
    """y_rows[r] = E_e(x_disp[r]) for every dispatched row r of expert e.

    Experts with no rows are skipped ([P1] §十四, [P2] sparse_moe).
    """
    R = x_disp.shape[0]
    y = np.zeros((R, W_down.shape[1]), dtype=np.float64)
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            y[r0:r1] = swiglu_expert(x_disp[r0:r1], W_gate[e], W_up[e], W_down[e])
    return y


# --------------------------------------------------------------------------
# Stage 7: combine
# --------------------------------------------------------------------------
def combine(y_rows, inv, g, y_shared=None):
    """out_t = [y_shared_t +] sum_j g_{t,j} * y_rows[inv[t, j]].

    [P2] "选好以后": outputs are weighted and ADDED back to their token,
    never overwritten or concatenated; [P5] §3 stage ④ restores token order
    and fuses by router weight; [P1] §八 adds the shared experts' output.
    """
    y_rows = np.asarray(y_rows, dtype=np.float64)
    inv = np.asarray(inv)
    T, k = inv.shape
    out = np.zeros((T, y_rows.shape[1]), dtype=np.float64)
    if y_shared is not None:
        out += np.asarray(y_shared, dtype=np.float64)
    for j in range(k):
        out += np.asarray(g, np.float64)[:, j:j + 1] * y_rows[inv[:, j]]
    return out


# --------------------------------------------------------------------------
# The whole layer
# --------------------------------------------------------------------------
def moe_forward(h, W_r, W_gate, W_up, W_down, k, score_kind=SOFTMAX,
                norm=NORM_SELECTED, sel_bias=None, b_r=None, shared=None):
    """Sparse forward, one expert at a time.

    Follows the per-expert loop of [P1] §十四 and [P2] sparse_moe: route,
    then for every expert gather its tokens, run the expert, weight by the
    gate and index-add into the output; plus the always-on shared expert of
    [P1] §八: y_t = sum_{s in Shared} E_s(h_t) + sum_{i in S_t} g_{t,i} E_i(h_t).
    ``shared`` is None or a tuple (Ws_gate, Ws_up, Ws_down).
    Returns (y [T,d], z [T,N], S [T,k], g [T,k]).
    """
    h = np.asarray(h, dtype=np.float64)
    z = router_logits(h, W_r, b_r)
    S, g, _, _ = route(z, k, score_kind, norm, sel_bias)
    y = np.zeros_like(h)
    if shared is not None:
        y += swiglu_expert(h, *shared)
    for e in range(W_gate.shape[0]):
        tok, slot = np.nonzero(S == e)
        if tok.size == 0:
            continue
        y_e = swiglu_expert(h[tok], W_gate[e], W_up[e], W_down[e])
        np.add.at(y, tok, g[tok, slot][:, None] * y_e)
    return y, z, S, g


def moe_forward_dense(h, W_r, W_gate, W_up, W_down, k, score_kind=SOFTMAX,
                      norm=NORM_SELECTED, sel_bias=None, b_r=None, shared=None):
    """Dense masked forward: every expert runs on every token.

    [P2] "怎么知道实现没把梯度弄丢": let all experts process all inputs, set
    the weight of unselected experts to zero, and sum; it must equal the
    sparse dispatch result. The gate matrix is [P3] §2.1's scattered gates.
    """
    h = np.asarray(h, dtype=np.float64)
    z = router_logits(h, W_r, b_r)
    S, g, _, _ = route(z, k, score_kind, norm, sel_bias)
    G = gate_matrix(S, g, W_gate.shape[0])
    y = np.zeros_like(h)
    if shared is not None:
        y += swiglu_expert(h, *shared)
    for e in range(W_gate.shape[0]):
        y += G[:, e:e + 1] * swiglu_expert(h, W_gate[e], W_up[e], W_down[e])
    return y, z, S, g


# --------------------------------------------------------------------------
# Brute-force helpers used only by the oracle's own pins
# --------------------------------------------------------------------------
def topk_by_rank_count(q_row, k):
    """Selection by counting, without sorting: expert i is selected iff fewer
    than k experts beat it, where j beats i when q_j > q_i, or q_j == q_i and
    j < i. Returns the selected indices ordered by that same relation."""
    q_row = list(map(float, q_row))
    N = len(q_row)
    beats = lambda j, i: q_row[j] > q_row[i] or (q_row[j] == q_row[i] and j < i)
    rank = [sum(1 for j in range(N) if j != i and beats(j, i)) for i in range(N)]
    chosen = [i for i in range(N) if rank[i] < k]
    return sorted(chosen, key=lambda i: rank[i])


def topk_by_subsets(q_row, k):
    """Exhaustive: the k-subset with the largest score sum; among equal sums
    the lexicographically smallest index tuple. Valid as a pin only when the
    scores of different subsets do not tie."""
    best = None
    for sub in itertools.combinations(range(len(q_row)), k):
        key = (-sum(float(q_row[i]) for i in sub), sub)
        if best is None or key < best:
            best = key
    return set(best[1])


# --------------------------------------------------------------------------
# Routing side statistics
# --------------------------------------------------------------------------
def router_probabilities(z, score_kind):
    """Per-token distribution over experts used by the balance statistics.

    Softmax router: p = softmax(z). Sigmoid router: the scores divided by
    their sum over all experts, so that each row sums to 1 (reading taken:
    the pages define the statistics with router probabilities, and a sigmoid
    router's scores are not a distribution until normalised)."""
    if score_kind == SOFTMAX:
        return softmax(z)
    s = sigmoid(z)
    return s / s.sum(axis=-1, keepdims=True)


def logsumexp(z):
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[..., 0]


def routing_stats(z, S, score_kind, N):
    """Balance and stability statistics of one routing decision.

    [P1] §五: f_i = share of routed (token, slot) pairs sent to expert i,
    P_i = mean router probability of expert i, L_balance = N * sum_i f_i P_i
    (equal to 1 when both are uniform); router z-loss
    L_z = (1/T) sum_t (log sum_i exp z_{t,i})^2. [P1] §十三 lists the per-expert
    load and the routing entropy among the quantities to monitor:
    H = (1/T) sum_t -sum_i p_{t,i} log p_{t,i}.
    Returns a dict with L_bal, L_z, entropy, P [N], f [N]."""
    z = np.asarray(z, dtype=np.float64)
    S = np.asarray(S)
    T, k = S.shape
    p = router_probabilities(z, score_kind)
    P = p.mean(axis=0)
    f = np.bincount(S.reshape(-1), minlength=N).astype(np.float64) / (T * k)
    with np.errstate(divide="ignore", invalid="ignore"):
        plogp = np.where(p > 0, p * np.log(p), 0.0)
    return dict(L_bal=float(N * np.sum(f * P)), L_z=float(np.mean(logsumexp(z) ** 2)),
                entropy=float(np.mean(-plogp.sum(axis=-1))), P=P, f=f)


# --------------------------------------------------------------------------
# Group-limited selection
# --------------------------------------------------------------------------
GROUP_MAX = "max"
GROUP_TOPM_SUM = "topm_sum"


def select_topk_grouped(q, k, n_group, topk_group, group_score=GROUP_MAX, top_m=2):
    """Group-limited top-k ([P2] "跨设备时，为什么还要先选组？").

    The N experts form n_group contiguous groups of N / n_group. Each group is
    scored by its largest selection score (GROUP_MAX) or by the sum of its
    top_m scores (GROUP_TOPM_SUM, the DeepSeek-V3 node score the page
    describes); the topk_group best groups are kept (equal group scores: lower
    group index first); the experts of every other group are masked with -inf
    (not 0, so that negative scores cannot win through the mask); the top-k
    then runs over the remaining experts with the usual order. Fewer than k
    remaining candidates is an error, as on the page."""
    q = np.asarray(q, dtype=np.float64)
    T, N = q.shape
    if n_group < 1 or N % n_group:
        raise ValueError("N must split into n_group equal groups")
    gs = N // n_group
    if not 1 <= topk_group <= n_group:
        raise ValueError("need 1 <= topk_group <= n_group")
    if topk_group * gs < k:
        raise ValueError("fewer candidates than k after group selection")
    qg = q.reshape(T, n_group, gs)
    if group_score == GROUP_MAX:
        sg = qg.max(axis=-1)
    elif group_score == GROUP_TOPM_SUM:
        if not 1 <= top_m <= gs:
            raise ValueError("need 1 <= top_m <= group size")
        sg = -np.sort(-qg, axis=-1)[..., :top_m].sum(axis=-1)
    else:
        raise ValueError(f"unknown group score {group_score!r}")
    kept = select_topk(sg, topk_group)
    mask = np.full((T, n_group), -np.inf)
    np.put_along_axis(mask, kept, 0.0, axis=-1)
    return select_topk((qg + mask[..., None]).reshape(T, N), k)


def route_grouped(z, k, n_group, topk_group, group_score=GROUP_MAX, top_m=2,
                  score_kind=SOFTMAX, norm=NORM_SELECTED, sel_bias=None):
    """route() with the selection limited to the best groups; gates as route()."""
    p = scores(z, score_kind)
    q = p if sel_bias is None else p + np.asarray(sel_bias, dtype=np.float64)[None, :]
    S = select_topk_grouped(q, k, n_group, topk_group, group_score, top_m)
    return S, gates_from_scores(p, S, norm), p, q


# --------------------------------------------------------------------------
# Expert capacity and token dropping
# --------------------------------------------------------------------------
def expert_capacity(T, k, N, capacity_factor):
    """C = ceil(capacity_factor * T * k / N) ([P1] §六 Expert Capacity)."""
    import math
    return int(math.ceil(capacity_factor * T * k / N))


def dispatch_capacity(S, N, C):
    """Dispatch with at most C rows per expert ([P1] §六: tokens beyond the
    capacity may be dropped; the page leaves the policy to the
    implementation). Reading taken: each expert keeps its first C (token,
    slot) pairs in token order and drops the rest; a dropped pair has
    inv = -1 and contributes nothing (the token keeps its other experts and
    the residual path); gates are not renormalised.
    Returns counts (kept rows per expert), offsets, row_token (kept rows
    only), inv [T,k] with -1 for dropped pairs."""
    S = np.asarray(S)
    T, k = S.shape
    full_counts, full_offsets, full_row_token, full_inv = dispatch(S, N)
    counts = np.minimum(full_counts, C)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    inv = np.full((T, k), -1, dtype=np.int64)
    row_token = np.empty(int(counts.sum()), dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(S[t, j])
            rank = int(full_inv[t, j] - full_offsets[e])   # position among e's pairs
            if rank < C:
                inv[t, j] = offsets[e] + rank
                row_token[offsets[e] + rank] = t
    return counts, offsets, row_token, inv


def moe_forward_capacity(h, W_r, W_gate, W_up, W_down, k, C, score_kind=SOFTMAX,
                         norm=NORM_SELECTED, sel_bias=None, b_r=None, shared=None):
    """The layer with expert capacity C: route, dispatch_capacity, experts on
    the kept rows, combine skipping dropped pairs. Returns (y, S, g, inv)."""
    h = np.asarray(h, dtype=np.float64)
    z = router_logits(h, W_r, b_r)
    S, g, _, _ = route(z, k, score_kind, norm, sel_bias)
    counts, offsets, row_token, inv = dispatch_capacity(S, W_gate.shape[0], C)
    y_rows = expert_rows(h[row_token], offsets, W_gate, W_up, W_down)
    y = np.zeros_like(h)
    if shared is not None:
        y += swiglu_expert(h, *shared)
    for t in range(h.shape[0]):
        for j in range(k):
            if inv[t, j] >= 0:
                y[t] += g[t, j] * y_rows[inv[t, j]]
    return y, S, g, inv


# --------------------------------------------------------------------------
# Expert Choice routing
# --------------------------------------------------------------------------
def expert_choice(z, C, score_kind=SOFTMAX):
    """Expert Choice ([P1] §九 routing table; [P2] "Token 选 expert，还是 expert
    选 token"): each expert picks the C tokens with the highest router score
    for it; a token can be picked by any number of experts (0..N).
    Scores p = softmax over experts per token (or sigmoid). Reading taken:
    equal scores go to the lower token index; an expert's picked tokens are
    listed in ascending token order (the order does not change the output).
    Returns (tokens [N, C] int64, gates [N, C] = p[token, expert], p)."""
    p = scores(z, score_kind)
    T, N = p.shape
    if not 0 <= C <= T:
        raise ValueError("need 0 <= C <= T")
    picked = select_topk(p.T, C) if C > 0 else np.zeros((N, 0), dtype=np.int64)
    tokens = np.sort(picked, axis=1)
    gates = np.take_along_axis(p.T, tokens, axis=1)
    return tokens, gates, p


def moe_forward_expert_choice(h, W_r, W_gate, W_up, W_down, C, score_kind=SOFTMAX,
                              b_r=None, shared=None):
    """y_t = [sum_s E_s(h_t)] + sum_{e : t picked by e} p_{t,e} E_e(h_t)."""
    h = np.asarray(h, dtype=np.float64)
    z = router_logits(h, W_r, b_r)
    tokens, gates, _ = expert_choice(z, C, score_kind)
    y = np.zeros_like(h)
    if shared is not None:
        y += swiglu_expert(h, *shared)
    for e in range(W_gate.shape[0]):
        toks = tokens[e]
        if toks.size:
            np.add.at(y, toks, gates[e][:, None] * swiglu_expert(h[toks], W_gate[e], W_up[e],
                                                                  W_down[e]))
    return y, tokens, gates
