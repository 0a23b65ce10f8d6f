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
