"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (a host program without an allocator of its own, or a
runtime that forbids device allocation while it runs). It keeps its scratch
in a fixed array inside the library, so its results must equal those of
moe_dispatch with a caller workspace, call after call. This file is collected
last on purpose."""
import ctypes

import pytest
import torch

from top_routing_grouped_bias_b300 import api


def _case(T, N, k, d, seed):
    gen = torch.Generator().manual_seed(seed)
    # k distinct experts per token: the k largest of N seeded uniforms
    idx = torch.rand((T, N), generator=gen).topk(k, dim=1).indices.to(torch.int32)
    h = torch.randn((T, d), generator=gen).to(torch.bfloat16)
    return idx, h


def _buffers(cfg, dev):
    R = cfg.T * cfg.k
    return dict(counts=torch.full((cfg.N,), -7, dtype=torch.int32, device=dev),
                offsets=torch.full((cfg.N + 1,), -7, dtype=torch.int32, device=dev),
                row_token=torch.full((R,), -7, dtype=torch.int32, device=dev),
                inv=torch.full((cfg.T, cfg.k), -7, dtype=torch.int32, device=dev),
                x_disp=torch.zeros((R, cfg.d), dtype=torch.bfloat16, device=dev))


@pytest.mark.gpu
def test_noalloc_dispatch_matches_workspace_dispatch_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a visible CUDA device")
    api.load()
    dev = "cuda"
    # calls in a row with different shapes, each reusing the array the one
    # before filled: the last fills the array exactly (ceil(65536 / 256) *
    # 1024 = 262144 entries), the third skips the row gather (x_disp NULL),
    # the fourth is small enough for the one-block count/scan/permute
    cases = ((5000, 256, 8, 64, 1, True), (777, 1024, 4, 128, 2, True),
             (3000, 64, 6, 32, 3, False), (1000, 8, 2, 64, 5, True),
             (65536, 1024, 2, 16, 4, True))
    for T, N, k, d, seed, gather in cases:
        cfg = api.make_config(T, d, N, k, 64)
        idx, h = _case(T, N, k, d, seed)
        idx, h = idx.to(dev), h.to(dev)
        ref = _buffers(cfg, dev)
        ws = api.alloc_workspace(cfg, dev)
        api.moe_dispatch(cfg, h, idx, ref["counts"], ref["offsets"], ref["row_token"],
                         ref["inv"], ref["x_disp"] if gather else None, ws)
        got = _buffers(cfg, dev)
        api.moe_dispatch_noalloc(cfg, h, idx, got["counts"], got["offsets"], got["row_token"],
                                 got["inv"], got["x_disp"] if gather else None)
        torch.cuda.synchronize()
        for key in ref:
            assert torch.equal(got[key], ref[key]), f"{key} differs (T={T}, N={N}, k={k})"
        if not gather:
            assert not got["x_disp"].any(), "x_disp written although it was not passed"
        assert int(got["counts"].sum()) == T * k


def test_noalloc_dispatch_rejects_sizes_beyond_its_scratch():
    """Host-side check, before anything is launched: ceil(T/256) * N must fit
    the fixed 262144-entry histogram array."""
    lib = api.load()
    fake = ctypes.c_void_p(1 << 20)
    too_big = api.make_config(65536 + 256, 64, 1024, 2, 64)
    assert lib.moe_dispatch_noalloc(ctypes.byref(too_big), fake, fake, fake, fake, fake, fake,
                                    fake, None) == api.MOE_ERR_WORKSPACE
    bad = api.make_config(64, 64, 4, 5, 64)                      # k > N
    assert lib.moe_dispatch_noalloc(ctypes.byref(bad), fake, fake, fake, fake, fake, fake,
                                    fake, None) == api.MOE_ERR_INVALID_ARG
