"""Python binding of libmoe_b300.so (include/moe.h): argument marshalling only.

Every function here takes torch tensors (or None), passes their device
pointers and the current CUDA stream to the C ABI, and raises ``MoeError`` on
a non-OK status. All arithmetic of the layer runs in the library's kernels;
there is no fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_CHECK = 6

DTYPES = {"bf16": 0, "f32": 1}
SCORES = {"softmax": 0, "sigmoid": 1}
NORMS = {"selected": 0, "none": 1}

# Every entry point declared in include/moe.h.
ENTRY_POINTS = (
    "moe_workspace_size", "moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine",
    "moe_forward", "moe_read_status", "moe_selftest_wait_timeout", "moe_status_string",
    "moe_dispatch_noalloc", "moe_route_stats", "moe_route_grouped", "moe_dispatch_capacity",
    "moe_forward_capacity", "moe_forward_expert_choice", "moe_expert_ffn_gather",
    "moe_expert_capacity",
)


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} failed: {status_string(status)} ({status})")


class MoeGroupConfig(ctypes.Structure):
    _fields_ = [("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("rule", ctypes.c_int32), ("top_m", ctypes.c_int32)]


GROUP_RULES = {"max": 0, "topm_sum": 1}


def make_group_config(n_group: int, topk_group: int, rule: str = "max",
                      top_m: int = 2) -> MoeGroupConfig:
    return MoeGroupConfig(int(n_group), int(topk_group), GROUP_RULES[rule], int(top_m))


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("N", ctypes.c_int32),
                ("k", ctypes.c_int32), ("ffn", ctypes.c_int32), ("ffn_shared", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("score", ctypes.c_int32), ("norm", ctypes.c_int32)]


_lib: Optional[ctypes.CDLL] = None
_vp, _sz, _i32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int32)


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m top_routing_grouped_bias_b300.build`")
    lib = ctypes.CDLL(path)
    cfgp = ctypes.POINTER(MoeConfig)
    lib.moe_workspace_size.argtypes = [cfgp]
    lib.moe_workspace_size.restype = _sz
    lib.moe_route.argtypes = [cfgp] + [_vp] * 8 + [_vp, _sz, _vp]
    lib.moe_dispatch.argtypes = [cfgp] + [_vp] * 7 + [_vp, _sz, _vp]
    lib.moe_dispatch_noalloc.argtypes = [cfgp] + [_vp] * 7 + [_vp]
    lib.moe_route_stats.argtypes = [cfgp] + [_vp] * 3 + [_vp, _sz, _vp]
    lib.moe_dispatch_capacity.argtypes = [cfgp, ctypes.c_int64] + [_vp] * 7 + [_vp, _sz, _vp]
    lib.moe_forward_capacity.argtypes = [cfgp, ctypes.c_int64] + [_vp] * 15 + [_vp, _sz, _vp]
    lib.moe_forward_expert_choice.argtypes = [cfgp, ctypes.c_int64] + [_vp] * 13 + [_vp, _sz, _vp]
    lib.moe_route_grouped.argtypes = [cfgp, ctypes.POINTER(MoeGroupConfig)] + [_vp] * 8 + \
        [_vp, _sz, _vp]
    lib.moe_expert_ffn.argtypes = [cfgp] + [_vp] * 11 + [_vp, _sz, _vp]
    lib.moe_expert_ffn_gather.argtypes = [cfgp] + [_vp] * 11 + [_vp, _sz, _vp]
    lib.moe_combine.argtypes = [cfgp] + [_vp] * 5 + [_vp]
    lib.moe_forward.argtypes = [cfgp] + [_vp] * 15 + [_vp, _sz, _vp]
    lib.moe_read_status.argtypes = [_vp, _sz, _i32p, _vp]
    lib.moe_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _vp, _sz, _vp]
    lib.moe_expert_capacity.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_double, ctypes.POINTER(ctypes.c_int64)]
    lib.moe_status_string.argtypes = [ctypes.c_int32]
    lib.moe_status_string.restype = ctypes.c_char_p
    for name in ENTRY_POINTS:
        if name not in ("moe_workspace_size", "moe_status_string"):
            getattr(lib, name).restype = ctypes.c_int32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def make_config(T: int, d: int, N: int, k: int, ffn: int, ffn_shared: int = 0,
                dtype: str = "bf16", score: str = "softmax", norm: str = "selected") -> MoeConfig:
    return MoeConfig(int(T), int(d), int(N), int(k), int(ffn), int(ffn_shared),
                     DTYPES[dtype], SCORES[score], NORMS[norm])


def config_for(w, T: Optional[int] = None) -> MoeConfig:
    """Config of a synth.Workload (optionally with another token count)."""
    return make_config(w.T if T is None else T, w.d, w.N, w.k, w.F, w.F_sh,
                       w.dtype, w.score, w.norm)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def workspace_size(cfg: MoeConfig) -> int:
    return int(load().moe_workspace_size(ctypes.byref(cfg)))


def alloc_workspace(cfg: MoeConfig, device="cuda") -> torch.Tensor:
    n = workspace_size(cfg)
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_workspace_size")
    ws = torch.zeros(n, dtype=torch.uint8, device=device)
    return ws


def moe_route(cfg, h, W_r, b_r, sel_bias, logits_in, logits_out, idx, gate, ws=None, stream=None):
    s = load().moe_route(ctypes.byref(cfg), _p(h), _p(W_r), _p(b_r), _p(sel_bias), _p(logits_in),
                         _p(logits_out), _p(idx), _p(gate), _p(ws),
                         0 if ws is None else ws.numel(), _stream(stream))
    _check(s, "moe_route")


def moe_dispatch(cfg, h, idx, counts, offsets, row_token, inv, x_disp, ws, stream=None):
    s = load().moe_dispatch(ctypes.byref(cfg), _p(h), _p(idx), _p(counts), _p(offsets),
                            _p(row_token), _p(inv), _p(x_disp), _p(ws), ws.numel(), _stream(stream))
    _check(s, "moe_dispatch")


def moe_dispatch_noalloc(cfg, h, idx, counts, offsets, row_token, inv, x_disp, stream=None):
    """moe_dispatch without a workspace, for callers that cannot allocate
    device memory: the library keeps the scratch in a fixed array of its own
    (at most ceil(T/256) * N = 262144 histogram entries). Calls that overlap
    on the GPU share that array and race."""
    s = load().moe_dispatch_noalloc(ctypes.byref(cfg), _p(h), _p(idx), _p(counts), _p(offsets),
                                    _p(row_token), _p(inv), _p(x_disp), _stream(stream))
    _check(s, "moe_dispatch_noalloc")


def moe_expert_ffn(cfg, x_disp, offsets, W_gate, W_up, W_down, y_rows, h=None, Ws_gate=None,
                   Ws_up=None, Ws_down=None, y_shared=None, ws=None, stream=None):
    s = load().moe_expert_ffn(ctypes.byref(cfg), _p(x_disp), _p(offsets), _p(W_gate), _p(W_up),
                              _p(W_down), _p(y_rows), _p(h), _p(Ws_gate), _p(Ws_up), _p(Ws_down),
                              _p(y_shared), _p(ws), 0 if ws is None else ws.numel(),
                              _stream(stream))
    _check(s, "moe_expert_ffn")


def moe_expert_ffn_gather(cfg, h, row_token, offsets, W_gate, W_up, W_down, y_rows,
                          Ws_gate=None, Ws_up=None, Ws_down=None, y_shared=None, ws=None,
                          stream=None):
    s = load().moe_expert_ffn_gather(ctypes.byref(cfg), _p(h), _p(row_token), _p(offsets),
                                     _p(W_gate), _p(W_up), _p(W_down), _p(y_rows), _p(Ws_gate),
                                     _p(Ws_up), _p(Ws_down), _p(y_shared), _p(ws),
                                     0 if ws is None else ws.numel(), _stream(stream))
    _check(s, "moe_expert_ffn_gather")


def moe_combine(cfg, y_rows, inv, gate, y_shared, out, stream=None):
    s = load().moe_combine(ctypes.byref(cfg), _p(y_rows), _p(inv), _p(gate), _p(y_shared),
                           _p(out), _stream(stream))
    _check(s, "moe_combine")


def moe_forward(cfg, h, W_r, b_r, sel_bias, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down,
                out, logits_out, idx, gate, counts, ws, stream=None):
    s = load().moe_forward(ctypes.byref(cfg), _p(h), _p(W_r), _p(b_r), _p(sel_bias), _p(W_gate),
                           _p(W_up), _p(W_down), _p(Ws_gate), _p(Ws_up), _p(Ws_down), _p(out),
                           _p(logits_out), _p(idx), _p(gate), _p(counts), _p(ws), ws.numel(),
                           _stream(stream))
    _check(s, "moe_forward")


def moe_route_grouped(cfg, grp, h, W_r, b_r, sel_bias, logits_in, logits_out, idx, gate,
                      ws=None, stream=None):
    s = load().moe_route_grouped(ctypes.byref(cfg), ctypes.byref(grp), _p(h), _p(W_r), _p(b_r),
                                 _p(sel_bias), _p(logits_in), _p(logits_out), _p(idx), _p(gate),
                                 _p(ws), 0 if ws is None else ws.numel(), _stream(stream))
    _check(s, "moe_route_grouped")


def expert_capacity(T: int, k: int, N: int, capacity_factor: float) -> int:
    """The library's moe_expert_capacity: C = ceil(capacity_factor * T * k / N)."""
    out = ctypes.c_int64(0)
    s = load().moe_expert_capacity(int(T), int(k), int(N), float(capacity_factor),
                                   ctypes.byref(out))
    _check(s, "moe_expert_capacity")
    return int(out.value)


def moe_dispatch_capacity(cfg, capacity, h, idx, counts, offsets, row_token, inv, x_disp, ws,
                          stream=None):
    s = load().moe_dispatch_capacity(ctypes.byref(cfg), int(capacity), _p(h), _p(idx),
                                     _p(counts), _p(offsets), _p(row_token), _p(inv), _p(x_disp),
                                     _p(ws), ws.numel(), _stream(stream))
    _check(s, "moe_dispatch_capacity")


def forward_capacity(cfg, capacity, inp: dict, outs: "Outputs", ws, stream=None):
    s = load().moe_forward_capacity(
        ctypes.byref(cfg), int(capacity), _p(inp["h"]), _p(inp["W_r"]), _p(inp.get("b_r")),
        _p(inp.get("sel_bias")), _p(inp["W_gate"]), _p(inp["W_up"]), _p(inp["W_down"]),
        _p(inp.get("Ws_gate")), _p(inp.get("Ws_up")), _p(inp.get("Ws_down")), _p(outs["out"]),
        _p(outs.get("logits")), _p(outs["idx"]), _p(outs["gate"]), _p(outs.get("counts")), _p(ws),
        ws.numel(), _stream(stream))
    _check(s, "moe_forward_capacity")


def forward_expert_choice(cfg, capacity, inp: dict, out, ws, logits=None, tokens=None,
                          gates=None, stream=None):
    s = load().moe_forward_expert_choice(
        ctypes.byref(cfg), int(capacity), _p(inp["h"]), _p(inp["W_r"]), _p(inp.get("b_r")),
        _p(inp["W_gate"]), _p(inp["W_up"]), _p(inp["W_down"]), _p(inp.get("Ws_gate")),
        _p(inp.get("Ws_up")), _p(inp.get("Ws_down")), _p(out), _p(logits), _p(tokens), _p(gates),
        _p(ws), ws.numel(), _stream(stream))
    _check(s, "moe_forward_expert_choice")


def moe_route_stats(cfg, logits, idx, stats, ws, stream=None):
    """stats [3 + 2N] fp32: L_bal, L_z, entropy, P[N], f[N]."""
    s = load().moe_route_stats(ctypes.byref(cfg), _p(logits), _p(idx), _p(stats), _p(ws),
                               ws.numel(), _stream(stream))
    _check(s, "moe_route_stats")


def read_status(ws: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(0)
    s = load().moe_read_status(_p(ws), ws.numel(), ctypes.byref(v), _stream(stream))
    _check(s, "moe_read_status")
    return int(v.value)


def selftest_wait_timeout(budget_ns: int, ws: torch.Tensor, stream=None):
    s = load().moe_selftest_wait_timeout(int(budget_ns), _p(ws), ws.numel(), _stream(stream))
    _check(s, "moe_selftest_wait_timeout")


# ---------------------------------------------------------------- helpers ---
class Outputs(dict):
    """Allocated output tensors of one forward call (attribute access)."""
    __getattr__ = dict.__getitem__


def alloc_outputs(cfg: MoeConfig, device="cuda", dtype=torch.bfloat16,
                  logits: bool = True) -> Outputs:
    T, d, N, k = cfg.T, cfg.d, cfg.N, cfg.k
    return Outputs(
        out=torch.empty((T, d), dtype=dtype, device=device),
        logits=torch.empty((T, N), dtype=torch.float32, device=device) if logits else None,
        idx=torch.empty((T, k), dtype=torch.int32, device=device),
        gate=torch.empty((T, k), dtype=torch.float32, device=device),
        counts=torch.empty((N,), dtype=torch.int32, device=device),
    )


def forward(cfg: MoeConfig, inp: dict, outs: Outputs, ws: torch.Tensor, stream=None):
    """moe_forward over a dict of inputs as synth.make_inputs returns."""
    moe_forward(cfg, inp["h"], inp["W_r"], inp.get("b_r"), inp.get("sel_bias"), inp["W_gate"],
                inp["W_up"], inp["W_down"], inp.get("Ws_gate"), inp.get("Ws_up"),
                inp.get("Ws_down"), outs["out"], outs.get("logits"), outs["idx"], outs["gate"],
                outs.get("counts"), ws, stream)


class HostPipeline:
    """moe_forward over batches that live in (pinned) host memory, with the
    host-to-device copy of the next batch and the device-to-host copy of the
    previous output running on their own streams while the current batch
    computes. Two device buffers alternate; events order every reuse.

    Only copies and launches are scheduled here; all arithmetic is the
    library's moe_forward.
    """

    def __init__(self, cfg: MoeConfig, weights: dict, dtype=torch.bfloat16, device="cuda"):
        dev = torch.device(device)
        self.cfg, self.weights, self.dev = cfg, weights, dev
        T, d = cfg.T, cfg.d
        self.h_dev = [torch.empty((T, d), dtype=dtype, device=dev) for _ in range(2)]
        self.outs = [alloc_outputs(cfg, dev, dtype, logits=False) for _ in range(2)]
        self.ws = alloc_workspace(cfg, dev)
        self.compute = torch.cuda.current_stream(dev)
        self.copy_in = torch.cuda.Stream(dev)
        self.copy_out = torch.cuda.Stream(dev)
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.in_ready, self.done, self.out_copied = ev(), ev(), ev()
        self.used = [False, False]

    def step(self, i: int, h_host: torch.Tensor, out_host: torch.Tensor):
        b = i % 2
        if self.used[b]:
            self.copy_in.wait_event(self.done[b])            # h_dev[b] no longer read
        with torch.cuda.stream(self.copy_in):
            self.h_dev[b].copy_(h_host, non_blocking=True)
            self.in_ready[b].record(self.copy_in)
        self.compute.wait_event(self.in_ready[b])
        if self.used[b]:
            self.compute.wait_event(self.out_copied[b])      # outs[b] drained to the host
        inp = dict(self.weights)
        inp["h"] = self.h_dev[b]
        forward(self.cfg, inp, self.outs[b], self.ws, self.compute)
        self.done[b].record(self.compute)
        self.copy_out.wait_event(self.done[b])
        with torch.cuda.stream(self.copy_out):
            out_host.copy_(self.outs[b]["out"], non_blocking=True)
            self.out_copied[b].record(self.copy_out)
        self.used[b] = True

    def drain(self):
        """Make the compute stream wait for every copy issued so far."""
        for b in range(2):
            if self.used[b]:
                self.compute.wait_event(self.out_copied[b])
