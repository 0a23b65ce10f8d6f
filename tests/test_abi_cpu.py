"""The C-ABI library loads without a GPU, exports every symbol include/moe.h
declares, and rejects bad arguments on the host before launching anything.
No compute call is made here."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    from top_routing_grouped_bias_b300 import build, api
    build.build()
    return api.load()


@pytest.fixture(scope="module")
def api():
    from top_routing_grouped_bias_b300 import api
    return api


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward"):
        assert required in names


def test_library_exports_every_declared_symbol(lib, api):
    names = declared_functions()
    assert set(names) == set(api.ENTRY_POINTS)
    for n in names:
        assert hasattr(lib, n), n


def test_exported_symbols_have_c_linkage():
    import subprocess
    from top_routing_grouped_bias_b300 import api as _api
    out = subprocess.run(["nm", "-D", "--defined-only", _api.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T (moe_\w+)", out))
    assert set(declared_functions()) <= exported


def test_status_strings(api, lib):
    assert api.status_string(0) == "MOE_OK"
    assert api.status_string(5) == "MOE_ERR_TIMEOUT"
    assert api.status_string(99) == "MOE_UNKNOWN_STATUS"


def test_workspace_size_valid_and_invalid(api, lib):
    cfg = api.make_config(4096, 4096, 8, 2, 14336)
    n = api.workspace_size(cfg)
    R = 4096 * 2
    # x_disp + y_rows + act dominate
    assert n >= R * 4096 * 2 * 2 + R * 14336 * 2
    assert n % 256 == 0
    for bad in (api.make_config(16, 4096, 8, 9, 14336),      # k > N
                api.make_config(16, 4096, 8, 0, 14336),      # k < 1
                api.make_config(16, 4100, 8, 2, 14336),      # d not a multiple of 8 (bf16)
                api.make_config(16, 4096, 8, 2, 14340),      # ffn not a multiple of 8
                api.make_config(16, 4096, 2048, 2, 14336),   # N > 1024
                api.make_config(-1, 4096, 8, 2, 14336),      # T < 0
                api.make_config(16, 4096, 32, 17, 256)):     # k > 16
        assert api.workspace_size(bad) == 0
    assert api.workspace_size(api.make_config(16, 132, 8, 2, 256, dtype="f32")) > 0
    assert api.workspace_size(api.make_config(16, 130, 8, 2, 256, dtype="f32")) == 0


def _cfg(api, **kw):
    base = dict(T=16, d=64, N=4, k=2, ffn=64)
    base.update(kw)
    return api.make_config(**base)


def test_host_validation_rejects_before_launch(api, lib):
    V = ctypes.c_void_p
    cfg = _cfg(api)
    fake = V(1 << 20)          # 16-byte aligned, never dereferenced: validation fails first
    odd = V((1 << 20) + 4)     # misaligned for a bf16 tensor
    # k > N
    bad = _cfg(api, k=5)
    assert lib.moe_route(ctypes.byref(bad), fake, fake, None, None, None, None, fake, fake, None,
                         0, None) == api.MOE_ERR_INVALID_ARG
    # null idx
    assert lib.moe_route(ctypes.byref(cfg), fake, fake, None, None, None, None, None, fake, None,
                         0, None) == api.MOE_ERR_INVALID_ARG
    # misaligned h
    assert lib.moe_route(ctypes.byref(cfg), odd, fake, None, None, None, None, fake, fake, None,
                         0, None) == api.MOE_ERR_INVALID_ARG
    # neither h nor logits
    assert lib.moe_route(ctypes.byref(cfg), None, fake, None, None, None, None, fake, fake, None,
                         0, None) == api.MOE_ERR_INVALID_ARG
    # null config
    assert lib.moe_combine(None, fake, fake, fake, None, fake, None) == api.MOE_ERR_INVALID_ARG
    # dispatch without workspace
    assert lib.moe_dispatch(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, fake, None, 0,
                            None) == api.MOE_ERR_WORKSPACE
    # workspace too small for the expert FFN
    assert lib.moe_expert_ffn(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, None, None,
                              None, None, None, fake, 256, None) == api.MOE_ERR_WORKSPACE
    # shared expert requested but its weights missing
    cfg_sh = _cfg(api, ffn_shared=64)
    big = api.workspace_size(cfg_sh)
    assert lib.moe_expert_ffn(ctypes.byref(cfg_sh), fake, fake, fake, fake, fake, fake, None, None,
                              None, None, None, fake, big, None) == api.MOE_ERR_INVALID_ARG
    # forward: workspace smaller than moe_workspace_size
    n = api.workspace_size(cfg)
    assert lib.moe_forward(ctypes.byref(cfg), fake, fake, None, None, fake, fake, fake, None, None,
                           None, fake, None, fake, fake, None, fake, n - 256,
                           None) == api.MOE_ERR_WORKSPACE
    # status read without a workspace
    v = ctypes.c_int32()
    assert lib.moe_read_status(None, 0, ctypes.byref(v), None) == api.MOE_ERR_INVALID_ARG


def test_route_stats_rejects_small_workspace(api, lib):
    """The statistics need the workspace's partial-sum region and its final
    counter: anything smaller than moe_workspace_size's dispatch prefix is
    refused on the host."""
    fake = ctypes.c_void_p(1 << 20)
    cfg = _cfg(api, T=1000, N=64, k=4)
    assert lib.moe_route_stats(ctypes.byref(cfg), fake, fake, fake, None, 0,
                               None) == api.MOE_ERR_WORKSPACE
    assert lib.moe_route_stats(ctypes.byref(cfg), fake, fake, fake, fake, 256,
                               None) == api.MOE_ERR_WORKSPACE
    assert lib.moe_route_stats(ctypes.byref(cfg), None, fake, fake, fake,
                               api.workspace_size(cfg), None) == api.MOE_ERR_INVALID_ARG


def test_zero_tokens_is_ok_without_launch(api, lib):
    fake = ctypes.c_void_p(1 << 20)
    cfg = _cfg(api, T=0)
    assert lib.moe_route(ctypes.byref(cfg), fake, fake, None, None, None, None, fake, fake, None,
                         0, None) == api.MOE_OK
    assert lib.moe_combine(ctypes.byref(cfg), fake, fake, fake, None, fake, None) == api.MOE_OK
    n = api.workspace_size(cfg)
    assert lib.moe_forward(ctypes.byref(cfg), fake, fake, None, None, fake, fake, fake, None, None,
                           None, fake, None, fake, fake, None, fake, n, None) == api.MOE_OK


def test_product_path_has_no_fallback(api):
    """Without the built library the binding raises instead of computing."""
    import importlib
    mod = importlib.import_module("top_routing_grouped_bias_b300.api")
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(RuntimeError):
            mod.load("/nonexistent/libmoe_b300.so")
    finally:
        mod._lib = saved


def test_product_sources_do_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "top_routing_grouped_bias_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "oracle/" not in src and "moe_oracle" not in src, f


def test_nvtx_ranges_enabled_by_environment(api):
    """MOE_NVTX=1 wraps every entry point in an NVTX range; without a tool
    attached the ranges are no-ops and the calls behave as before (checked
    here on the zero-token path, in a fresh process so that the variable is
    read at the first call)."""
    import subprocess
    import sys
    code = (
        "import ctypes, sys\n"
        "sys.path.insert(0, '.')\n"
        "from top_routing_grouped_bias_b300 import api\n"
        "lib = api.load()\n"
        "cfg = api.make_config(0, 64, 4, 2, 64)\n"
        "fake = ctypes.c_void_p(1 << 20)\n"
        "n = api.workspace_size(cfg)\n"
        "s1 = lib.moe_route(ctypes.byref(cfg), fake, fake, None, None, None, None, fake, fake, None, 0, None)\n"
        "s2 = lib.moe_forward(ctypes.byref(cfg), fake, fake, None, None, fake, fake, fake, None, None,"
        " None, fake, None, fake, fake, None, fake, n, None)\n"
        "print(s1, s2)\n")
    env = dict(os.environ, MOE_NVTX="1")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == [str(api.MOE_OK), str(api.MOE_OK)]


def test_expert_capacity_through_the_abi_matches_the_oracle(api, lib):
    """moe_expert_capacity (pure host arithmetic, no GPU needed) gives the
    oracle's C = ceil(cf * T * k / N) on a grid that includes fractional
    factors, exact multiples and a factor of zero; invalid inputs are
    rejected."""
    import ctypes
    from oracle import moe_oracle as O
    for T in (0, 1, 4, 7, 4096, 8192, 65536, 100003):
        for k, N in ((1, 1), (2, 4), (2, 8), (8, 256), (1, 128), (3, 7), (16, 1024)):
            for cf in (0.0, 0.5, 1.0, 1.25, 1.5, 2.0, 0.3, 1.1, 3.75):
                assert api.expert_capacity(T, k, N, cf) == O.expert_capacity(T, k, N, cf), (T, k, N, cf)
    out = ctypes.c_int64(-5)
    for args in ((4, 0, 4, 1.0), (4, 5, 4, 1.0), (-1, 2, 4, 1.0), (4, 2, 4, -0.5),
                 (4, 2, 4, float("nan")), (4, 2, 4, float("inf")), (2 ** 40, 16, 1, 1.0)):
        assert lib.moe_expert_capacity(*args, ctypes.byref(out)) == api.MOE_ERR_INVALID_ARG, args
    assert out.value == -5
    assert lib.moe_expert_capacity(4, 2, 4, 1.0, None) == api.MOE_ERR_INVALID_ARG
