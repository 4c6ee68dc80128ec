"""The C-ABI library builds for sm_103a, loads without a GPU and exports
every entry point that include/ep_api.h declares; host-only calls work."""
import ctypes
import os
import re

import pytest

from combine_ep_layout_06_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "ep_api.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.load()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["ep_workspace_size", "ep_create", "ep_destroy", "ep_layout",
              "ep_dispatch_send", "ep_dispatch_recv", "ep_dispatch",
              "ep_dispatch_outputs", "ep_get_combine_input_buffer",
              "ep_combine_send", "ep_combine_recv", "ep_combine", "ep_reset",
              "ep_get_error", "ep_status_str"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), n
    assert set(_declared()) <= set(_lib.SIGNATURES)


def test_status_strings(L):
    for code, name in _lib.STATUS_NAMES.items():
        assert L.ep_status_str(code).decode() == name


def _cfg(**kw):
    base = dict(world_size=8, num_experts=256, topk=8, hidden=7168,
                max_tokens_per_rank=4096, max_recv_tokens_per_rank=0,
                dispatch_dtype=0, early_notify=0, fused_recv=0, combine_dtype=0,
                wait_timeout_ns=0)
    base.update(kw)
    return _lib.EpConfigC(**base)


def _size(L, **kw):
    n = ctypes.c_size_t(0)
    c = _cfg(**kw)
    st = L.ep_workspace_size(ctypes.byref(c), ctypes.byref(n))
    return st, n.value


def test_workspace_size_and_config_validation(L):
    st, n = _size(L)
    assert st == 0
    W, T, H, k = 8, 4096, 7168, 8
    cap = W * T
    # receive payload + registered combine buffer dominate
    assert n >= W * cap * H * 2 * 2
    assert n < W * cap * (H * 2 * 2 + 4096) + (1 << 26)
    st8, n8 = _size(L, dispatch_dtype=1)
    assert st8 == 0 and n8 < n
    bad = [dict(world_size=0), dict(world_size=33), dict(num_experts=255),
           dict(topk=0), dict(topk=33), dict(hidden=7170), dict(hidden=0),
           dict(max_tokens_per_rank=0), dict(dispatch_dtype=1, hidden=7168 + 8),
           dict(dispatch_dtype=7), dict(max_recv_tokens_per_rank=-1),
           dict(fused_recv=1, early_notify=0), dict(combine_dtype=1, hidden=7176),
           dict(combine_dtype=5), dict(hidden=(1 << 24) + 8),
           dict(hidden=1 << 25), dict(dispatch_dtype=1, hidden=16384 + 128)]
    for b in bad:
        assert _size(L, **b)[0] == 3, b      # EP_ERR_INVALID_ARGS
    assert _size(L, max_recv_tokens_per_rank=100)[1] < n
    st32, n32 = _size(L, combine_dtype=2)         # fp32 combine rows
    assert st32 == 0 and n32 > n


def test_create_rejects_bad_workspace_without_touching_the_gpu(L):
    c = _cfg()
    h = ctypes.c_void_p()
    assert L.ep_create(ctypes.byref(c), None, 0, ctypes.byref(h)) == 3
    assert L.ep_create(ctypes.byref(c), ctypes.c_void_p(0x1001), 1 << 40,
                       ctypes.byref(h)) == 3          # not 256-byte aligned
    assert L.ep_destroy(None) == 3


def test_hidden_size_upper_bound(L):
    """H up to 2^24 is accepted (a row's byte count stays in an int), above
    it the config is rejected."""
    st, n = _size(L, hidden=1 << 24, max_tokens_per_rank=1, world_size=1,
                  num_experts=1, topk=1)
    assert st == 0 and n >= (1 << 24) * 2 * 2
    assert _size(L, hidden=(1 << 24) + 8, max_tokens_per_rank=1, world_size=1,
                 num_experts=1, topk=1)[0] == 3


def test_nvtx_build_switch_compiles(tmp_path):
    """The entry points' NVTX ranges (compiled in with -DEP_NVTX=1, off in
    the default build) compile for sm_103a."""
    import subprocess
    src = os.path.join(ROOT, "combine_ep_layout_06_gb300", "csrc", "ep_api.cu")
    cmd = [build._nvcc(), *build.NVCC_FLAGS, "-DEP_NVTX=1", "-c", src,
           "-o", str(tmp_path / "ep_api_nvtx.o")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
