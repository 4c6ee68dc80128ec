"""The no-allocation layout entry point, ep_layout_noalloc.

It serves callers that cannot allocate device memory or pass a workspace:
code inside another framework's memory pool that only sees raw tensor
pointers, and serving paths where cudaMalloc is forbidden because it can
synchronise the device and can fail under memory pressure.  Its scratch is a
fixed array inside the library, shared by every call, so these tests call it
twice in a row on different layouts and compare each result with the layout
the existing entry points (ep_dispatch through the op) produce; integer
results must be identical.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from combine_ep_layout_06_gb300 import _lib
from combine_ep_layout_06_gb300 import inputs as gen
from gpu_helpers import make_op, to_device

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _noalloc(L, wl, idx, nt):
    W, T = wl.world_size, wl.max_tokens_per_rank
    dev = idx.device
    pos = torch.full((W, T, W), -7, dtype=torch.int32, device=dev)
    sc = torch.full((W, W), -7, dtype=torch.int32, device=dev)
    rc = torch.full((W,), -7, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    counts = (ctypes.c_int32 * W)(*[int(n) for n in nt])
    st = L.ep_layout_noalloc(W, wl.num_experts, wl.topk, T, P(idx.data_ptr()),
                             counts, P(pos.data_ptr()), P(sc.data_ptr()),
                             P(rc.data_ptr()), P(err.data_ptr()),
                             P(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, pos.cpu().numpy(), sc.cpu().numpy(), rc.cpu().numpy(), int(err.item())


def _existing(wl, inp):
    op = make_op(wl)
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx, num_tokens=[int(n) for n in inp.num_tokens])
    torch.cuda.synchronize()
    return (op.pos.cpu().numpy(), op.send_counts.cpu().numpy(),
            op.recv_count.cpu().numpy())


def test_layout_noalloc_matches_existing_entry_point_twice():
    L = _lib.load()
    cases = [
        gen.WORKLOADS["dsv3"].scaled(4096, hidden=8),       # full token count
        gen.WORKLOADS["mixtral"].scaled(2000, hidden=8),    # zero-token ranks
    ]
    for i, wl in enumerate(cases):
        nt = None if i == 0 else gen.ragged_num_tokens(wl)
        inp = gen.make_inputs(wl, num_tokens=nt)
        idx = torch.from_numpy(inp.indices).cuda()
        st, pos, sc, rc, err = _noalloc(L, wl, idx, inp.num_tokens)
        assert st == 0
        ref_pos, ref_sc, ref_rc = _existing(wl, inp)
        assert np.array_equal(rc, ref_rc)
        assert np.array_equal(sc, ref_sc)
        assert np.array_equal(pos, ref_pos)
        assert err == 0


def test_layout_noalloc_at_its_scratch_limit():
    """W = 32 ranks and T = 4128 tokens: exactly the 4128 chunks the scratch
    holds, so the scan covers the whole array; twice in a row, against the
    existing entry point."""
    L = _lib.load()
    wl = gen.Workload("limit", 32, 64, 2, 4128, 8)
    for nt in (None, gen.ragged_num_tokens(wl)):
        inp = gen.make_inputs(wl, num_tokens=nt)
        idx = torch.from_numpy(inp.indices).cuda()
        st, pos, sc, rc, err = _noalloc(L, wl, idx, inp.num_tokens)
        assert st == 0 and err == 0
        ref_pos, ref_sc, ref_rc = _existing(wl, inp)
        assert np.array_equal(rc, ref_rc)
        assert np.array_equal(sc, ref_sc)
        assert np.array_equal(pos, ref_pos)


def test_layout_noalloc_reports_out_of_range_ids():
    """Expert ids outside [0, E) set the error bit and add no destination,
    as in the existing entry point."""
    L = _lib.load()
    wl = gen.WORKLOADS["dsv3"].scaled(300, hidden=8)
    inp = gen.make_inputs(wl)
    inp.indices[0, 5, 1] = wl.num_experts + 3
    inp.indices[3, 299, 0] = -1
    inp.indices[7, 0, :] = 1 << 30                 # a token with no valid id
    idx = torch.from_numpy(inp.indices).cuda()
    st, pos, sc, rc, err = _noalloc(L, wl, idx, inp.num_tokens)
    assert st == 0
    assert err & _lib.EP_DEVERR_BAD_INDEX
    assert np.all(pos[7, 0] == -1)
    ref_pos, ref_sc, ref_rc = _existing(wl, inp)
    assert np.array_equal(rc, ref_rc)
    assert np.array_equal(sc, ref_sc)
    assert np.array_equal(pos, ref_pos)


def test_layout_noalloc_rejects_sizes_beyond_its_scratch():
    L = _lib.load()
    W, T = 32, 4200                       # 32 * ceil(4200/32) = 4224 chunks
    idx = torch.zeros((W, T, 2), dtype=torch.int32, device="cuda")
    out = torch.zeros(W * T * W, dtype=torch.int32, device="cuda")
    counts = (ctypes.c_int32 * W)(*([T] * W))
    st = L.ep_layout_noalloc(W, 64, 2, T, P(idx.data_ptr()), counts,
                             P(out.data_ptr()), P(out.data_ptr()),
                             P(out.data_ptr()), None,
                             P(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.EP_ERR_INVALID_ARGS
