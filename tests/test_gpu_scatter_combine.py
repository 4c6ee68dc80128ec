"""GPU parity of the scatter combine (the expert side pushes each received
row's output to a per-token staging area; the source side reduces the staged
rows in ascending rank order): output bit-exact against the oracle's combine
(the same ordered fp32 sum), staging rows bit-exact against their definition,
fused and split paths equal."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_06_gb300 import inputs as gen
from gpu_helpers import bits, make_op, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T,H,ragged", [
    ("tiny", 128, 256, True), ("dsv3", 150, 1024, False), ("dsv3", 150, 7168, True),
    ("mixtral", 200, 512, False), ("ll_decode", 128, 512, True)])
def test_scatter_combine_parity(name, T, H, ragged):
    wl = gen.WORKLOADS[name].scaled(T, hidden=H)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl) if ragged else None)
    op = make_op(wl, combine_mode="scatter")
    res = run_gpu(op, inp)
    ref = oracle.run_all(inp, cap=op.cap)
    for s in range(wl.world_size):
        n = int(inp.num_tokens[s])
        assert np.array_equal(res["combined"][s, :n], ref["combined"][s, :n])
        assert np.array_equal(res["combined_w"][s, :n].view(np.uint32),
                              ref["combined_w"][s, :n].view(np.uint32))
    # the staging area: token (s,t)'s d-th destination row is y_r[pos]
    stage = bits(op.combine_stage)            # [W][T][maxd][H]
    for s in range(wl.world_size):
        for t in range(int(inp.num_tokens[s])):
            dests = [r for r in range(wl.world_size) if ref["pos"][s, t, r] >= 0]
            for d, r in enumerate(dests):
                assert np.array_equal(stage[s, t, d], ref["y"][r, ref["pos"][s, t, r]])
    assert op.get_error() == (0, 0)


def test_scatter_split_streams_and_fused_receive_equal_gather():
    wl = gen.WORKLOADS["ll_decode"].scaled(128, hidden=2048)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
    gather = run_gpu(make_op(wl), inp)
    for kw in [dict(), dict(early_notify=True), dict(early_notify=True, fused_recv=True)]:
        op = make_op(wl, combine_mode="scatter", **kw)
        res = run_gpu(op, inp, split=True)
        for s in range(wl.world_size):
            n = int(inp.num_tokens[s])
            assert np.array_equal(res["combined"][s, :n], gather["combined"][s, :n])
        assert op.get_error() == (0, 0)


def test_scatter_mode_needs_bf16_registered_rows():
    from combine_ep_layout_06_gb300 import EpError
    wl = gen.WORKLOADS["tiny"]
    with pytest.raises(EpError):
        make_op(wl, combine_mode="scatter", combine_dtype="fp32")
    op = make_op(wl, combine_mode="scatter")
    inp = gen.make_inputs(wl)
    run_gpu(op, inp)
    with pytest.raises(EpError):
        op.combine(input=torch.zeros_like(op.combine_input))
