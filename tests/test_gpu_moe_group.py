"""GPU parity of the standard-MoE conversion (per-local-expert grouping of
the received rows and the weighted un-grouping before combine) against the
CPU oracle: layout, slots and copied rows bit-exact, un-grouped rows and
the combined output bit-exact (same fp32 order)."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_06_gb300 import inputs as gen
from gpu_helpers import bits, make_op, to_device

pytestmark = pytest.mark.gpu


def _group_and_check(wl, inp, gcap=0, dup=False, random_y=False):
    W, k = wl.world_size, wl.topk
    cap = W * wl.max_tokens_per_rank
    gcap = gcap or cap * k
    op = make_op(wl, max_grouped_rows_per_rank=gcap)
    x, w, idx = to_device(inp)
    nt = [int(n) for n in inp.num_tokens]
    op.dispatch(x, w, None, idx, num_tokens=nt)
    op.moe_group()
    torch.cuda.synchronize()
    res = oracle.run_all(inp, cap=cap)
    count, offset, slot = oracle.expert_layout(wl, res["recv_count"], res["out_idx"], cap)
    assert np.array_equal(op.moe_count.cpu().numpy(), count)
    assert np.array_equal(op.moe_offset.cpu().numpy(), offset)
    got_slot = op.moe_entry_slot.cpu().numpy()
    assert np.array_equal(got_slot, slot)
    xg, xs, src, gw = oracle.group_rows(wl, res["recv_count"], res["out"], res["out_scales"],
                                        res["out_w"], slot, cap, gcap)
    used = [min(int(count[r].sum()), gcap) for r in range(W)]
    gx, gsrc, gww = bits(op.moe_x), op.moe_src.cpu().numpy(), op.moe_w.cpu().numpy()
    for r in range(W):
        n = used[r]
        assert np.array_equal(gx[r, :n], xg[r, :n])
        assert np.array_equal(gsrc[r, :n], src[r, :n])
        assert np.array_equal(gww[r, :n].view(np.uint32), gw[r, :n].view(np.uint32))
        if wl.fp8:
            assert np.array_equal(op.moe_x_scales.cpu().numpy()[r, :n].view(np.uint32),
                                  xs[r, :n].view(np.uint32))
    # expert outputs: identity copies of the grouped bf16 rows, or seeded rows
    if random_y or wl.fp8:
        g = torch.Generator().manual_seed(5)
        yg = torch.randn((W, gcap, wl.hidden), generator=g).to(torch.bfloat16)
        yg_bits = bits(yg)
        op.moe_y.copy_(yg.cuda())
    else:
        op.moe_y.copy_(op.moe_x)
        yg_bits = xg
    op.moe_ungroup()
    out, out_w = op.combine(weights=op.out_w)
    torch.cuda.synchronize()
    y = oracle.ungroup(wl, res["recv_count"], res["out_w"], slot, yg_bits, cap, gcap)
    gy = bits(op.combine_input)
    for r in range(W):
        n = min(res["recv_count"][r], cap)
        assert np.array_equal(gy[r, :n], y[r, :n]), r
    exp, _ = oracle.combine(wl, inp.num_tokens, res["pos"], y, None, cap)
    got = bits(out)
    for s in range(W):
        n = int(inp.num_tokens[s])
        assert np.array_equal(got[s, :n], exp[s, :n])
    return op, count


@pytest.mark.parametrize("name,T,H,ragged", [
    ("tiny", 128, 256, False), ("dsv3", 100, 1024, True), ("mixtral", 200, 512, False),
    ("ll_decode", 128, 512, True), ("dsv3_fp8_zipf", 90, 512, True)])
def test_moe_grouping_parity(name, T, H, ragged):
    wl = gen.WORKLOADS[name].scaled(T, hidden=H)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl) if ragged else None)
    op, count = _group_and_check(wl, inp)
    assert op.get_error() == (0, 0)


@pytest.mark.parametrize("W,E,k", [(2, 32, 12), (2, 64, 32)])
def test_moe_grouping_many_entries_per_row(W, E, k):
    """Rows holding more than 8 entries: the un-grouping's 16- and 32-entry
    bodies (and, with duplicates, up to k entries of one expert)."""
    wl = gen.Workload("many", W, E, k, 60, 256)
    inp = gen.make_inputs(wl)
    if k > E // W:
        rng = np.random.default_rng(3)
        inp.indices[...] = rng.integers(0, E, size=inp.indices.shape)
    op, _ = _group_and_check(wl, inp, random_y=True)
    assert op.get_error() == (0, 0)


def test_moe_grouping_duplicates_and_random_expert_outputs():
    wl = gen.Workload("dupg", 4, 16, 5, 70, 256)
    inp = gen.make_inputs(wl)
    rng = np.random.default_rng(11)
    inp.indices[...] = rng.integers(0, 16, size=inp.indices.shape)
    op, _ = _group_and_check(wl, inp, random_y=True)
    assert op.get_error() == (0, 0)


def test_moe_grouping_capacity_overflow_is_bounded():
    wl = gen.WORKLOADS["dsv3"].scaled(64, hidden=256)
    inp = gen.make_inputs(wl)
    res = oracle.run_all(inp)
    count, _, _ = oracle.expert_layout(wl, res["recv_count"], res["out_idx"], res["cap"])
    gcap = int(count.sum(axis=1).min()) - 5          # every rank overflows a little
    op, _ = _group_and_check(wl, inp, gcap=gcap)
    st, mask = op.get_error()
    assert st == 9 and mask & 0x2


def test_moe_ungroup_needs_a_grouping():
    from combine_ep_layout_06_gb300 import EpError
    wl = gen.WORKLOADS["tiny"]
    op = make_op(wl, max_grouped_rows_per_rank=512)
    with pytest.raises(EpError) as e:
        op.moe_ungroup()
    assert e.value.status == 6
    inp = gen.make_inputs(wl)
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    op.moe_group()
    op.dispatch(x, w, None, idx)                      # a new dispatch drops it
    with pytest.raises(EpError):
        op.moe_ungroup()
