"""Full-size parity of the next rows, at the sizes the benchmark times:
the pre-quantised FP8 pass-through dispatch (whole receive buffers against
the oracle's copy), the standard-MoE grouping (counts, offsets and every
entry slot in full; grouped rows sampled) and un-grouping (every row), the
FP8 combine payload and the scatter combine (every combined token)."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_06_gb300 import inputs as gen
from gpu_helpers import bits, make_op, to_device

pytestmark = pytest.mark.gpu


def test_fullsize_prequant_dispatch():
    wl = gen.WORKLOADS["dsv3_fp8_zipf"]
    inp = gen.make_inputs(wl)
    x8, sc = gen.draw_fp8_payload(wl)
    op = make_op(wl)
    _, w, idx = to_device(inp)
    op.dispatch(torch.from_numpy(x8).cuda(), w, torch.from_numpy(sc).cuda(), idx)
    torch.cuda.synchronize()
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    assert np.array_equal(op.pos.cpu().numpy(), pos)
    ref = oracle.dispatch_prequant(wl, x8, sc, inp.weights, inp.indices, inp.num_tokens,
                                   pos, op.cap)
    for r in range(wl.world_size):
        n = int(rc[r])
        assert np.array_equal(op.out[r, :n].cpu().numpy(), ref["out"][r, :n])
        assert np.array_equal(op.out_scales[r, :n].cpu().numpy().view(np.uint32),
                              ref["out_scales"][r, :n].view(np.uint32))
        assert np.array_equal(op.src_pos[r, :n].cpu().numpy(), ref["src_pos"][r, :n])
    assert op.get_error() == (0, 0)


def test_fullsize_moe_grouping():
    wl = gen.WORKLOADS["dsv3"]
    inp = gen.make_inputs(wl)
    gcap = 40960
    op = make_op(wl, max_grouped_rows_per_rank=gcap)
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    op.moe_group()
    torch.cuda.synchronize()
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    meta = oracle.dispatch(wl, inp.x_bits, inp.weights, inp.indices, inp.num_tokens, pos,
                           op.cap, payload=False)
    count, offset, slot = oracle.expert_layout(wl, rc, meta["out_idx"], op.cap)
    assert np.array_equal(op.moe_count.cpu().numpy(), count)
    assert np.array_equal(op.moe_offset.cpu().numpy(), offset)
    assert np.array_equal(op.moe_entry_slot.cpu().numpy(), slot)
    assert op.get_error() == (0, 0)
    # sampled grouped rows: slot q of rank r holds received row p = src // k
    rng = np.random.default_rng(4)
    src = op.moe_src.cpu().numpy()
    gw = op.moe_w.cpu().numpy()
    for r in range(wl.world_size):
        n = int(count[r].sum())
        for q in rng.integers(0, n, size=12):
            p, j = divmod(int(src[r, q]), wl.topk)
            assert slot[r, p, j] == q
            assert gw[r, q] == meta["out_w"][r, p, j]
            d = oracle.dispatch_rows(wl, inp.x_bits, inp.weights, inp.indices,
                                     inp.num_tokens, pos, [r], [p])
            assert np.array_equal(bits(op.moe_x[r, int(q)]), d["out"][0])


def test_fullsize_fp8_combine_payload():
    """The FP8 combine payload at full size (DeepSeek-V3 shape, the
    3-CTA-per-SM form): the identity expert's codes and scales and every
    combined token against the oracle."""
    wl = gen.WORKLOADS["dsv3"]
    inp = gen.make_inputs(wl)
    op = make_op(wl, combine_dtype="fp8_e4m3")
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    op.identity_expert()
    out, out_w = op.combine(weights=op.out_w, indices=idx)
    torch.cuda.synchronize()
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    cap = int(rc.max())
    d = oracle.dispatch(wl, inp.x_bits, inp.weights, inp.indices, inp.num_tokens, pos, cap)
    yq, ysc = oracle.identity_expert_fp8(wl, rc, d["out"], d["out_scales"], d["out_w"],
                                         d["out_idx"], cap)
    for r in range(wl.world_size):
        n = int(rc[r])
        assert np.array_equal(op.combine_input[r, :n].cpu().numpy(), yq[r, :n]), r
        assert np.array_equal(op.combine_input_scales[r, :n].cpu().numpy().view(np.uint32),
                              ysc[r, :n].view(np.uint32)), r
    exp, exp_w = oracle.combine_fp8(wl, inp.num_tokens, pos, yq, ysc, d["out_w"], cap)
    assert np.array_equal(bits(out), exp)
    assert np.array_equal(out_w.cpu().numpy().view(np.uint32), exp_w.view(np.uint32))
    assert op.get_error() == (0, 0)


def test_fullsize_scatter_combine():
    """The scatter combine at full size (DeepSeek-V3 shape): every combined
    token and its weights against the oracle's ordered sum."""
    wl = gen.WORKLOADS["dsv3"]
    inp = gen.make_inputs(wl)
    op = make_op(wl, combine_mode="scatter")
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    op.identity_expert()
    out, out_w = op.combine(weights=op.out_w, indices=idx)
    torch.cuda.synchronize()
    rc = oracle.layout(wl, inp.indices, inp.num_tokens)[2]
    ref = oracle.run_all(inp, cap=int(rc.max()))
    assert np.array_equal(bits(out), ref["combined"])
    assert np.array_equal(out_w.cpu().numpy().view(np.uint32),
                          ref["combined_w"].view(np.uint32))
    assert op.get_error() == (0, 0)


def test_fullsize_moe_ungroup():
    """Standard-MoE un-grouping at full size (DeepSeek-V3 shape): with the
    grouped rows as the experts' output, every received row of the combine
    input against the oracle's weighted per-row sum, then every combined
    token."""
    wl = gen.WORKLOADS["dsv3"]
    inp = gen.make_inputs(wl)
    gcap = 40960
    op = make_op(wl, max_grouped_rows_per_rank=gcap)
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    op.moe_group()
    op.moe_y.copy_(op.moe_x)                     # identity experts on the grouped rows
    op.moe_ungroup()
    out, _ = op.combine(indices=idx)
    torch.cuda.synchronize()
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    cap = op.cap
    meta = oracle.dispatch(wl, inp.x_bits, inp.weights, inp.indices, inp.num_tokens, pos,
                           cap, payload=False)
    count, offset, slot = oracle.expert_layout(wl, rc, meta["out_idx"], cap)
    yg = bits(op.moe_y)                          # [W][gcap][H], checked by the grouping test
    y = oracle.ungroup(wl, rc, meta["out_w"], slot, yg, cap, gcap)
    got = bits(op.combine_input)
    for r in range(wl.world_size):
        n = int(rc[r])
        assert np.array_equal(got[r, :n], y[r, :n]), r
    exp, _ = oracle.combine(wl, inp.num_tokens, pos, y, None, cap)
    assert np.array_equal(bits(out), exp)
    assert op.get_error() == (0, 0)
