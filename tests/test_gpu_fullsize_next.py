"""Full-size parity of the next rows, at the sizes the benchmark times:
the pre-quantised FP8 pass-through dispatch (whole receive buffers against
the oracle's copy) and the standard-MoE grouping (counts, offsets and every
entry slot in full; grouped rows sampled)."""
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
