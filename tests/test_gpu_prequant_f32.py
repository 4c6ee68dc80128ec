"""GPU parity of the pre-quantised FP8 pass-through dispatch (the pages'
dispatch takes `scales` beside `input`; a backend "can carry
already-quantized FP8 payloads") and of the fp32 combine input, against the
CPU oracle.  Integer / byte results bit-exact; combine output within 1 bf16
ulp and expected bit-exact (same ascending-rank fp32 order)."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_06_gb300 import inputs as gen
from gpu_helpers import bits, make_op, to_device, ulp_diff_bf16

pytestmark = pytest.mark.gpu


def _run_prequant(op, inp, x8, sc, split=False):
    _, w, idx = to_device(inp)
    dx = torch.from_numpy(x8).cuda()
    ds = torch.from_numpy(sc).cuda()
    nt = [int(n) for n in inp.num_tokens]
    if split:
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        s1.wait_stream(torch.cuda.current_stream())
        op.dispatch_send(dx, w, ds, idx, num_tokens=nt, stream=s1)
        op.dispatch_recv(stream=s2)
        op.identity_expert(stream=s2)
        op.combine_send(stream=s2)
        out, out_w = op.combine_recv(weights=op.out_w, indices=idx, stream=s1)
        torch.cuda.current_stream().wait_stream(s1)
    else:
        op.dispatch(dx, w, ds, idx, num_tokens=nt)
        op.identity_expert()
        out, out_w = op.combine(weights=op.out_w, indices=idx)
    torch.cuda.synchronize()
    return out, out_w


def _check_combined(wl, inp, out, out_w, exp, exp_w):
    got = bits(out)
    for s in range(wl.world_size):
        n = int(inp.num_tokens[s])
        assert ulp_diff_bf16(got[s, :n], exp[s, :n]).max(initial=0) <= 1
        assert np.array_equal(got[s, :n], exp[s, :n])
        assert np.array_equal(out_w[s, :n].cpu().numpy().view(np.uint32),
                              exp_w[s, :n].view(np.uint32))


@pytest.mark.parametrize("T,H,ragged", [(200, 7168, False), (200, 7168, True),
                                        (45, 384, True), (40, 16384, False)])
def test_prequant_dispatch_parity(T, H, ragged):
    wl = gen.WORKLOADS["dsv3_fp8_zipf"].scaled(T, hidden=H)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl) if ragged else None)
    x8, sc = gen.draw_fp8_payload(wl, seed=T + H)
    op = make_op(wl)
    out, out_w = _run_prequant(op, inp, x8, sc)
    cap = op.cap
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    ref = oracle.dispatch_prequant(wl, x8, sc, inp.weights, inp.indices,
                                   inp.num_tokens, pos, cap)
    assert np.array_equal(op.pos.cpu().numpy(), pos)
    assert np.array_equal(op.recv_count.cpu().numpy(), rc)
    got_out = bits(op.out)
    got_sc = op.out_scales.cpu().numpy()
    for r in range(wl.world_size):
        n = rc[r]
        assert np.array_equal(got_out[r, :n], ref["out"][r, :n])
        assert np.array_equal(got_sc[r, :n].view(np.uint32), ref["out_scales"][r, :n].view(np.uint32))
        assert np.array_equal(op.src_pos.cpu().numpy()[r, :n], ref["src_pos"][r, :n])
        assert np.array_equal(op.out_idx.cpu().numpy()[r, :n], ref["out_idx"][r, :n])
    y = oracle.identity_expert(wl, rc, ref["out"], ref["out_scales"], ref["out_w"],
                               ref["out_idx"], cap, fp8=True)
    assert all(np.array_equal(bits(op.combine_input)[r, :rc[r]], y[r, :rc[r]])
               for r in range(wl.world_size))
    exp, exp_w = oracle.combine(wl, inp.num_tokens, pos, y, ref["out_w"], cap)
    _check_combined(wl, inp, out, out_w, exp, exp_w)
    assert op.get_error() == (0, 0)


@pytest.mark.parametrize("name,ragged", [("dsv3", False), ("dsv3", True),
                                         ("dsv3_fp8_zipf", True), ("mixtral", False),
                                         ("ll_decode", True)])
def test_fp32_combine_parity(name, ragged):
    T = {"dsv3": 150, "dsv3_fp8_zipf": 150, "mixtral": 200, "ll_decode": 128}[name]
    wl = gen.WORKLOADS[name].scaled(T, hidden=1024)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl) if ragged else None)
    _check_fp32_combine(wl, inp)


@pytest.mark.parametrize("W,E,k", [(16, 32, 12), (32, 64, 32)])
def test_fp32_combine_wide_topk(W, E, k):
    """More than 8 destination ranks per token: the 16- and 32-row fp32 gathers."""
    wl = gen.Workload("wide", W, E, k, 40, 256)
    _check_fp32_combine(wl, gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl)))


def _check_fp32_combine(wl, inp):
    op = make_op(wl, combine_dtype="fp32")
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx, num_tokens=[int(n) for n in inp.num_tokens])
    op.identity_expert()
    out, out_w = op.combine(weights=op.out_w, indices=idx)
    torch.cuda.synchronize()
    res = oracle.run_all(inp, cap=op.cap)
    y32 = oracle.identity_expert_f32(wl, res["recv_count"], res["out"], res["out_scales"],
                                     res["out_w"], res["out_idx"], op.cap)
    gy = op.combine_input.cpu().numpy()
    for r in range(wl.world_size):
        n = res["recv_count"][r]
        assert np.array_equal(gy[r, :n].view(np.uint32), y32[r, :n].view(np.uint32))
    exp, exp_w = oracle.combine_f32(wl, inp.num_tokens, res["pos"], y32, res["out_w"], op.cap)
    _check_combined(wl, inp, out, out_w, exp, exp_w)


def test_prequant_split_streams_with_fp32_combine():
    wl = gen.WORKLOADS["ll_decode"].scaled(128, hidden=2048)
    wl = gen.dataclasses.replace(wl, fp8=True)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
    x8, sc = gen.draw_fp8_payload(wl, seed=3)
    outs = []
    for kw in [dict(), dict(early_notify=True, fused_recv=True)]:
        op = make_op(wl, combine_dtype="fp32", **kw)
        out, out_w = _run_prequant(op, inp, x8, sc, split=bool(kw))
        outs.append((bits(out), out_w.cpu().numpy()))
        assert op.get_error() == (0, 0)
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    cap = wl.world_size * wl.max_tokens_per_rank
    ref = oracle.dispatch_prequant(wl, x8, sc, inp.weights, inp.indices,
                                   inp.num_tokens, pos, cap)
    y32 = oracle.identity_expert_f32(wl, rc, ref["out"], ref["out_scales"], ref["out_w"],
                                     ref["out_idx"], cap, fp8=True)
    exp, exp_w = oracle.combine_f32(wl, inp.num_tokens, pos, y32, ref["out_w"], cap)
    for got, gw in outs:
        for s in range(wl.world_size):
            n = int(inp.num_tokens[s])
            assert np.array_equal(got[s, :n], exp[s, :n])
            assert np.array_equal(gw[s, :n].view(np.uint32), exp_w[s, :n].view(np.uint32))


def test_prequant_needs_fp8_dispatch_and_matching_shapes():
    wl = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(wl)
    op = make_op(wl)                    # bf16 dispatch
    x, w, idx = to_device(inp)
    sc = torch.ones((2, 128, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        op.dispatch(x.view(torch.uint8)[..., :256], w, sc, idx)
    import ctypes
    nt = (ctypes.c_int32 * 2)(128, 128)
    P = ctypes.c_void_p
    st = P(torch.cuda.current_stream().cuda_stream)
    assert op.L.ep_dispatch(op.h, P(x.data_ptr()), P(w.data_ptr()), P(sc.data_ptr()),
                            P(idx.data_ptr()), nt, st) == 3
