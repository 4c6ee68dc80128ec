"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars (from the method's definition): layout, counts, positions, src_pos,
carried weights / ids, bf16 payloads, FP8 codes and scales, and the identity
expert's rows are bit-exact; combine is within 1 bf16 ulp (relative error
<= 2^-8) and, because both sides add in the same ascending-rank fp32 order,
is expected bit-exact as well (checked separately).

Sizes: every workload's routing recipe at token counts the oracle finishes in
seconds (several 32-token layout chunks and a ragged tail), plus the
full-size DeepSeek-V3-shaped and FP8 workloads in the launch configuration
the benchmark times, checked on sampled rows and tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_06_gb300 import inputs as gen
from gpu_helpers import make_op, run_gpu, ulp_diff_bf16, to_device, bits

pytestmark = pytest.mark.gpu


def _compare(wl, inp, res, cap, exact_combine=True):
    ref = oracle.run_all(inp, cap=cap)
    assert np.array_equal(res["recv_count"], ref["recv_count"])
    assert np.array_equal(res["send_counts"], ref["C"])
    assert np.array_equal(res["pos"], ref["pos"])
    for r in range(wl.world_size):
        n = min(int(ref["recv_count"][r]), cap)
        assert np.array_equal(res["src_pos"][r, :n], ref["src_pos"][r, :n])
        assert np.array_equal(res["out_w"][r, :n].view(np.uint32),
                              ref["out_w"][r, :n].view(np.uint32))
        assert np.array_equal(res["out_idx"][r, :n], ref["out_idx"][r, :n])
        assert np.array_equal(res["out"][r, :n], ref["out"][r, :n]), r
        if wl.fp8:
            assert np.array_equal(res["out_scales"][r, :n].view(np.uint32),
                                  ref["out_scales"][r, :n].view(np.uint32))
        assert np.array_equal(res["y"][r, :n], ref["y"][r, :n]), r
    for s in range(wl.world_size):
        n = int(inp.num_tokens[s])
        got, exp = res["combined"][s, :n], ref["combined"][s, :n]
        assert ulp_diff_bf16(got, exp).max(initial=0) <= 1
        if exact_combine:
            assert np.array_equal(got, exp)
        assert np.array_equal(res["combined_w"][s, :n].view(np.uint32),
                              ref["combined_w"][s, :n].view(np.uint32))
    return ref


SMALL = {
    # name: (T, H)
    "tiny": (128, 256),
    "dsv3": (200, 7168),
    "dsv3_fp8_zipf": (200, 7168),
    "ll_decode": (128, 7168),
    "mixtral": (300, 4096),
}


@pytest.mark.parametrize("ragged", [False, True])
@pytest.mark.parametrize("name", list(SMALL))
def test_parity_all_workloads(name, ragged):
    T, H = SMALL[name]
    wl = gen.WORKLOADS[name].scaled(T, hidden=H)
    nt = gen.ragged_num_tokens(wl) if ragged else None
    inp = gen.make_inputs(wl, num_tokens=nt)
    op = make_op(wl)
    res = run_gpu(op, inp)
    _compare(wl, inp, res, op.cap)
    if name == "mixtral" and not ragged:
        assert res["recv_count"][6] == 0 and res["recv_count"][7] == 0


@pytest.mark.parametrize("H,fp8", [(264, False), (8, False), (384, True),
                                   (128, True), (16384, True)])
def test_parity_ragged_hidden_sizes(H, fp8):
    """Row lengths that are not a whole number of warp-wide vectors, an odd
    number of FP8 blocks, one block, and the largest FP8 row."""
    wl = gen.Workload("h", 4, 16, 3, 45, H, fp8=fp8)
    inp = gen.make_inputs(wl, num_tokens=[45, 17, 0, 33])
    op = make_op(wl)
    _compare(wl, inp, run_gpu(op, inp), op.cap)


def test_parity_fp8_special_blocks():
    """All-zero blocks, -0 inside nonzero blocks, values at the saturation
    boundary and tiny values that round to FP8 subnormals or zero."""
    wl = gen.Workload("fp8s", 2, 4, 2, 40, 512, fp8=True)
    inp = gen.make_inputs(wl)
    xb = inp.x_bits
    xb[0, 0, :] = 0                          # all blocks zero
    xb[0, 1, 128:256] = 0x8000               # a block of -0 only
    xb[0, 2, 5] = 0x8000                     # -0 in a nonzero block
    xb[1, 3, :128] = 0x3F80                  # all 1.0: every code 0x7E
    xb[1, 4, 0] = 0x4780                     # 65536 next to N(0,1) values
    xb[1, 5, 256:384] = 0x0001               # smallest subnormal bf16s
    xb[1, 5, 300] = 0x3F80
    op = make_op(wl)
    _compare(wl, inp, run_gpu(op, inp), op.cap)


def test_parity_single_rank_and_top1():
    for wl in [gen.Workload("w1", 1, 4, 2, 70, 256),
               gen.Workload("k1", 5, 10, 1, 70, 256),
               gen.Workload("all", 4, 4, 4, 70, 256)]:
        inp = gen.make_inputs(wl)
        op = make_op(wl)
        _compare(wl, inp, run_gpu(op, inp), op.cap)


def test_parity_duplicate_experts_and_wide_world():
    wl = gen.Workload("dup", 32, 64, 6, 40, 128)
    inp = gen.make_inputs(wl)
    rng = np.random.default_rng(2)
    inp.indices[...] = rng.integers(0, 64, size=inp.indices.shape)  # duplicates
    op = make_op(wl)
    _compare(wl, inp, run_gpu(op, inp), op.cap)


@pytest.mark.parametrize("W,E,k,fp8", [(16, 32, 12, False), (32, 64, 32, False),
                                        (32, 64, 32, True)])
def test_parity_wide_topk(W, E, k, fp8):
    """More than 8 destination ranks per token: the combine's 16- and 32-row
    gathers, one stream and split with the fused receive."""
    wl = gen.Workload("wide", W, E, k, 40, 256, fp8=fp8)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
    op = make_op(wl)
    _compare(wl, inp, run_gpu(op, inp), op.cap)
    op2 = make_op(wl, early_notify=True, fused_recv=True)
    _compare(wl, inp, run_gpu(op2, inp, split=True), op2.cap)
    assert op.get_error() == (0, 0) and op2.get_error() == (0, 0)


def test_parity_long_rows_take_the_register_copy():
    """bf16 rows of 88 KB do not fit the bulk copy's shared-memory ring; the
    register copy moves them."""
    wl = gen.Workload("long", 2, 4, 2, 40, 45056)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
    op = make_op(wl)
    _compare(wl, inp, run_gpu(op, inp), op.cap)
    assert op.get_error() == (0, 0)


def test_empty_batch():
    wl = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(wl, num_tokens=[0, 0])
    op = make_op(wl)
    res = run_gpu(op, inp)
    assert res["recv_count"].tolist() == [0, 0]
    assert np.all(res["pos"] == -1)
    assert np.all(res["send_counts"] == 0)


def test_split_streams_equal_fused_path():
    wl = gen.WORKLOADS["ll_decode"]
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
    fused = run_gpu(make_op(wl), inp)
    for kw in [dict(), dict(early_notify=True),
               dict(early_notify=True, fused_recv=True)]:
        op = make_op(wl, **kw)
        split = run_gpu(op, inp, split=True)
        for key in fused:
            if fused[key] is None:
                continue
            if key in ("out", "y", "src_pos", "out_w", "out_idx"):
                for r in range(wl.world_size):
                    n = fused["recv_count"][r]
                    assert np.array_equal(fused[key][r, :n], split[key][r, :n]), key
            elif key in ("combined", "combined_w"):
                for s in range(wl.world_size):
                    n = inp.num_tokens[s]
                    assert np.array_equal(fused[key][s, :n], split[key][s, :n]), key
            else:
                assert np.array_equal(fused[key], split[key]), key
        st, mask = op.get_error()
        assert st == 0 and mask == 0
        if kw.get("early_notify"):
            # every (destination, source) pair was notified, zero-count ones too
            assert np.all(op.dispatch_flags.cpu().numpy() == op.epochs()[0])
            assert np.all(op.combine_flags.cpu().numpy() == op.epochs()[1])


def test_determinism_repeated_runs():
    wl = gen.WORKLOADS["dsv3"].scaled(256, hidden=1024)
    inp = gen.make_inputs(wl)
    op = make_op(wl)
    first = run_gpu(op, inp)
    for _ in range(9):
        again = run_gpu(op, inp)
        for key, v in first.items():
            if v is not None:
                assert np.array_equal(v, again[key]), key


def test_routing_replay_equals_full_dispatch():
    wl = gen.WORKLOADS["dsv3"].scaled(96, hidden=512)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
    op = make_op(wl)
    x, w, idx = to_device(inp)
    nt = [int(n) for n in inp.num_tokens]
    op.layout(idx, num_tokens=nt)
    x2 = torch.randn_like(x, dtype=torch.float32).to(torch.bfloat16)
    op.dispatch_send_replay(x2, w, idx, num_tokens=nt)
    op.dispatch_recv()
    torch.cuda.synchronize()
    replay_out = bits(op.out).copy()
    inp2 = gen.Inputs(wl, bits(x2).reshape(inp.x_bits.shape), inp.weights,
                      inp.indices, inp.num_tokens)
    ref = oracle.run_all(inp2, cap=op.cap)
    for r in range(wl.world_size):
        n = ref["recv_count"][r]
        assert np.array_equal(replay_out[r, :n], ref["out"][r, :n])


def test_graph_capture_replay_equals_eager():
    wl = gen.WORKLOADS["ll_decode"]
    inp = gen.make_inputs(wl)
    op = make_op(wl)
    x, w, idx = to_device(inp)
    nt = [int(n) for n in inp.num_tokens]
    eager = run_gpu(op, inp)
    out = torch.empty((wl.world_size, wl.max_tokens_per_rank, wl.hidden),
                      dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        op.dispatch(x, w, None, idx, num_tokens=nt, stream=s)   # warm-up
        op.combine(out=out, stream=s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            op.dispatch(x, w, None, idx, num_tokens=nt, stream=s)
            op.identity_expert(stream=s)
            op.combine(out=out, stream=s)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), eager["combined"])
    assert np.array_equal(op.recv_count.cpu().numpy(), eager["recv_count"])


def test_routing_replay_after_one_call_dispatch():
    """The one-call dispatch computes its layout inside the copy kernel and
    leaves it for routing replay."""
    wl = gen.WORKLOADS["dsv3"].scaled(96, hidden=512)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
    op = make_op(wl)
    x, w, idx = to_device(inp)
    nt = [int(n) for n in inp.num_tokens]
    op.dispatch(x, w, None, idx, num_tokens=nt)
    x2 = torch.randn_like(x, dtype=torch.float32).to(torch.bfloat16)
    op.dispatch_send_replay(x2, w, idx, num_tokens=nt)
    op.dispatch_recv()
    torch.cuda.synchronize()
    inp2 = gen.Inputs(wl, bits(x2).reshape(inp.x_bits.shape), inp.weights,
                      inp.indices, inp.num_tokens)
    ref = oracle.run_all(inp2, cap=op.cap)
    assert np.array_equal(op.pos.cpu().numpy(), ref["pos"])
    assert np.array_equal(op.send_counts.cpu().numpy(), ref["C"])
    out = bits(op.out)
    for r in range(wl.world_size):
        n = ref["recv_count"][r]
        assert np.array_equal(out[r, :n], ref["out"][r, :n])


@pytest.mark.parametrize("fp8", [False, True])
def test_routing_replay_after_a_dispatch_that_computed_its_own_layout(fp8):
    """At most 8 chunks of 32 tokens the copy kernel computes the layout
    itself, and its CTA 0 writes the layout state (masks, chunk offsets,
    group bases, send counts, recv_count) that routing replay, the receive
    step and combine read: a replay with new rows and an early-notification
    receive must then give the oracle's results."""
    wl = gen.Workload("self", 4, 16, 3, 60, 256, fp8=fp8)       # 4 x 2 = 8 chunks
    inp = gen.make_inputs(wl, num_tokens=[60, 33, 0, 51])
    for kw in (dict(), dict(early_notify=True)):
        op = make_op(wl, **kw)
        x, w, idx = to_device(inp)
        nt = [int(n) for n in inp.num_tokens]
        op.dispatch(x, w, None, idx, num_tokens=nt)
        x2 = torch.randn_like(x, dtype=torch.float32).to(torch.bfloat16)
        op.dispatch_send_replay(x2, w, idx, num_tokens=nt)
        op.dispatch_recv()
        op.identity_expert()
        out, out_w = op.combine(weights=op.out_w, indices=idx)
        torch.cuda.synchronize()
        inp2 = gen.Inputs(wl, bits(x2).reshape(inp.x_bits.shape), inp.weights,
                          inp.indices, inp.num_tokens)
        ref = oracle.run_all(inp2, cap=op.cap)
        assert np.array_equal(op.recv_count.cpu().numpy(), ref["recv_count"])
        assert np.array_equal(op.send_counts.cpu().numpy(), ref["C"])
        assert np.array_equal(op.pos.cpu().numpy(), ref["pos"])
        got_out = bits(op.out)
        for r in range(wl.world_size):
            n = int(ref["recv_count"][r])
            assert np.array_equal(got_out[r, :n], ref["out"][r, :n]), r
        got = bits(out)
        for s_ in range(wl.world_size):
            n = int(inp.num_tokens[s_])
            assert np.array_equal(got[s_, :n], ref["combined"][s_, :n]), s_
        assert op.get_error() == (0, 0)


@pytest.mark.parametrize("name,fp8", [("ll_decode", False), ("dsv3", False), ("dsv3", True)])
def test_captured_graph_replayed_on_new_routing(name, fp8):
    """A captured one-call dispatch + combine replayed after the inputs were
    overwritten in place (new tokens and routing, same shapes) gives the new
    inputs' results: nothing of an earlier replay's layout is taken for the
    current one."""
    wl = gen.WORKLOADS[name].scaled(128 if name == "ll_decode" else 200, hidden=1024)
    wl = gen.dataclasses.replace(wl, fp8=fp8)
    inps = [gen.make_inputs(wl, seed=sd) for sd in (0, 7, 0)]
    op = make_op(wl)
    x, w, idx = to_device(inps[0])
    nt = [int(n) for n in inps[0].num_tokens]
    out = torch.empty((wl.world_size, wl.max_tokens_per_rank, wl.hidden),
                      dtype=torch.bfloat16, device="cuda")
    out_w = torch.empty((wl.world_size, wl.max_tokens_per_rank, wl.topk), device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        op.dispatch(x, w, None, idx, num_tokens=nt, stream=s)   # warm-up
        op.identity_expert(stream=s)
        op.combine(weights=op.out_w, out=out, out_weights=out_w, stream=s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            op.dispatch(x, w, None, idx, num_tokens=nt, stream=s)
            op.identity_expert(stream=s)
            op.combine(weights=op.out_w, out=out, out_weights=out_w, stream=s)
    for inp in inps:
        x2, w2, idx2 = to_device(inp)
        x.copy_(x2)
        w.copy_(w2)
        idx.copy_(idx2)
        out.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        res = oracle.run_all(inp, cap=op.cap)
        assert np.array_equal(op.recv_count.cpu().numpy(), res["recv_count"])
        assert np.array_equal(op.pos.cpu().numpy(), res["pos"])
        got = bits(out)
        for s_ in range(wl.world_size):
            n = int(inp.num_tokens[s_])
            assert np.array_equal(got[s_, :n], res["combined"][s_, :n]), s_
    assert op.get_error() == (0, 0)


# --------------------------------------------------------------- full size

def _compare_per_rank(wl, inp, op, res, ref):
    """Every received row and every combined token of a large case, rank by
    rank (the device rows are fetched one rank at a time)."""
    assert np.array_equal(res["recv_count"], ref["recv_count"])
    assert np.array_equal(res["send_counts"], ref["C"])
    assert np.array_equal(res["pos"], ref["pos"])
    for r in range(wl.world_size):
        n = int(ref["recv_count"][r])
        assert np.array_equal(res["src_pos"][r, :n], ref["src_pos"][r, :n]), r
        assert np.array_equal(res["out_idx"][r, :n], ref["out_idx"][r, :n]), r
        assert np.array_equal(res["out_w"][r, :n].view(np.uint32),
                              ref["out_w"][r, :n].view(np.uint32)), r
        assert np.array_equal(bits(op.out[r, :n]), ref["out"][r, :n]), r
        if wl.fp8:
            assert np.array_equal(bits(op.out_scales[r, :n]),
                                  ref["out_scales"][r, :n].view(np.uint32)), r
        assert np.array_equal(bits(op.combine_input[r, :n]), ref["y"][r, :n]), r
    for s in range(wl.world_size):
        n = int(inp.num_tokens[s])
        assert np.array_equal(res["combined"][s, :n], ref["combined"][s, :n]), s
        assert np.array_equal(res["combined_w"][s, :n].view(np.uint32),
                              ref["combined_w"][s, :n].view(np.uint32)), s


@pytest.mark.parametrize("name", ["dsv3", "dsv3_fp8_zipf", "mixtral"])
def test_parity_full_size_every_token(name):
    """The benchmark's workloads at full size, in the launch configuration the
    benchmark times (one-call dispatch, then the gather above 4096 tokens),
    compared with the oracle on everything: layout, every received row with
    its metadata, every identity-expert row and every combined token."""
    wl = gen.WORKLOADS[name]
    inp = gen.make_inputs(wl)
    rc = oracle.layout(wl, inp.indices, inp.num_tokens)[2]
    ref = oracle.run_all(inp, cap=int(rc.max()))   # rows past the counts stay out
    op = make_op(wl)
    res = run_gpu(op, inp, payload=False)
    _compare_per_rank(wl, inp, op, res, ref)
    assert op.get_error() == (0, 0)


@pytest.mark.parametrize("ragged", [False, True])
@pytest.mark.parametrize("name", ["dsv3", "dsv3_fp8_zipf", "mixtral", "ll_decode"])
def test_parity_above_the_few_token_switch(name, ragged):
    """More than 4096 tokens (the combine's switch between its few-token and
    bandwidth forms) at a reduced hidden size, compared element by element."""
    wl = gen.WORKLOADS[name]
    wl = wl.scaled(640 if wl.world_size == 8 else 320, hidden=1024)
    nt = gen.ragged_num_tokens(wl) if ragged else None
    if ragged:                     # keep more than 4096 present tokens
        nt = np.maximum(nt, wl.max_tokens_per_rank - 40)
        nt[-1] = 0
    inp = gen.make_inputs(wl, num_tokens=nt)
    assert int(inp.num_tokens.sum()) > 4096
    op = make_op(wl)
    _compare(wl, inp, run_gpu(op, inp), op.cap)


def test_capacity_overflow_is_bounded_and_reported():
    wl = gen.WORKLOADS["dsv3_fp8_zipf"].scaled(128, hidden=256)
    inp = gen.make_inputs(wl)
    ref_rc = oracle.layout(wl, inp.indices, inp.num_tokens)[2]
    cap = int(np.sort(ref_rc)[len(ref_rc) // 2])       # half the ranks overflow
    op = make_op(wl, cap=cap)
    op.workspace.fill_(0xAB)                          # sentinel everywhere
    op.reset()
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    torch.cuda.synchronize()
    # the buffer after src_pos in every segment is untouched by dispatch
    assert np.all(bits(op.combine_input) == 0xABAB)
    st, mask = op.get_error()
    assert st == 9 and mask & 0x2                     # EP_ERR_CAPACITY
    res = run_gpu(op, inp)
    # rows < cap exact (an overflowing write would corrupt the next buffer
    # of the segment, which is compared too); dropped rows match the oracle
    _compare(wl, inp, res, cap)


@pytest.mark.parametrize("name,fp8", [("dsv3", False), ("dsv3_fp8_zipf", True), ("ll_decode", False)])
def test_receive_rows_past_the_count_are_untouched(name, fp8):
    """Every byte of the workspace starts as a sentinel; after a dispatch the
    receive rows at or past recv_count[r] (payload, scales, weights, ids,
    src_pos) still hold it: the copy writes exactly the counted rows."""
    wl = gen.WORKLOADS[name].scaled(96, hidden=1024)
    wl = gen.dataclasses.replace(wl, fp8=fp8)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
    op = make_op(wl)
    op.workspace.fill_(0xAB)
    op.reset()
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx, num_tokens=[int(n) for n in inp.num_tokens])
    torch.cuda.synchronize()
    rc = op.recv_count.cpu().numpy()
    assert int(rc.sum()) > 0
    views = [op.out, op.out_w, op.out_idx, op.src_pos] + ([op.out_scales] if fp8 else [])
    for r in range(wl.world_size):
        n = int(rc[r])
        for v in views:
            tail = v[r, n:].contiguous().view(torch.uint8).cpu().numpy()
            assert np.all(tail == 0xAB), (r, v.shape)
            head = v[r, :n].contiguous().view(torch.uint8).cpu().numpy()
            assert n == 0 or not np.all(head == 0xAB)
    assert op.get_error() == (0, 0)


def test_bad_expert_index_is_ignored_and_reported():
    wl = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(wl)
    good = inp.indices.copy()
    bad = inp.indices.copy()
    bad[0, 5, 1] = wl.num_experts + 3                 # out of range
    bad[1, 7, 0] = -1
    op = make_op(wl)
    x, w, _ = to_device(inp)
    op.dispatch(x, w, None, torch.from_numpy(bad).cuda())
    torch.cuda.synchronize()
    st, mask = op.get_error()
    assert st == 10 and mask & 0x1                    # EP_ERR_BAD_INDEX
    # same destination sets as replacing the bad entry by a valid duplicate
    good[0, 5, 1] = good[0, 5, 0]
    good[1, 7, 0] = good[1, 7, 1]
    pos, C, rc = oracle.layout(wl, good, inp.num_tokens)
    assert np.array_equal(op.pos.cpu().numpy(), pos)
    assert np.array_equal(op.recv_count.cpu().numpy(), rc)


def test_combine_index_mismatch_is_reported():
    wl = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(wl)
    op = make_op(wl)
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    other = idx.clone()
    ref_pos = oracle.layout(wl, inp.indices, inp.num_tokens)[0]
    if (ref_pos[0, 0] >= 0).all():
        other[0, 0, :] = torch.tensor([0, 1], dtype=torch.int32)   # rank {0}
    else:
        other[0, 0, :] = torch.tensor([0, 4], dtype=torch.int32)   # ranks {0,1}
    op.combine(indices=other)
    st, mask = op.get_error()
    assert st == 6 and mask & 0x8
    op.combine(indices=idx)
    assert op.get_error() == (0, 0)


def test_out_of_order_calls_return_bad_state():
    from combine_ep_layout_06_gb300 import EpError
    wl = gen.WORKLOADS["tiny"]
    op = make_op(wl)
    inp = gen.make_inputs(wl)
    x, w, idx = to_device(inp)
    with pytest.raises(EpError) as e:
        op.combine()
    assert e.value.status == 6
    with pytest.raises(EpError) as e:
        op.dispatch_recv()
    assert e.value.status == 6
    with pytest.raises(EpError) as e:
        op.combine_recv()
    assert e.value.status == 6
    op.dispatch(x, w, None, idx)
    op.combine()
    op.reset()
    with pytest.raises(EpError) as e:
        op.combine()
    assert e.value.status == 6
    op.dispatch_send(x, w, None, idx)
    with pytest.raises(EpError) as e:
        op.dispatch_send(x, w, None, idx)            # send twice
    assert e.value.status == 6
    # combine while the send waits for its receive phase
    with pytest.raises(EpError) as e:
        op.combine()
    assert e.value.status == 6
    with pytest.raises(EpError) as e:
        op.combine_send()
    assert e.value.status == 6
    op.dispatch_recv()
    op.combine_send()
    with pytest.raises(EpError) as e:
        op.combine_send()                            # combine send twice
    assert e.value.status == 6
    op.combine_recv()
    assert op.get_error() == (0, 0)


def test_get_error_waits_for_its_own_stream_only():
    """ep_get_error reads the error word in its stream's order and waits for
    that stream alone: a long kernel on another stream is still running when
    it returns."""
    wl = gen.WORKLOADS["tiny"]
    op = make_op(wl)
    inp = gen.make_inputs(wl)
    x, w, idx = to_device(inp)
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    op.dispatch(x, w, None, idx, stream=a)
    done_b = torch.cuda.Event()
    with torch.cuda.stream(b):
        torch.cuda._sleep(2_000_000_000)             # about a second of spinning
        done_b.record(b)
    assert op.get_error(a) == (0, 0)
    assert not done_b.query()                        # b was not waited for
    torch.cuda.synchronize()
    assert done_b.query()


def test_host_argument_checks():
    from combine_ep_layout_06_gb300 import EpError
    wl = gen.WORKLOADS["tiny"]
    op = make_op(wl)
    inp = gen.make_inputs(wl)
    x, w, idx = to_device(inp)
    L = op.L
    import ctypes
    nt = (ctypes.c_int32 * 2)(128, 128)
    bad_nt = (ctypes.c_int32 * 2)(129, 0)
    st = torch.cuda.current_stream().cuda_stream
    P = ctypes.c_void_p
    # misaligned x (2 bytes off), num_tokens > T, scales given, null pointers
    assert L.ep_dispatch(op.h, P(x.data_ptr() + 2), P(w.data_ptr()), None,
                         P(idx.data_ptr()), nt, P(st)) == 3
    assert L.ep_dispatch(op.h, P(x.data_ptr()), P(w.data_ptr()), None,
                         P(idx.data_ptr()), bad_nt, P(st)) == 3
    assert L.ep_dispatch(op.h, P(x.data_ptr()), P(w.data_ptr()),
                         P(w.data_ptr()), P(idx.data_ptr()), nt, P(st)) == 3
    assert L.ep_dispatch(op.h, None, P(w.data_ptr()), None,
                         P(idx.data_ptr()), nt, P(st)) == 3
    with pytest.raises(ValueError):
        op.dispatch(x.float(), w, None, idx)


def test_dropped_notification_times_out():
    """A ready flag that the test drops (cleared after the send completed):
    the receive's bounded wait gives up and reports EP_ERR_TIMEOUT, and the
    context stays usable."""
    wl = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(wl)
    op = make_op(wl, early_notify=True, wait_timeout_ns=2_000_000)
    x, w, idx = to_device(inp)
    op.dispatch_send(x, w, None, idx)
    torch.cuda.synchronize()
    op.dispatch_flags[1, 0] = 0                       # drop (0 -> 1)'s notice
    op.dispatch_recv()
    st, mask = op.get_error()
    assert st == 8 and mask & 0x4
    # the combine side: a combine flag dropped before the fused receive
    op2 = make_op(wl, early_notify=True, fused_recv=True,
                  wait_timeout_ns=2_000_000)
    op2.dispatch(x, w, None, idx)
    op2.combine_send()
    torch.cuda.synchronize()
    op2.combine_flags[0, 1] = 0
    op2.combine_recv()
    st, mask = op2.get_error()
    assert st == 8 and mask & 0x4
    # both ops keep working
    res = run_gpu(op2, inp)
    _compare(wl, inp, res, op2.cap)


def test_repeated_steps_alternating_inputs_stay_exact():
    """Sixty back-to-back one-call steps (layout, the copy launched after it,
    combine launched after that), cycling through three routings without
    synchronising in between, each result compared bit for bit with the
    oracle: nothing of one step leaks into the next."""
    wl = gen.WORKLOADS["dsv3"].scaled(256, hidden=1024)
    inps = [gen.make_inputs(wl, seed=sd,
                            num_tokens=gen.ragged_num_tokens(wl, seed=sd) if sd else None)
            for sd in (0, 5, 9)]
    refs = [oracle.run_all(inp, cap=wl.world_size * wl.max_tokens_per_rank) for inp in inps]
    dev = [to_device(inp) for inp in inps]
    nts = [[int(n) for n in inp.num_tokens] for inp in inps]
    op = make_op(wl)
    outs = [torch.empty((wl.world_size, wl.max_tokens_per_rank, wl.hidden),
                        dtype=torch.bfloat16, device="cuda") for _ in range(60)]
    for i in range(60):
        x, w, idx = dev[i % 3]
        op.dispatch(x, w, None, idx, num_tokens=nts[i % 3])
        op.identity_expert()
        op.combine(weights=op.out_w, out=outs[i])
    torch.cuda.synchronize()
    for i in range(60):
        got, ref, inp = bits(outs[i]), refs[i % 3], inps[i % 3]
        for s in range(wl.world_size):
            n = int(inp.num_tokens[s])
            assert np.array_equal(got[s, :n], ref["combined"][s, :n]), (i, s)
    assert op.get_error() == (0, 0)


def test_handles_on_two_host_threads():
    """Two handles with different row sizes driven from two host threads at
    once, each on its own stream: both results exact (the per-device launch
    settings they share are raised, never lowered, under concurrency)."""
    import threading
    cases = []
    for H in (7168, 2048):
        wl = gen.WORKLOADS["dsv3"].scaled(96, hidden=H)
        inp = gen.make_inputs(wl, seed=H)
        cases.append((wl, inp, oracle.run_all(inp, cap=wl.world_size * wl.max_tokens_per_rank)))
    errors = []

    def worker(wl, inp, ref):
        try:
            torch.cuda.set_device(0)
            op = make_op(wl)
            x, w, idx = to_device(inp)
            st = torch.cuda.Stream()
            out = torch.empty((wl.world_size, wl.max_tokens_per_rank, wl.hidden),
                              dtype=torch.bfloat16, device="cuda")
            with torch.cuda.stream(st):
                for _ in range(20):
                    op.dispatch(x, w, None, idx, stream=st)
                    op.identity_expert(stream=st)
                    op.combine(weights=op.out_w, out=out, stream=st)
            st.synchronize()
            if not np.array_equal(bits(out), ref["combined"]):
                errors.append(f"H={wl.hidden}: combined differs")
            if op.get_error(st) != (0, 0):
                errors.append(f"H={wl.hidden}: device error")
        except Exception as e:   # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=c) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
