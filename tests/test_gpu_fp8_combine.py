"""GPU parity of the FP8 combine payload (expert rows as E4M3 codes plus
one fp32 scale per 128 elements, dequantised as fl32(value(q) * scale) and
summed in ascending rank order) against the CPU oracle: the identity
expert's codes and scales bit-exact, the combined output bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_06_gb300 import inputs as gen
from gpu_helpers import bits, make_op, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T,H,ragged", [
    ("dsv3", 150, 1024, False), ("dsv3", 150, 7168, True), ("dsv3_fp8_zipf", 120, 1024, True),
    ("mixtral", 200, 512, False), ("ll_decode", 128, 384, True), ("tiny", 128, 256, True),
    ("dsv3", 640, 1024, False), ("mixtral", 640, 512, True)])   # > 4096 tokens: the 3-CTA form
def test_fp8_combine_payload_parity(name, T, H, ragged):
    wl = gen.WORKLOADS[name].scaled(T, hidden=H)
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl) if ragged else None)
    _check_fp8_combine(wl, inp)


def test_fp8_combine_payload_wide_topk():
    """32 destination ranks per token: the 32-row FP8 gather."""
    wl = gen.Workload("wide", 32, 64, 32, 40, 256)
    _check_fp8_combine(wl, gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl)))


def _check_fp8_combine(wl, inp):
    op = make_op(wl, combine_dtype="fp8_e4m3")
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx, num_tokens=[int(n) for n in inp.num_tokens])
    op.identity_expert()
    out, out_w = op.combine(weights=op.out_w, indices=idx)
    torch.cuda.synchronize()
    res = oracle.run_all(inp, cap=op.cap)
    yq, ysc = oracle.identity_expert_fp8(wl, res["recv_count"], res["out"], res["out_scales"],
                                         res["out_w"], res["out_idx"], op.cap)
    gq = op.combine_input.cpu().numpy()
    gs = op.combine_input_scales.cpu().numpy()
    for r in range(wl.world_size):
        n = res["recv_count"][r]
        assert np.array_equal(gq[r, :n], yq[r, :n]), r
        assert np.array_equal(gs[r, :n].view(np.uint32), ysc[r, :n].view(np.uint32)), r
    exp, exp_w = oracle.combine_fp8(wl, inp.num_tokens, res["pos"], yq, ysc, res["out_w"], op.cap)
    got = bits(out)
    for s in range(wl.world_size):
        n = int(inp.num_tokens[s])
        assert np.array_equal(got[s, :n], exp[s, :n])
        assert np.array_equal(out_w[s, :n].cpu().numpy().view(np.uint32),
                              exp_w[s, :n].view(np.uint32))
    assert op.get_error() == (0, 0)


def test_fp8_combine_payload_split_and_fused_receive():
    wl = gen.WORKLOADS["ll_decode"].scaled(128, hidden=1024)
    inp = gen.make_inputs(wl)
    x, w, idx = to_device(inp)
    outs = []
    for kw in [dict(), dict(early_notify=True, fused_recv=True)]:
        op = make_op(wl, combine_dtype="fp8_e4m3", **kw)
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        s1.wait_stream(torch.cuda.current_stream())
        op.dispatch_send(x, w, None, idx, stream=s1)
        op.dispatch_recv(stream=s2)
        op.identity_expert(stream=s2)
        op.combine_send(stream=s2)
        out, _ = op.combine_recv(stream=s1)
        torch.cuda.synchronize()
        outs.append(bits(out))
        assert op.get_error() == (0, 0)
    assert np.array_equal(outs[0], outs[1])


def test_fp8_combine_rejects_user_rows_and_bad_hidden():
    from combine_ep_layout_06_gb300 import EpError
    wl = gen.WORKLOADS["tiny"]
    op = make_op(wl, combine_dtype="fp8_e4m3")
    inp = gen.make_inputs(wl)
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    with pytest.raises(ValueError):
        op.combine(input=torch.zeros_like(op.combine_input))
    with pytest.raises(EpError):
        make_op(gen.Workload("h", 2, 8, 2, 16, 200), combine_dtype="fp8_e4m3")


def test_fp8_combine_every_code_and_extreme_scales():
    """Codes and scales written straight into the registered buffer: every
    E4M3 code (subnormals, signed zeros, and the NaN codes in odd rows only,
    so that even rows carry no NaN) under scales from 2^-149 to 2^126,
    subnormal, zero and overflowing products included.  The combined output
    equals the oracle's bit for bit; where the oracle's sum is NaN the
    device's is NaN as well (a NaN's payload bits are not fixed)."""
    wl = gen.Workload("codes", 4, 16, 4, 64, 512)
    inp = gen.make_inputs(wl)
    op = make_op(wl, combine_dtype="fp8_e4m3")
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    torch.cuda.synchronize()
    W, cap, H = wl.world_size, op.cap, wl.hidden
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, size=(W, cap, H)).astype(np.uint8)
    codes[:, :, :256] = np.arange(256, dtype=np.uint8)
    even = codes[:, 0::2]
    even[(even & 0x7F) == 0x7F] -= 1                  # no NaN code in even rows
    codes[:, 0::2] = even
    nb = H // 128
    exps = rng.integers(-149, 127, size=(W, cap, nb))
    scales = np.ldexp(rng.uniform(1.0, 2.0, size=(W, cap, nb)), exps).astype(np.float32)
    special = np.array([0.0, 2.0 ** -149, 2.0 ** -126, np.nextafter(np.float32(256), 0),
                        256.0, 2.0 ** 126], np.float32)
    scales[:, :special.size, 0] = special
    scales[:, :, 1] = np.ldexp(np.float32(1.5), rng.integers(-20, 12, size=(W, cap)))
    op.combine_input.copy_(torch.from_numpy(codes))
    op.combine_input_scales.copy_(torch.from_numpy(scales))
    out, out_w = op.combine(weights=op.out_w, indices=idx)
    torch.cuda.synchronize()
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    exp, exp_w = oracle.combine_fp8(wl, inp.num_tokens, pos, codes, scales,
                                    op.out_w.cpu().numpy(), cap)
    got = bits(out)
    isnan = lambda b: ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)   # noqa: E731
    assert np.array_equal(isnan(got), isnan(exp))
    ok = ~isnan(exp)
    assert np.array_equal(got[ok], exp[ok])
    assert isnan(exp).any() and ok.any()
    assert op.get_error() == (0, 0)
