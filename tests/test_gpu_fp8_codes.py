"""Every FP8 code and block scale of the fused quantising dispatch over
16384 rows of H=7168 (117 M elements) against the oracle's E4M3 encoder,
plus rows built to hit exact round-to-nearest ties (block amax 448, so the
scale is exactly 1 and the midpoints between E4M3 values are bf16-exact),
rows of values that land in E4M3's subnormal range, and signed zeros."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_06_gb300 import inputs as gen
from gpu_helpers import make_op, to_device

pytestmark = pytest.mark.gpu


def _tie_row(H, sign):
    mids = [(1 + m / 8 + 1 / 16) * 2.0 ** e for e in range(-6, 8) for m in range(8)]
    row = np.zeros(H, np.float32)
    for b in range(H // 128):
        blk = np.array([448.0] + [sign * v for v in mids], np.float32)
        row[b * 128:b * 128 + blk.size] = blk[:128]
    return row


def test_fused_fp8_codes_match_the_oracle_everywhere():
    H = 7168
    wl = gen.Workload("codes", 2, 2, 1, 8192, H, fp8=True)
    inp = gen.make_inputs(wl)
    xf = np.zeros((4, H), np.float32)
    xf[0] = _tie_row(H, 1.0)
    xf[1] = _tie_row(H, -1.0)
    xf[2] = np.linspace(-1.0, 1.0, H).astype(np.float32) * 2.0 ** -14
    xf[2, ::128] = 1.0                         # amax 1: most values E4M3-subnormal
    xf[3] = -0.0
    xf[3, 7] = 3.0
    inp.x_bits[0, :4] = (xf.view(np.uint32) >> 16).astype(np.uint16)
    op = make_op(wl)
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    torch.cuda.synchronize()
    rc = op.recv_count.cpu().numpy()
    for r in range(2):
        n = int(rc[r])
        src = op.src_pos[r, :n].cpu().numpy()
        s_, t_ = np.divmod(src, wl.max_tokens_per_rank)
        q, sc = oracle.quant_rows(inp.x_bits[s_, t_])
        assert np.array_equal(op.out[r, :n].cpu().numpy(), q), r
        assert np.array_equal(op.out_scales[r, :n].cpu().numpy().view(np.uint32), sc.view(np.uint32))


def _every_value_under(maxima):
    """Blocks of 128 bf16 values: block max A first, then every bf16
    magnitude m <= A with both signs (zero-padded), for each A in maxima."""
    blocks = []
    for a in maxima:
        mags = np.arange(0, a + 1, dtype=np.uint16)
        vals = np.concatenate([mags, mags | np.uint16(0x8000)])
        nblk = -(-vals.size // 127)
        body = np.zeros(nblk * 127, np.uint16)
        body[:vals.size] = vals
        blk = np.empty((nblk, 128), np.uint16)
        blk[:, 0] = a
        blk[:, 1:] = body.reshape(nblk, 127)
        blocks.append(blk)
    return np.concatenate(blocks)


def test_fused_fp8_codes_every_bf16_value_under_many_block_maxima():
    """The quotient x / scale for every bf16 x (|x| <= block max A) under
    510 maxima spanning every bf16 exponent (mantissa all-zero and all-one),
    plus every maximum whose scale A/448 lies near 2^-90, where the kernel
    switches between its reciprocal-and-correction quotient and a plain
    IEEE division."""
    maxima = [(e << 7) | m for e in range(255) for m in (0x00, 0x7F) if (e << 7) | m]
    maxima += [(e << 7) | m for e in range(44, 48) for m in range(128)]
    maxima = sorted(set(maxima))
    blocks = _every_value_under(maxima)
    H = 7168
    per_row = H // 128
    rows = -(-blocks.shape[0] // per_row)
    W = 2
    T = -(-rows // W)
    pad = np.zeros((W * T * per_row - blocks.shape[0], 128), np.uint16)
    x_bits = np.concatenate([blocks, pad]).reshape(W, T, H)
    wl = gen.Workload("every_x", W, 2, 1, T, H, fp8=True)
    inp = gen.make_inputs(wl)
    inp.x_bits[...] = x_bits
    op = make_op(wl)
    x, w, idx = to_device(inp)
    op.dispatch(x, w, None, idx)
    torch.cuda.synchronize()
    rc = op.recv_count.cpu().numpy()
    assert int(rc.sum()) == W * T
    for r in range(W):
        n = int(rc[r])
        src = op.src_pos[r, :n].cpu().numpy()
        s_, t_ = np.divmod(src, wl.max_tokens_per_rank)
        q, sc = oracle.quant_rows(inp.x_bits[s_, t_])
        assert np.array_equal(op.out[r, :n].cpu().numpy(), q), r
        assert np.array_equal(op.out_scales[r, :n].cpu().numpy().view(np.uint32), sc.view(np.uint32))
    assert op.get_error() == (0, 0)


def test_fp8_quotient_and_scale_identities_over_every_bf16_pair():
    """The fused quantisation's arithmetic over every positive finite bf16
    block maximum a and every finite bf16 x with |x| <= a, both signs: the
    block scale equals the IEEE quotient a / 448 for every a, and the E4M3
    code of the dispatch's quotient (reciprocal plus one correction where the
    scale is >= 2^-90, a plain division below) equals the code of the IEEE
    quotient x / scale for every pair.  The library runs the dispatch
    kernel's own device functions; the cast of an IEEE quotient is itself
    pinned to the oracle's encoder by the tests above."""
    import ctypes
    from combine_ep_layout_06_gb300 import _lib
    L = _lib.load()
    counts = torch.zeros(4, dtype=torch.int64, device="cuda")
    st = L.ep_test_fp8_quotient_check(ctypes.c_void_p(counts.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    pairs, code_diff, scale_diff, fast = counts.cpu().tolist()
    n_max = 0x7F7F                               # bf16 0x0001 .. 0x7F7F
    assert pairs == sum(2 * (a + 1) for a in range(1, n_max + 1))
    assert scale_diff == 0
    assert code_diff == 0
    # most pairs take the reciprocal form (scale >= 2^-90, i.e. a >= 448 * 2^-90)
    assert fast > pairs // 2
