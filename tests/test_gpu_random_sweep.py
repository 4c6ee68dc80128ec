"""A seeded sweep of random shapes and options, each compared with the CPU
oracle element by element: world sizes 1..32, experts per rank 1..8, top-k
1..12, ragged token counts with empty ranks, hidden sizes from 8 to 2048,
duplicate experts, receive capacities below the worst case (overflow
reported and the kept rows exact), the fused FP8 dispatch, fp32 and FP8
combine input, scatter combine, split phases with early notification and
the fused receive."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_06_gb300 import inputs as gen
from gpu_helpers import bits, make_op, run_gpu, to_device
from test_gpu_parity import _compare

pytestmark = pytest.mark.gpu

N_CASES = 40


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    while True:
        W = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 24, 32]))
        Er = int(rng.choice([1, 2, 4, 8]))
        E = W * Er
        k = int(rng.integers(1, min(E, 12) + 1))
        T = int(rng.integers(1, 201))
        fp8 = bool(rng.random() < 0.3)
        H = int(rng.choice([128, 256, 384, 1024, 2048])) if fp8 else \
            int(rng.choice([8, 16, 24, 136, 256, 1000, 2048]))
        if W * W * T * H <= 24_000_000:
            break
    opts = {}
    mode = int(rng.integers(0, 6))
    if mode == 1:
        opts["combine_dtype"] = "fp32"
    elif mode == 2 and H % 128 == 0:
        opts["combine_dtype"] = "fp8_e4m3"
    elif mode == 3:
        opts["combine_mode"] = "scatter"
    elif mode == 4:
        opts.update(early_notify=True, fused_recv=True)
    split = bool(rng.random() < 0.3)
    wl = gen.Workload(f"sweep{seed}", W, E, k, T, H, fp8=fp8, seed=seed)
    nt = rng.integers(0, T + 1, size=W).astype(np.int32)
    if W > 1 and rng.random() < 0.5:
        nt[rng.integers(0, W)] = 0
    nt[rng.integers(0, W)] = T
    inp = gen.make_inputs(wl, num_tokens=nt)
    if rng.random() < 0.2:                       # duplicate experts inside a token
        inp.indices[...] = rng.integers(0, E, size=inp.indices.shape)
    cap = 0
    if rng.random() < 0.2:
        rc = oracle.layout(wl, inp.indices, inp.num_tokens)[2]
        cap = max(1, int(rc.max()) - int(rng.integers(0, 5)))
    return wl, inp, cap, opts, split


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_shapes_and_options(seed):
    wl, inp, cap, opts, split = _case(seed)
    op = make_op(wl, cap=cap, **opts)
    eff_cap = op.cap
    rc = oracle.layout(wl, inp.indices, inp.num_tokens)[2]
    overflow = bool((rc > eff_cap).any())
    ydt = opts.get("combine_dtype", "bf16")
    if ydt == "bf16":
        res = run_gpu(op, inp, split=split)
        _compare(wl, inp, res, eff_cap)
    else:
        x, w, idx = to_device(inp)
        nt = [int(n) for n in inp.num_tokens]
        op.dispatch(x, w, None, idx, num_tokens=nt)
        op.identity_expert()
        out, out_w = op.combine(weights=op.out_w, indices=idx)
        torch.cuda.synchronize()
        pos, C, rcount = oracle.layout(wl, inp.indices, inp.num_tokens)
        d = oracle.dispatch(wl, inp.x_bits, inp.weights, inp.indices, inp.num_tokens, pos,
                            eff_cap)
        if ydt == "fp32":
            y = oracle.identity_expert_f32(wl, rcount, d["out"], d["out_scales"], d["out_w"],
                                           d["out_idx"], eff_cap)
            exp, exp_w = oracle.combine_f32(wl, inp.num_tokens, pos, y, d["out_w"], eff_cap)
        else:
            yq, ysc = oracle.identity_expert_fp8(wl, rcount, d["out"], d["out_scales"],
                                                 d["out_w"], d["out_idx"], eff_cap)
            exp, exp_w = oracle.combine_fp8(wl, inp.num_tokens, pos, yq, ysc, d["out_w"],
                                            eff_cap)
        got = bits(out)
        got_w = out_w.cpu().numpy()
        for s in range(wl.world_size):
            n = int(inp.num_tokens[s])
            assert np.array_equal(got[s, :n], exp[s, :n]), s
            assert np.array_equal(got_w[s, :n].view(np.uint32), exp_w[s, :n].view(np.uint32)), s
    st, mask = op.get_error()
    bad_ids = bool(((inp.indices < 0) | (inp.indices >= wl.num_experts)).any())
    assert not bad_ids
    assert (mask & 0x2 != 0) == overflow       # EP_DEVERR_CAPACITY exactly when a rank overflows
    assert mask & ~0x2 == 0
