"""Pins for the CPU oracle: every check here compares it with something other
than itself -- hand-derived values from the format definitions and a worked
example, torch's CPU casts, a sort-based brute force, closed forms, special
cases that reduce to textbook operations, and invariants of the method.

Method: ROCm MORI "Communication APIs" page, "MORI-EP (Expert Parallelism)",
table "EpDispatchCombineOp methods"; "Validation before tuning" (identity
expert); "EPv2 configuration and lifecycle" (FP8 = OCP E4M3).
"""
import dataclasses
import json
import os

import numpy as np
import pytest
import torch

import bruteforce as bf
import oracle
from combine_ep_layout_06_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((float.fromhex(parts[0]), int(parts[1], 16)))
    return rows


def _f32_bits(v):
    return np.array(v, np.float32).view(np.uint32)


# ----------------------------------------------------------------- scalars

def test_bf16_rne_golden():
    for v, code in _read_table("bf16_rne_definition.txt"):
        got = int(oracle.bf16_rne(np.array([v], np.float32))[0])
        assert got == code, (v.hex(), hex(got), hex(code))


def test_bf16_rne_matches_torch_cast():
    rng = np.random.default_rng(5)
    u = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) < np.float32(3.38e38))]
    # exact ties and near-ties around every kept pattern
    base = rng.integers(0, 2**32, size=1 << 16, dtype=np.uint64).astype(np.uint32)
    ties = ((base & 0xFFFF0000) | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties) & (np.abs(ties) < np.float32(3.38e38))]
    allv = np.concatenate([f, ties])
    ref = bf.torch_bf16_bits(allv)
    assert np.array_equal(oracle.bf16_rne(allv), ref)


def test_e4m3_golden():
    for v, code in _read_table("e4m3_ocp_definition.txt"):
        got = int(oracle.e4m3_encode(np.array([v], np.float32))[0])
        assert got == code, (v.hex(), hex(got), hex(code))


def test_e4m3_value_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]           # drop the two NaNs
    assert np.array_equal(oracle.e4m3_value(codes).view(np.uint32),
                          bf.torch_e4m3_value(codes).view(np.uint32))


def test_e4m3_encode_matches_torch_on_all_bf16_patterns():
    """Every finite bf16 value divided by sampled scales, |v| < 464 (torch's
    cast does not saturate: at 464 and beyond it gives NaN)."""
    pats = np.arange(1 << 16, dtype=np.uint32)
    x = (pats << 16).view(np.float32)
    x = x[np.isfinite(x)]
    rng = np.random.default_rng(7)
    scales = np.concatenate([
        np.float32([1.0, 2.0 ** -6, 7.0 / 448, 0.75, 3.0, 2.0 ** 20]),
        (rng.random(6, dtype=np.float32) * 4 + 1e-3).astype(np.float32)])
    for sc in scales:
        with np.errstate(over="ignore"):
            v = (x / np.float32(sc)).astype(np.float32)
        m = np.abs(v) < 464
        got = oracle.e4m3_encode(v[m])
        assert np.array_equal(got, bf.torch_e4m3(v[m])), sc
        big = v[~m & np.isfinite(v)]
        exp = np.where(np.signbit(big), 0xFE, 0x7E).astype(np.uint8)
        assert np.array_equal(oracle.e4m3_encode(big), exp)


def test_quant_block_golden():
    g = json.load(open(os.path.join(GOLDEN, "fp8_block_hand.json")))
    H = g["H"]
    x = np.zeros(H, np.float32)
    for i, v in g["block0_nonzero"].items():
        x[int(i)] = v
    for i, v in g["block1_nonzero"].items():
        x[128 + int(i)] = v
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)   # all values bf16-exact
    assert np.array_equal(oracle.bf16_to_f32(xb), x)
    q, sc = oracle.quant_rows(xb[None, :])
    assert sc[0].tolist() == g["scales"]
    exp = np.full(H, int(g["other_codes"], 16), np.uint8)
    for i, c in g["block0_codes_nonzero"].items():
        exp[int(i)] = int(c, 16)
    assert np.array_equal(q[0], exp)


def test_quant_properties_random_rows():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 1024)) * rng.choice(
        [1e-6, 1e-2, 1.0, 30.0, 1e4], size=(64, 1))).astype(np.float32)
    xb = bf.torch_bf16_bits(x)
    xf = bf.to_f32(xb)
    q, sc = oracle.quant_rows(xb)
    blocks = np.abs(xf).reshape(64, 8, 128)
    a = blocks.max(axis=2)
    # scale is the IEEE fp32 quotient amax/448
    assert np.array_equal(sc, (a / np.float32(448)).astype(np.float32))
    # the element holding the block amax encodes to +-448
    qa = q.reshape(64, 8, 128)
    am = blocks.argmax(axis=2)
    top = np.take_along_axis(qa, am[..., None], axis=2)[..., 0]
    assert np.all((top == 0x7E) | (top == 0xFE))
    # dequantisation error bound of E4M3 (3 mantissa bits, subnormal 2^-9)
    deq = oracle.e4m3_value(q).reshape(64, 8, 128) * sc[..., None]
    err = np.abs(deq - xf.reshape(64, 8, 128))
    bound = np.abs(xf.reshape(64, 8, 128)) * 2.0 ** -4 + sc[..., None] * 2.0 ** -10
    assert np.all(err <= bound * (1 + 1e-6))
    # brute-force block quantiser (numpy division + torch cast) agrees
    for i in range(0, 64, 7):
        for b in range(8):
            qq, ss = bf.quant_block(xb[i, b * 128:(b + 1) * 128])
            assert ss == sc[i, b]
            assert np.array_equal(qq, q[i, b * 128:(b + 1) * 128])


# ---------------------------------------------------------- hand example

def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_w2_e4_k2.json")))
    wl = gen.Workload("hand", g["W"], g["E"], g["k"], g["T"], g["H"])
    idx = np.array(g["indices"], np.int32)
    w = np.array(g["weights"], np.float32)
    x = np.array(g["x"], np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    nt = np.array(g["num_tokens"], np.int32)
    pos, C, rc = oracle.layout(wl, idx, nt)
    assert pos.tolist() == g["pos"]
    assert C.tolist() == g["send_counts"]
    assert rc.tolist() == g["recv_count"]
    cap = wl.world_size * wl.max_tokens_per_rank
    d = oracle.dispatch(wl, xb, w, idx, nt, pos, cap)
    for r in range(wl.world_size):
        n = rc[r]
        assert d["src_pos"][r, :n].tolist() == g["src_pos"][r]
        for p, sp in enumerate(g["src_pos"][r]):
            s, t = divmod(sp, wl.max_tokens_per_rank)
            assert np.array_equal(d["out"][r, p], xb[s, t])
    y = oracle.identity_expert(wl, rc, d["out"], None, d["out_w"],
                               d["out_idx"], cap)
    out, out_w = oracle.combine(wl, nt, pos, y, d["out_w"], cap)
    for s in range(wl.world_size):
        for t in range(wl.max_tokens_per_rank):
            if g["combined"][s][t] is None:
                continue
            assert oracle.bf16_to_f32(out[s, t]).tolist() == g["combined"][s][t]
            assert out_w[s, t].tolist() == g["combined_weights"][s][t]


# ------------------------------------------------------------- brute force

def _random_case(rng, W, Er, k, T, H, dup=False, fp8=False):
    E = W * Er
    k = min(k, E)
    wl = gen.Workload("rand", W, E, k, T, H, fp8=fp8)
    inp = gen.make_inputs(wl, num_tokens=rng.integers(0, T + 1, size=W),
                          seed=int(rng.integers(1 << 30)))
    if dup:
        inp.indices[...] = rng.integers(0, E, size=inp.indices.shape)
    return wl, inp


def _check_against_bruteforce(wl, inp):
    W, E, T, H, k = (wl.world_size, wl.num_experts, wl.max_tokens_per_rank,
                     wl.hidden, wl.topk)
    res = oracle.run_all(inp)
    cap = res["cap"]
    disp = bf.dispatch(inp.x_bits, inp.weights, inp.indices, inp.num_tokens,
                       W, E, fp8=wl.fp8)
    ys = {}
    for r in range(W):
        d = disp[r]
        n = len(d["rows"])
        assert res["recv_count"][r] == n
        assert np.array_equal(res["src_pos"][r, :n], d["src_pos"])
        assert np.array_equal(res["out_w"][r, :n], d["out_w"])
        assert np.array_equal(res["out_idx"][r, :n], d["out_idx"])
        if n:
            assert np.array_equal(res["out"][r, :n], d["out"])
            if wl.fp8:
                assert np.array_equal(res["out_scales"][r, :n], d["out_scales"])
        ys[r] = bf.identity_expert(d, r, W, E, fp8=wl.fp8)
        for i in range(n):
            assert np.array_equal(res["y"][r, i], ys[r][i])
        # pos is the inverse of the receive list
        for i, (s, t) in enumerate(d["rows"]):
            assert res["pos"][s, t, r] == i
    w_in = {r: disp[r]["out_w"] for r in range(W)}
    out, out_w = bf.combine(disp, ys, w_in, W, T, H, k, inp.num_tokens)
    for (s, t), row in out.items():
        assert np.array_equal(res["combined"][s, t], row), (s, t)
        assert np.array_equal(res["combined_w"][s, t], out_w[(s, t)])
    # absent tokens are routed nowhere
    for s in range(W):
        assert np.all(res["pos"][s, inp.num_tokens[s]:] == -1)


@pytest.mark.parametrize("seed", range(12))
def test_oracle_matches_bruteforce_random_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    W = int(rng.integers(1, 6))
    Er = int(rng.choice([1, 2, 4]))
    k = int(rng.integers(1, 5))
    T = int(rng.choice([1, 2, 7, 13]))
    wl, inp = _random_case(rng, W, Er, k, T, 16, dup=bool(seed % 3 == 0))
    _check_against_bruteforce(wl, inp)


def test_oracle_matches_bruteforce_tiny_workload():
    wl = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
    _check_against_bruteforce(wl, inp)
    _check_against_bruteforce(wl, gen.make_inputs(wl))


@pytest.mark.parametrize("seed", range(3))
def test_oracle_matches_bruteforce_fp8(seed):
    rng = np.random.default_rng(300 + seed)
    wl, inp = _random_case(rng, 3, 2, 2, 5, 256, fp8=True)
    # an all-zero block and a -0 inside a nonzero block
    inp.x_bits[0, 0, :128] = 0
    inp.x_bits[0, 0, 5] = 0x8000
    inp.x_bits[1, 0, 130] = 0x8000
    _check_against_bruteforce(wl, inp)


# -------------------------------------------------- invariants, all workloads

def _reduced(name):
    wl = gen.WORKLOADS[name]
    return wl.scaled(min(wl.max_tokens_per_rank, 512), hidden=256)


@pytest.mark.parametrize("name", list(gen.WORKLOADS))
def test_layout_invariants_all_workloads(name):
    wl = _reduced(name)
    W, T, Er = wl.world_size, wl.max_tokens_per_rank, wl.experts_per_rank
    inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    ranks = inp.indices // Er
    ndest = np.array([[len(set(ranks[s, t])) if t < inp.num_tokens[s] else 0
                       for t in range(T)] for s in range(W)])
    P = ndest.sum()
    assert rc.sum() == P
    assert np.array_equal(C.sum(axis=1), ndest.sum(axis=1))
    assert np.array_equal(C.sum(axis=0), rc)
    cap = W * T
    d = oracle.dispatch(wl, inp.x_bits, inp.weights, inp.indices,
                        inp.num_tokens, pos, cap, fp8=False)
    for r in range(W):
        sp = d["src_pos"][r, :rc[r]]
        assert np.all(np.diff(sp) > 0)                     # stable order
        exp = sorted(s * T + t for s in range(W)
                     for t in range(inp.num_tokens[s]) if r in set(ranks[s, t]))
        assert sp.tolist() == exp                          # bijection
        s_, t_ = np.divmod(sp, T)
        assert np.array_equal(d["out"][r, :rc[r]], inp.x_bits[s_, t_])
        assert np.array_equal(d["out_idx"][r, :rc[r]], inp.indices[s_, t_])
    if name == "mixtral":
        assert rc[6] == 0 and rc[7] == 0
        full = inp.num_tokens[:, None] > np.arange(T)[None, :]
        assert np.all(ndest[full] == 2)


def test_special_case_single_rank_is_identity():
    wl = gen.Workload("w1", 1, 4, 2, 33, 64)
    inp = gen.make_inputs(wl, num_tokens=[29])
    res = oracle.run_all(inp)
    assert res["recv_count"].tolist() == [29]
    assert np.array_equal(res["out"][0, :29], inp.x_bits[0, :29])
    assert res["src_pos"][0, :29].tolist() == list(range(29))
    # combine of a single rank returns the expert output unchanged
    out, _ = oracle.combine(wl, inp.num_tokens, res["pos"], res["y"], None, 33)
    assert np.array_equal(out[0, :29], res["y"][0, :29])


def test_special_case_top1_is_stable_counting_sort():
    wl = gen.Workload("k1", 4, 8, 1, 50, 16)
    inp = gen.make_inputs(wl)
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    dest = (inp.indices[..., 0] // wl.experts_per_rank).reshape(-1)
    order = np.argsort(dest, kind="stable")
    slot = np.empty_like(order)
    starts = np.concatenate([[0], np.cumsum(np.bincount(dest, minlength=4))])
    slot[order] = np.arange(dest.size) - starts[dest[order]]
    got = pos.reshape(-1, 4)[np.arange(dest.size), dest]
    assert np.array_equal(got, slot)
    # with one destination per token combine returns y's row bit-exact
    res = oracle.run_all(inp)
    for g in range(dest.size):
        s, t = divmod(g, 50)
        r = dest[g]
        assert np.array_equal(res["combined"][s, t],
                              res["y"][r, pos[s, t, r]])


def test_special_case_every_token_to_every_rank():
    W = 3
    wl = gen.Workload("all", W, W, W, 9, 16)
    inp = gen.make_inputs(wl, num_tokens=[9, 4, 6])
    res = oracle.run_all(inp)
    src = [s * 9 + t for s in range(W) for t in range(inp.num_tokens[s])]
    for r in range(W):
        assert res["src_pos"][r, :len(src)].tolist() == src


# ------------------------------------------------------------ closed forms

@pytest.mark.parametrize("name", ["tiny", "dsv3", "dsv3_fp8_zipf", "mixtral"])
def test_identity_expert_returns_input(name):
    """With sum_j w = 1 each token's local alphas add to ~1, so combine
    returns x (bf16) or dequant(x) (FP8) within the rounding of one bf16
    product per rank, the fp32 sum and the final bf16 rounding."""
    wl = _reduced(name).scaled(64, hidden=256)
    inp = gen.make_inputs(wl)
    res = oracle.run_all(inp)
    x = bf.to_f32(inp.x_bits)
    out = bf.to_f32(res["combined"])
    if wl.fp8:
        q, sc = oracle.quant_rows(inp.x_bits.reshape(-1, wl.hidden))
        ref = (oracle.e4m3_value(q) * np.repeat(sc, 128, axis=1)).reshape(x.shape)
    else:
        ref = x
    nd = np.array([[len(set(inp.indices[s, t] // wl.experts_per_rank))
                    for t in range(wl.max_tokens_per_rank)]
                   for s in range(wl.world_size)])[..., None]
    tol = np.abs(ref) * (2.0 ** -8 * (nd + 1) + 1e-6)
    assert np.all(np.abs(out - ref) <= tol)


def test_masked_expert_weights_sum_back_exactly():
    wl = _reduced("dsv3").scaled(64, hidden=64)
    inp = gen.make_inputs(wl)
    res = oracle.run_all(inp)
    Er = wl.experts_per_rank
    w_in = res["out_w"].copy()
    for r in range(wl.world_size):
        w_in[r][res["out_idx"][r] // Er != r] = 0.0
    _, out_w = oracle.combine(wl, inp.num_tokens, res["pos"], res["y"], w_in,
                              res["cap"])
    assert np.array_equal(out_w, inp.weights)


def test_combine_within_fp32_bound_of_fp64_sum():
    wl = _reduced("dsv3").scaled(32, hidden=128)
    inp = gen.make_inputs(wl)
    res = oracle.run_all(inp)
    rng = np.random.default_rng(3)
    y = bf.torch_bf16_bits(rng.standard_normal(res["y"].shape).astype(np.float32) * 100)
    out, _ = oracle.combine(wl, inp.num_tokens, res["pos"], y, None, res["cap"])
    yf = bf.to_f32(y).astype(np.float64)
    W, T = wl.world_size, wl.max_tokens_per_rank
    for s in range(W):
        for t in range(T):
            terms = [yf[r, res["pos"][s, t, r]] for r in range(W)
                     if res["pos"][s, t, r] >= 0]
            exact = np.sum(terms, axis=0)
            mag = np.sum(np.abs(terms), axis=0)
            got = bf.to_f32(out[s, t]).astype(np.float64)
            bound = np.abs(exact) * 2.0 ** -8 + mag * len(terms) * 2.0 ** -24 * 1.01
            assert np.all(np.abs(got - exact) <= bound)


def test_validation_rejects_out_of_contract_inputs():
    wl = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(wl)
    bad = inp.indices.copy()
    bad[1, 3, 0] = wl.num_experts
    with pytest.raises(oracle.OracleError):
        oracle.layout(wl, bad, inp.num_tokens)
    with pytest.raises(oracle.OracleError):
        oracle.layout(wl, inp.indices, [wl.max_tokens_per_rank + 1, 0])
    with pytest.raises(oracle.OracleError):
        oracle.validate(dataclasses.replace(wl, num_experts=7), inp.indices,
                        inp.num_tokens)


def test_combine_order_is_ascending_rank():
    """y rows 1, 2^-24, -1 on ranks 0, 1, 2: ascending order gives
    ((0 + 1) + 2^-24) - 1 = 0 (the middle sum ties back to 1.0), while
    descending gives ((0 - 1) + 2^-24) + 1 = 2^-24.  Hand-derived."""
    W = 3
    wl = gen.Workload("order", W, W, W, 1, 8)
    idx = np.array([[[0, 1, 2]], [[0, 1, 2]], [[0, 1, 2]]], np.int32)
    nt = np.array([1, 0, 0], np.int32)
    pos, _, rc = oracle.layout(wl, idx, nt)
    assert pos[0, 0].tolist() == [0, 0, 0]
    vals = np.float32([1.0, 2.0 ** -24, -1.0])
    y = np.zeros((W, W, 8), np.uint16)
    for r in range(W):
        y[r, 0, :] = (np.full(8, vals[r], np.float32).view(np.uint32) >> 16)
    out, _ = oracle.combine(wl, nt, pos, y, None, W)
    assert np.all(out[0, 0] == 0x0000)


@pytest.mark.parametrize("seed", range(4))
def test_combine_matches_bruteforce_wide_range(seed):
    rng = np.random.default_rng(500 + seed)
    wl, inp = _random_case(rng, 5, 2, 4, 9, 32)
    res = oracle.run_all(inp)
    W, E, T, H, k = 5, wl.num_experts, 9, 32, wl.topk
    disp = bf.dispatch(inp.x_bits, inp.weights, inp.indices, inp.num_tokens,
                       W, E)
    mag = 2.0 ** rng.integers(-20, 21, size=res["y"].shape)
    y = bf.torch_bf16_bits((rng.standard_normal(res["y"].shape) * mag)
                           .astype(np.float32))
    ys = {r: [y[r, i] for i in range(len(disp[r]["rows"]))] for r in range(W)}
    out, _ = bf.combine(disp, ys, None, W, T, H, k, inp.num_tokens)
    got, _ = oracle.combine(wl, inp.num_tokens, res["pos"], y, None, res["cap"])
    for (s, t), row in out.items():
        assert np.array_equal(got[s, t], row)


def test_sampled_row_functions_agree_with_whole_buffer_functions():
    """The per-row forms used for full-size sampling give the same rows as
    the whole-buffer forms pinned above."""
    for name in ["dsv3", "dsv3_fp8_zipf"]:
        wl = _reduced(name).scaled(40, hidden=256)
        inp = gen.make_inputs(wl, num_tokens=gen.ragged_num_tokens(wl))
        res = oracle.run_all(inp)
        rng = np.random.default_rng(9)
        rc = res["recv_count"]
        ranks = np.array([r for r in range(wl.world_size) if rc[r] > 0])
        rr = rng.choice(ranks, size=20)
        pp = np.array([rng.integers(0, rc[r]) for r in rr])
        d = oracle.dispatch_rows(wl, inp.x_bits, inp.weights, inp.indices,
                                 inp.num_tokens, res["pos"], rr, pp)
        assert np.array_equal(d["out"], res["out"][rr, pp])
        assert np.array_equal(d["src_pos"], res["src_pos"][rr, pp])
        if wl.fp8:
            assert np.array_equal(d["out_scales"], res["out_scales"][rr, pp])
        y = oracle.identity_rows(wl, rr, d["out"], d["out_scales"], d["out_w"],
                                 d["out_idx"])
        assert np.array_equal(y, res["y"][rr, pp])
        T = wl.max_tokens_per_rank
        for g in rng.choice(wl.world_size * T, size=10):
            s, t = divmod(int(g), T)
            if t >= inp.num_tokens[s]:
                continue
            rows = [res["y"][r, res["pos"][s, t, r]] for r in range(wl.world_size)
                    if res["pos"][s, t, r] >= 0]
            assert np.array_equal(oracle.combine_gathered(np.array(rows)),
                                  res["combined"][s, t])


# ------------------------------------------- pre-quantised FP8, fp32 combine

@pytest.mark.parametrize("seed", range(3))
def test_prequant_dispatch_matches_bruteforce(seed):
    rng = np.random.default_rng(700 + seed)
    wl, inp = _random_case(rng, 4, 2, 3, 11, 256, fp8=True)
    x8, sc = gen.draw_fp8_payload(wl, seed=seed)
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    cap = wl.world_size * wl.max_tokens_per_rank
    d = oracle.dispatch_prequant(wl, x8, sc, inp.weights, inp.indices,
                                 inp.num_tokens, pos, cap)
    ref = bf.dispatch_prequant(x8, sc, inp.weights, inp.indices, inp.num_tokens,
                               wl.world_size, wl.num_experts)
    for r in range(wl.world_size):
        n = len(ref[r]["rows"])
        assert rc[r] == n
        if n:
            assert np.array_equal(d["out"][r, :n], ref[r]["out"])
            assert np.array_equal(d["out_scales"][r, :n].view(np.uint32),
                                  ref[r]["out_scales"].view(np.uint32))
        assert np.array_equal(d["src_pos"][r, :n], ref[r]["src_pos"])
    # quantising first and passing the codes through equals the fused path
    q, s = oracle.quant_rows(inp.x_bits.reshape(-1, wl.hidden))
    d2 = oracle.dispatch_prequant(wl, q.reshape(x8.shape), s.reshape(sc.shape),
                                  inp.weights, inp.indices, inp.num_tokens, pos, cap)
    fused = oracle.dispatch(wl, inp.x_bits, inp.weights, inp.indices,
                            inp.num_tokens, pos, cap)
    for r in range(wl.world_size):
        assert np.array_equal(d2["out"][r, :rc[r]], fused["out"][r, :rc[r]])
        assert np.array_equal(d2["out_scales"][r, :rc[r]], fused["out_scales"][r, :rc[r]])


def test_payload_draw_has_no_nan_codes():
    wl = gen.Workload("p", 2, 4, 2, 16, 256, fp8=True)
    x8, sc = gen.draw_fp8_payload(wl)
    assert not np.any((x8 & 0x7F) == 0x7F)
    assert np.all(sc > 0) and np.all(np.isfinite(oracle.e4m3_value(x8)))


@pytest.mark.parametrize("fp8", [False, True])
def test_fp32_combine_matches_bruteforce(fp8):
    rng = np.random.default_rng(800 + int(fp8))
    wl, inp = _random_case(rng, 5, 2, 4, 9, 256, fp8=fp8)
    res = oracle.run_all(inp)
    W, E, T, H = wl.world_size, wl.num_experts, wl.max_tokens_per_rank, wl.hidden
    cap = res["cap"]
    y32 = oracle.identity_expert_f32(wl, res["recv_count"], res["out"],
                                     res["out_scales"], res["out_w"],
                                     res["out_idx"], cap)
    # rounding the fp32 identity rows to bf16 gives the (pinned) bf16 rows
    for r in range(W):
        n = res["recv_count"][r]
        assert np.array_equal(bf.torch_bf16_bits(y32[r, :n]), res["y"][r, :n])
    disp = bf.dispatch(inp.x_bits, inp.weights, inp.indices, inp.num_tokens,
                       W, E, fp8=fp8)
    ys = {r: bf.identity_expert_f32(disp[r], r, W, E, fp8=fp8) for r in range(W)}
    for r in range(W):
        for i in range(len(ys[r])):
            assert np.array_equal(ys[r][i].view(np.uint32), y32[r, i].view(np.uint32))
    # wide-range fp32 rows: the ordered fp32 sum
    mag = 2.0 ** rng.integers(-30, 31, size=y32.shape)
    yw = (rng.standard_normal(y32.shape) * mag).astype(np.float32)
    ysw = {r: [yw[r, i] for i in range(len(disp[r]["rows"]))] for r in range(W)}
    exp = bf.combine_f32(disp, ysw, W, T, H, inp.num_tokens)
    got, _ = oracle.combine_f32(wl, inp.num_tokens, res["pos"], yw, None, cap)
    for (s, t), row in exp.items():
        assert np.array_equal(got[s, t], row)


def test_fp32_combine_order_is_ascending_rank():
    W = 3
    wl = gen.Workload("order32", W, W, W, 1, 8)
    idx = np.array([[[0, 1, 2]], [[0, 1, 2]], [[0, 1, 2]]], np.int32)
    nt = np.array([1, 0, 0], np.int32)
    pos, _, _ = oracle.layout(wl, idx, nt)
    y = np.zeros((W, W, 8), np.float32)
    y[0, 0] = 1.0
    y[1, 0] = 2.0 ** -24
    y[2, 0] = -1.0
    out, _ = oracle.combine_f32(wl, nt, pos, y, None, W)
    assert np.all(out[0, 0] == 0)


# ------------------------------------------------- standard-MoE conversion

@pytest.mark.parametrize("seed,fp8,dup", [(0, False, False), (1, False, True),
                                          (2, True, False), (3, False, True)])
def test_expert_grouping_matches_bruteforce(seed, fp8, dup):
    rng = np.random.default_rng(900 + seed)
    wl, inp = _random_case(rng, 3, 4, 3, 13, 256 if fp8 else 32, dup=dup, fp8=fp8)
    res = oracle.run_all(inp)
    cap = res["cap"]
    W, Er, k = wl.world_size, wl.experts_per_rank, wl.topk
    count, offset, slot = oracle.expert_layout(wl, res["recv_count"], res["out_idx"], cap)
    gcap = cap * k
    xg, xs, src, gw = oracle.group_rows(wl, res["recv_count"], res["out"],
                                        res["out_scales"], res["out_w"], slot, cap, gcap)
    for r in range(W):
        n = res["recv_count"][r]
        groups = bf.expert_groups(res["out_idx"][r, :n], r, Er)
        q = 0
        for e in range(Er):
            ent = groups.get(e, [])
            assert count[r, e] == len(ent) and offset[r, e] == q
            for (p, j) in ent:
                assert slot[r, p, j] == q
                assert np.array_equal(xg[r, q], res["out"][r, p])
                if fp8:
                    assert np.array_equal(xs[r, q], res["out_scales"][r, p])
                assert src[r, q] == p * k + j and gw[r, q] == res["out_w"][r, p, j]
                q += 1
        assert count[r].sum() == sum(len(v) for v in groups.values())
        nonlocal_ = (res["out_idx"][r, :n] // Er) != r
        assert np.all(slot[r, :n][nonlocal_] == -1) and np.all(slot[r, n:] == -1)
    # un-grouping with arbitrary expert outputs: weighted ordered sums
    yg = bf.torch_bf16_bits(rng.standard_normal((W, gcap, wl.hidden)).astype(np.float32))
    y = oracle.ungroup(wl, res["recv_count"], res["out_w"], slot, yg, cap, gcap)
    for r in range(W):
        for p in range(res["recv_count"][r]):
            pairs = [(res["out_w"][r, p, j], yg[r, slot[r, p, j]]) for j in range(k)
                     if slot[r, p, j] >= 0]
            exp = bf.ungroup_row(None, pairs)
            assert np.array_equal(y[r, p], exp)


def test_grouped_identity_experts_give_back_the_input():
    """Identity experts per entry (yg = xg) un-grouped and combined return x
    within the rounding of the weighted sums."""
    wl = _reduced("dsv3").scaled(48, hidden=128)
    inp = gen.make_inputs(wl)
    res = oracle.run_all(inp)
    cap = res["cap"]
    count, offset, slot = oracle.expert_layout(wl, res["recv_count"], res["out_idx"], cap)
    gcap = cap * wl.topk
    xg, _, _, _ = oracle.group_rows(wl, res["recv_count"], res["out"], None,
                                    res["out_w"], slot, cap, gcap)
    y = oracle.ungroup(wl, res["recv_count"], res["out_w"], slot, xg, cap, gcap)
    out, _ = oracle.combine(wl, inp.num_tokens, res["pos"], y, None, cap)
    x = bf.to_f32(inp.x_bits)
    got = bf.to_f32(out)
    assert np.all(np.abs(got - x) <= np.abs(x) * 2.0 ** -8 * 12)
    # every token's k selections land in exactly one group slot each
    assert count.sum() == wl.world_size * wl.max_tokens_per_rank * wl.topk


# ------------------------------------------------- FP8 combine payload

def test_fp8_quant_of_fp32_rows_matches_numpy_and_torch():
    rng = np.random.default_rng(21)
    v = (rng.standard_normal((20, 512)) * 2.0 ** rng.integers(-30, 30, size=(20, 1))).astype(np.float32)
    v[3, :128] = 0.0
    v[4, 5] = -0.0
    q, sc = oracle.quant_rows_f32(v)
    for i in range(20):
        for b in range(4):
            blk = v[i, b * 128:(b + 1) * 128]
            a = np.float32(np.abs(blk).max())
            if a == 0:
                assert sc[i, b] == 0 and np.all(q[i, b * 128:(b + 1) * 128] == 0)
                continue
            s = np.float32(a / np.float32(448))
            assert sc[i, b] == s
            assert np.array_equal(q[i, b * 128:(b + 1) * 128],
                                  bf.torch_e4m3((blk / s).astype(np.float32)))


@pytest.mark.parametrize("fp8", [False, True])
def test_fp8_combine_payload_matches_bruteforce(fp8):
    rng = np.random.default_rng(1000 + int(fp8))
    wl, inp = _random_case(rng, 4, 2, 3, 10, 256, fp8=fp8)
    res = oracle.run_all(inp)
    W, T, H, cap = wl.world_size, wl.max_tokens_per_rank, wl.hidden, res["cap"]
    yq, ysc = oracle.identity_expert_fp8(wl, res["recv_count"], res["out"], res["out_scales"],
                                         res["out_w"], res["out_idx"], cap)
    y32 = oracle.identity_expert_f32(wl, res["recv_count"], res["out"], res["out_scales"],
                                     res["out_w"], res["out_idx"], cap)
    for r in range(W):
        n = res["recv_count"][r]
        if n:
            q2, s2 = oracle.quant_rows_f32(y32[r, :n])
            assert np.array_equal(yq[r, :n], q2) and np.array_equal(ysc[r, :n], s2)
    deq = (bf.torch_e4m3_value(yq) * np.repeat(ysc, 128, axis=2)).astype(np.float32)
    disp = bf.dispatch(inp.x_bits, inp.weights, inp.indices, inp.num_tokens, W,
                       wl.num_experts, fp8=fp8)
    ys = {r: [deq[r, i] for i in range(len(disp[r]["rows"]))] for r in range(W)}
    exp = bf.combine_f32(disp, ys, W, T, H, inp.num_tokens)
    got, _ = oracle.combine_fp8(wl, inp.num_tokens, res["pos"], yq, ysc, None, cap)
    for (s, t), row in exp.items():
        assert np.array_equal(got[s, t], row)
    # identity closed form: within the E4M3 step of the combined rows
    x = bf.to_f32(inp.x_bits)
    if fp8:
        q, s = oracle.quant_rows(inp.x_bits.reshape(-1, H))
        x = (oracle.e4m3_value(q) * np.repeat(s, 128, axis=1)).reshape(x.shape)
    o = bf.to_f32(got)
    for s_ in range(W):
        n = inp.num_tokens[s_]
        if n == 0:
            continue
        assert np.all(np.abs(o[s_, :n] - x[s_, :n]) <= np.abs(x[s_, :n]) * 0.2 +
                      np.abs(x[s_, :n]).max() * 2.0 ** -9)


def test_input_recipe_properties_at_full_size():
    """The seeded synthetic inputs have the recipe's stated properties at the
    benchmark sizes: distinct top-k experts per token, weights summing to 1
    within fp32, E[|D|] of uniform routing equal to its closed form
    W * (1 - C(E-Er, k) / C(E, k)), Zipf routing visibly skewed across experts
    and ranks,
    Mixtral routing confined to experts 0-5, and x with the stated sigma."""
    from math import comb
    for name in ["dsv3", "dsv3_fp8_zipf", "mixtral"]:
        wl = gen.WORKLOADS[name]
        inp = gen.make_inputs(wl)
        W, E, k, Er = wl.world_size, wl.num_experts, wl.topk, wl.experts_per_rank
        idx = inp.indices.reshape(-1, k)
        srt = np.sort(idx, axis=1)
        assert np.all(srt[:, 1:] != srt[:, :-1]), name           # distinct experts
        assert np.all((idx >= 0) & (idx < E))
        assert np.allclose(inp.weights.sum(axis=-1), 1.0, atol=1e-6), name
        ranks = idx // Er
        nd = np.array([len(set(r)) for r in ranks.tolist()])
        per_rank = np.bincount(np.concatenate([np.unique(r) for r in ranks.tolist()]),
                               minlength=W)
        if name == "dsv3":
            exact = W * (1 - comb(E - Er, k) / comb(E, k))
            assert abs(nd.mean() - exact) < 0.02, (nd.mean(), exact)
            assert per_rank.max() / per_rank.mean() < 1.02
        if name == "dsv3_fp8_zipf":
            assert per_rank.max() / per_rank.mean() > 1.3          # skewed ranks
            cnt = np.bincount(idx.ravel(), minlength=E)
            assert np.sort(cnt)[-1] > 20 * np.median(cnt)          # a few hot experts
        if name == "mixtral":
            assert idx.max() <= 5 and np.all(nd == 2)
        x = (inp.x_bits[0, :512].astype(np.uint32) << 16).view(np.float32)
        sigma = np.sqrt(2.0) if name == "mixtral" else 1.0
        assert abs(x.std() / sigma - 1) < 0.01, (name, x.std())


@pytest.mark.parametrize("fp8", [False, True])
def test_threaded_range_form_equals_whole_buffer_form(fp8):
    """The timed CPU baseline runs the oracle's dispatch, identity expert and
    combine over disjoint token / row ranges on several threads; the result
    is bit-identical to the single whole-buffer calls (the pinned form)."""
    wl = gen.Workload("thr", 4, 16, 3, 97, 256, fp8=fp8)
    inp = gen.make_inputs(wl, num_tokens=[97, 40, 0, 61])
    ref = oracle.run_all(inp)
    cap = ref["cap"]
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    pos, C, rc = oracle.layout(wl, inp.indices, inp.num_tokens)
    bufs = oracle.dispatch_buffers(wl, cap)
    for v in bufs.values():
        v.fill(0)
    nt = np.ascontiguousarray(inp.num_tokens, np.int32)
    oracle.run_ranges(lambda a, b: oracle.dispatch_into(
        wl, inp.x_bits, inp.weights, inp.indices, nt, pos, cap, bufs, a, b), W * T, 5)
    y = np.zeros((W, cap, H), np.uint16)
    oracle.run_ranges(lambda a, b: oracle.identity_expert_into(
        wl, rc, bufs, cap, y, a, b), W * cap, 7)
    out = np.zeros((W, T, H), np.uint16)
    out_w = np.zeros((W, T, k), np.float32)
    oracle.run_ranges(lambda a, b: oracle.combine_into(
        wl, nt, pos, y, bufs["out_w"], cap, out, out_w, a, b), W * T, 3)
    for key in ("out", "out_w", "out_idx", "src_pos"):
        assert np.array_equal(bufs[key], ref[key]), key
    if fp8:
        assert np.array_equal(bufs["out_scales"].view(np.uint32),
                              ref["out_scales"].view(np.uint32))
    assert np.array_equal(y, ref["y"])
    assert np.array_equal(out, ref["combined"])
    assert np.array_equal(out_w.view(np.uint32), ref["combined_w"].view(np.uint32))
