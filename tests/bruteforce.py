"""Brute-force MoE dispatch / combine for tiny inputs (pure Python + numpy).

A second, deliberately different construction used to pin the C oracle:
each rank's receive list is built by collecting the (source rank, source
token) pairs routed to it into a Python list and sorting it, and combine
finds each token's rows through a dict keyed by (s, t).  The FP8 encoder is
torch's CPU cast to float8_e4m3fn and the bf16 rounding is torch's CPU cast
to bfloat16; scales and quotients are numpy float32 divisions.

Definitions: ROCm MORI "Communication APIs" page, "MORI-EP (Expert
Parallelism)", table "EpDispatchCombineOp methods" (dispatch, combine,
get_dispatch_src_token_pos); "Validation before tuning" (identity expert).
"""
from __future__ import annotations

import numpy as np
import torch


def to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def torch_bf16_bits(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def torch_e4m3(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def torch_e4m3_value(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float32).numpy()


def quant_block(xb):
    """FP8 block: scale = f32(amax / 448), codes = e4m3(f32(x / scale))."""
    xf = to_f32(xb)
    a = np.float32(np.abs(xf).max())
    if a == 0:
        return np.zeros(xb.shape, np.uint8), np.float32(0)
    sc = np.float32(a) / np.float32(448.0)
    q = torch_e4m3(xf / sc)
    return q, np.float32(sc)


def receive_lists(idx, num_tokens, W, E):
    """{r: sorted list of (s, t)} for every rank r."""
    Er = E // W
    lists = {r: [] for r in range(W)}
    for s in range(W):
        for t in range(int(num_tokens[s])):
            for r in sorted({int(e) // Er for e in idx[s, t]}):
                lists[r].append((s, t))
    return {r: sorted(v) for r, v in lists.items()}


def dispatch(x_bits, w, idx, num_tokens, W, E, fp8=False):
    """Per rank r: dict(rows=[(s,t)...], out, out_scales, out_w, out_idx,
    src_pos) with one entry per received row, in receive order."""
    T = x_bits.shape[1]
    res = {}
    for r, rows in receive_lists(idx, num_tokens, W, E).items():
        outs, scs = [], []
        for (s, t) in rows:
            if fp8:
                H = x_bits.shape[2]
                qs, ss = [], []
                for b in range(H // 128):
                    q, sc = quant_block(x_bits[s, t, b * 128:(b + 1) * 128])
                    qs.append(q)
                    ss.append(sc)
                outs.append(np.concatenate(qs))
                scs.append(np.array(ss, np.float32))
            else:
                outs.append(x_bits[s, t].copy())
        res[r] = dict(
            rows=rows,
            out=np.array(outs) if outs else None,
            out_scales=np.array(scs) if scs else None,
            out_w=np.array([w[s, t] for s, t in rows], np.float32).reshape(-1, w.shape[2]),
            out_idx=np.array([idx[s, t] for s, t in rows], np.int32).reshape(-1, idx.shape[2]),
            src_pos=np.array([s * T + t for s, t in rows], np.int32),
        )
    return res


def identity_expert(d, r, W, E, fp8=False):
    """y rows of rank r: bf16(f32(v * alpha)), alpha = ordered f32 sum of
    the weights whose expert is on rank r."""
    Er = E // W
    ys = []
    for i in range(len(d["rows"])):
        alpha = np.float32(0)
        for j in range(d["out_idx"].shape[1]):
            if int(d["out_idx"][i, j]) // Er == r:
                alpha = np.float32(alpha + d["out_w"][i, j])
        if fp8:
            H = d["out"].shape[1]
            vals = torch_e4m3_value(d["out"][i])
            sc = np.repeat(d["out_scales"][i], 128)[:H]
            v = (vals * sc).astype(np.float32)
        else:
            v = to_f32(d["out"][i])
        ys.append(torch_bf16_bits((v * alpha).astype(np.float32)))
    return ys


def combine(disp, ys, w_in, W, T, H, k, num_tokens):
    """out[(s,t)] = bf16(sum over r ascending of f32(y_r row)), and the same
    ordered f32 sum of the w_in rows.  Returns dicts keyed by (s, t)."""
    where = {}
    for r in range(W):
        for i, st in enumerate(disp[r]["rows"]):
            where.setdefault(st, []).append((r, i))
    out, out_w = {}, {}
    for s in range(W):
        for t in range(int(num_tokens[s])):
            acc = np.zeros(H, np.float32)
            accw = np.zeros(k, np.float32)
            for r, i in sorted(where.get((s, t), [])):
                acc = (acc + to_f32(ys[r][i])).astype(np.float32)
                if w_in is not None:
                    accw = (accw + w_in[r][i]).astype(np.float32)
            out[(s, t)] = torch_bf16_bits(acc)
            out_w[(s, t)] = accw
    return out, out_w


def dispatch_prequant(x8, sc, w, idx, num_tokens, W, E):
    """Pre-quantised payload: per rank, the received codes and scales rows."""
    T = x8.shape[1]
    res = {}
    for r, rows in receive_lists(idx, num_tokens, W, E).items():
        res[r] = dict(rows=rows,
                      out=np.array([x8[s, t] for s, t in rows]).reshape(-1, x8.shape[2]),
                      out_scales=np.array([sc[s, t] for s, t in rows],
                                          np.float32).reshape(-1, sc.shape[2]),
                      src_pos=np.array([s * T + t for s, t in rows], np.int32))
    return res


def identity_expert_f32(d, r, W, E, fp8=False):
    """fp32 rows f32(v * alpha) of rank r (no bf16 rounding)."""
    Er = E // W
    ys = []
    for i in range(len(d["rows"])):
        alpha = np.float32(0)
        for j in range(d["out_idx"].shape[1]):
            if int(d["out_idx"][i, j]) // Er == r:
                alpha = np.float32(alpha + d["out_w"][i, j])
        if fp8:
            H = d["out"].shape[1]
            v = (torch_e4m3_value(d["out"][i]) * np.repeat(d["out_scales"][i], 128)[:H]).astype(np.float32)
        else:
            v = to_f32(d["out"][i])
        ys.append((v * alpha).astype(np.float32))
    return ys


def combine_f32(disp, ys, W, T, H, num_tokens):
    """out[(s,t)] = bf16(sum over r ascending of the fp32 rows)."""
    where = {}
    for r in range(W):
        for i, st in enumerate(disp[r]["rows"]):
            where.setdefault(st, []).append((r, i))
    out = {}
    for s in range(W):
        for t in range(int(num_tokens[s])):
            acc = np.zeros(H, np.float32)
            for r, i in sorted(where.get((s, t), [])):
                acc = (acc + ys[r][i]).astype(np.float32)
            out[(s, t)] = torch_bf16_bits(acc)
    return out


def expert_groups(out_idx_rows, r, Er):
    """Entries of rank r as a dict e -> sorted list of (p, j), by listing
    every local selection and sorting by (expert, p, j)."""
    ent = []
    for p, ids in enumerate(out_idx_rows):
        for j, g in enumerate(ids):
            if int(g) // Er == r:
                ent.append((int(g) - r * Er, p, j))
    groups = {}
    for e, p, j in sorted(ent):
        groups.setdefault(e, []).append((p, j))
    return groups


def ungroup_row(w_row, ys):
    """bf16(sum over the row's entries, j ascending, of f32(w_j * y_j))."""
    acc = None
    for w, y in ys:
        prod = (np.float32(w) * to_f32(y)).astype(np.float32)
        if acc is None:
            acc = np.zeros_like(prod)
        acc = (acc + prod).astype(np.float32)
    return None if acc is None else torch_bf16_bits(acc)
