"""Helpers of the GPU tests: run the CUDA path through the C ABI binding on
seeded inputs and bring the results back as numpy arrays."""
from __future__ import annotations

import numpy as np
import torch

from combine_ep_layout_06_gb300.op import (EpDispatchCombineConfig,
                                           EpDispatchCombineOp)


def make_op(wl, cap=0, **kw):
    cfg = EpDispatchCombineConfig(
        world_size=wl.world_size, num_experts=wl.num_experts, topk=wl.topk,
        hidden=wl.hidden, max_tokens_per_rank=wl.max_tokens_per_rank,
        max_recv_tokens_per_rank=cap,
        dispatch_dtype="fp8_e4m3" if wl.fp8 else "bf16", **kw)
    return EpDispatchCombineOp(cfg)


def to_device(inp, dev="cuda"):
    x = torch.from_numpy(inp.x_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    w = torch.from_numpy(inp.weights).to(dev)
    idx = torch.from_numpy(inp.indices).to(dev)
    return x, w, idx


def bits(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of a tensor as a numpy array."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy().view(np.uint32)
    return t.numpy()


def run_gpu(op, inp, identity=True, with_weights=True, split=False,
            payload=True):
    """Dispatch, identity expert, combine.  Returns numpy results (without
    the receive payload and expert rows when payload=False)."""
    x, w, idx = to_device(inp)
    nt = [int(n) for n in inp.num_tokens]
    if split:
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        s1.wait_stream(torch.cuda.current_stream())
        op.dispatch_send(x, w, None, idx, num_tokens=nt, stream=s1)
        op.dispatch_recv(stream=s2)
        if identity:
            op.identity_expert(stream=s2)
        op.combine_send(stream=s2)
        out, out_w = op.combine_recv(weights=op.out_w if with_weights else None,
                                     indices=idx, stream=s1)
        torch.cuda.current_stream().wait_stream(s1)
    else:
        op.dispatch(x, w, None, idx, num_tokens=nt)
        if identity:
            op.identity_expert()
        out, out_w = op.combine(weights=op.out_w if with_weights else None,
                                indices=idx)
    torch.cuda.synchronize()
    res = dict(
        recv_count=op.recv_count.cpu().numpy().copy(),
        send_counts=op.send_counts.cpu().numpy().copy(),
        pos=op.pos.cpu().numpy().copy(),
        src_pos=op.src_pos.cpu().numpy().copy(),
        out_w=op.out_w.cpu().numpy().copy(),
        out_idx=op.out_idx.cpu().numpy().copy(),
        out=bits(op.out) if payload else None,
        y=bits(op.combine_input) if payload else None,
        combined=bits(out),
        combined_w=None if out_w is None else out_w.cpu().numpy().copy(),
    )
    if op.out_scales is not None and payload:
        res["out_scales"] = op.out_scales.cpu().numpy().copy()
    return res


def ulp_diff_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in bf16 ulps, via the sign-magnitude ordering of the bits."""
    def key(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(key(a) - key(b))
