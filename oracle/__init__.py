"""CPU oracle for MoE token layout, dispatch and combine (test infrastructure).

Only ``tests/``, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  It wraps the plain scalar C in ``ep_oracle.c``
(compiled here with gcc, no CUDA) and hands numpy arrays in and out.  It
shares no code with the CUDA library.

Definitions followed: ROCm MORI "Communication APIs" page, section
"MORI-EP (Expert Parallelism)", table "EpDispatchCombineOp methods"
(dispatch / combine / get_dispatch_src_token_pos), plus the readings stated
in the header of ``ep_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libep_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle library with gcc (seconds).  Returns its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64


def _declare(L):
    sig = {
        "or_bf16_rne": (ctypes.c_uint16, [ctypes.c_float]),
        "or_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "or_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
        "or_e4m3_value": (ctypes.c_float, [ctypes.c_uint8]),
        "or_bf16_rne_array": (None, [_P, _P, _L]),
        "or_e4m3_encode_array": (None, [_P, _P, _L]),
        "or_e4m3_value_array": (None, [_P, _P, _L]),
        "or_quant_rows": (None, [_P, _L, _I, _P, _P]),
        "or_validate": (_I, [_I, _I, _I, _I, _I, _I, _P, _P]),
        "or_layout": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
        "or_dispatch": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                             _P, _P, _P, _P, _P]),
        "or_dispatch_rows": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                                  _P, _P, _I, _P, _P, _P, _P, _P]),
        "or_identity_expert": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                    _P, _P]),
        "or_identity_rows": (_I, [_I, _I, _I, _I, _I, _P, _I, _P, _P, _P,
                                  _P, _P]),
        "or_combine_gathered": (_I, [_I, _I, _P, _P]),
        "or_dispatch_prequant": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                                      _P, _P, _P, _P, _P, _P]),
        "or_identity_expert_f32": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                        _P, _P]),
        "or_combine_f32": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
        "or_expert_layout": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P]),
        "or_group_rows": (_I, [_I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                               _P, _P, _P, _P]),
        "or_ungroup": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
        "or_identity_expert_fp8": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                        _P, _P, _P, _P]),
        "or_combine_fp8": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
        "or_quant_block_f32": (None, [_P, _I, _P, _P]),
        "or_combine": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
        "or_dispatch_range": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                                   _P, _P, _P, _P, _P, _L, _L]),
        "or_identity_expert_range": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                          _P, _P, _L, _L]),
        "or_combine_range": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                  _L, _L]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ scalars

def bf16_rne(v) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even (element-wise)."""
    v = _c(v, np.float32)
    o = np.empty(v.shape, np.uint16)
    lib().or_bf16_rne_array(_p(v), _p(o), v.size)
    return o


def bf16_to_f32(b) -> np.ndarray:
    b = _c(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def e4m3_encode(v) -> np.ndarray:
    """fp32 -> OCP E4M3 code, RNE, satfinite, sign kept (element-wise)."""
    v = _c(v, np.float32)
    o = np.empty(v.shape, np.uint8)
    lib().or_e4m3_encode_array(_p(v), _p(o), v.size)
    return o


def e4m3_value(q) -> np.ndarray:
    q = _c(q, np.uint8)
    o = np.empty(q.shape, np.float32)
    lib().or_e4m3_value_array(_p(q), _p(o), q.size)
    return o


def quant_rows(x_bits) -> tuple[np.ndarray, np.ndarray]:
    """Per-128-element-block FP8 quantisation of bf16 rows [n][H]."""
    x = _c(x_bits, np.uint16)
    n, H = x.shape
    q = np.empty((n, H), np.uint8)
    sc = np.empty((n, H // 128), np.float32)
    lib().or_quant_rows(_p(x), n, H, _p(q), _p(sc))
    return q, sc


# ------------------------------------------------------------ whole method

class OracleError(ValueError):
    pass


def validate(wl, idx, num_tokens, fp8=None):
    idx = _c(idx, np.int32)
    nt = _c(num_tokens, np.int32)
    fp8 = wl.fp8 if fp8 is None else fp8
    rc = lib().or_validate(wl.world_size, wl.num_experts, wl.topk,
                           wl.max_tokens_per_rank, wl.hidden, int(fp8),
                           _p(idx), _p(nt))
    if rc != 0:
        raise OracleError("inputs outside the method's contract")


def layout(wl, idx, num_tokens):
    """Returns (pos int32 [W][T][W], C int32 [W][W], recv_count int32 [W])."""
    W, T, k = wl.world_size, wl.max_tokens_per_rank, wl.topk
    idx = _c(idx, np.int32)
    nt = _c(num_tokens, np.int32)
    validate(wl, idx, nt)
    scratch = np.empty((W, T, W), np.uint8)
    pos = np.empty((W, T, W), np.int32)
    C = np.empty((W, W), np.int32)
    rc = np.empty(W, np.int32)
    lib().or_layout(W, wl.num_experts, k, T, _p(idx), _p(nt), _p(scratch),
                    _p(pos), _p(C), _p(rc))
    return pos, C, rc


def dispatch(wl, x_bits, w, idx, num_tokens, pos, cap, fp8=None,
             payload=True):
    """Dispatched receive buffers, dense [W][cap][...].  Unwritten rows are
    zero.  With payload=False only out_w / out_idx / src_pos are filled."""
    W, T, H, k = (wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk)
    fp8 = wl.fp8 if fp8 is None else fp8
    x = _c(x_bits, np.uint16)
    w = _c(w, np.float32)
    idx = _c(idx, np.int32)
    nt = _c(num_tokens, np.int32)
    pos = _c(pos, np.int32)
    out = None
    if payload:
        out = np.zeros((W, cap, H), np.uint8 if fp8 else np.uint16)
    nb = H // 128 if fp8 else 0
    scales = np.zeros((W, cap, max(nb, 1)), np.float32)
    out_w = np.zeros((W, cap, k), np.float32)
    out_idx = np.zeros((W, cap, k), np.int32)
    src = np.zeros((W, cap), np.int32)
    lib().or_dispatch(W, k, T, H, cap, int(fp8), _p(x), _p(w), _p(idx),
                      _p(nt), _p(pos), _p(out), _p(scales), _p(out_w),
                      _p(out_idx), _p(src))
    return dict(out=out, out_scales=scales[..., :nb], out_w=out_w,
                out_idx=out_idx, src_pos=src)


def dispatch_rows(wl, x_bits, w, idx, num_tokens, pos, ranks, slots, fp8=None):
    """What dispatch writes to the receive slots (ranks[i], slots[i])."""
    W, T, H, k = (wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk)
    fp8 = wl.fp8 if fp8 is None else fp8
    ranks = _c(ranks, np.int32)
    slots = _c(slots, np.int32)
    n = ranks.size
    nb = H // 128 if fp8 else 0
    out = np.zeros((n, H), np.uint8 if fp8 else np.uint16)
    sc = np.zeros((n, max(nb, 1)), np.float32)
    ow = np.zeros((n, k), np.float32)
    oi = np.zeros((n, k), np.int32)
    sp = np.zeros(n, np.int32)
    rc = lib().or_dispatch_rows(
        W, k, T, H, int(fp8), _p(_c(x_bits, np.uint16)), _p(_c(w, np.float32)),
        _p(_c(idx, np.int32)), _p(_c(num_tokens, np.int32)),
        _p(_c(pos, np.int32)), _p(ranks), _p(slots), n, _p(out), _p(sc),
        _p(ow), _p(oi), _p(sp))
    if rc != 0:
        raise OracleError("a sampled slot has no source token")
    return dict(out=out, out_scales=sc[:, :nb], out_w=ow, out_idx=oi,
                src_pos=sp)


def identity_expert(wl, recv_count, payload, scales, out_w, out_idx, cap,
                    fp8=None):
    """Identity-expert output y uint16 [W][cap][H] (rows past the count 0)."""
    W, H, k = wl.world_size, wl.hidden, wl.topk
    fp8 = wl.fp8 if fp8 is None else fp8
    y = np.zeros((W, cap, H), np.uint16)
    nb = H // 128 if fp8 else 0
    sc = (_c(scales, np.float32) if fp8
          else np.zeros((W, cap, 1), np.float32))
    pl = _c(payload, np.uint8 if fp8 else np.uint16)
    lib().or_identity_expert(W, wl.num_experts, k, H, cap, int(fp8),
                             _p(_c(recv_count, np.int32)), _p(pl), _p(sc),
                             _p(_c(out_w, np.float32)),
                             _p(_c(out_idx, np.int32)), _p(y))
    return y


def identity_rows(wl, ranks, payload, scales, w, idx, fp8=None):
    """Identity-expert output of listed rows (row i received on ranks[i])."""
    fp8 = wl.fp8 if fp8 is None else fp8
    ranks = _c(ranks, np.int32)
    n = ranks.size
    H = wl.hidden
    y = np.zeros((n, H), np.uint16)
    sc = (_c(scales, np.float32) if fp8 else np.zeros((n, 1), np.float32))
    lib().or_identity_rows(wl.world_size, wl.num_experts, wl.topk, H, int(fp8),
                           _p(ranks), n,
                           _p(_c(payload, np.uint8 if fp8 else np.uint16)),
                           _p(sc), _p(_c(w, np.float32)), _p(_c(idx, np.int32)),
                           _p(y))
    return y


def combine_gathered(rows):
    """Combine sum of one token's rows [nd][H] given in ascending rank order."""
    rows = _c(rows, np.uint16)
    nd, H = rows.shape
    out = np.zeros(H, np.uint16)
    if lib().or_combine_gathered(nd, H, _p(rows), _p(out)) != 0:
        raise OracleError("too many rows")
    return out


def combine(wl, num_tokens, pos, y, w_in, cap):
    """Returns (out uint16 [W][T][H], out_w float32 [W][T][k] or None)."""
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    out = np.zeros((W, T, H), np.uint16)
    out_w = np.zeros((W, T, k), np.float32) if w_in is not None else None
    lib().or_combine(W, k, T, H, cap, _p(_c(num_tokens, np.int32)),
                     _p(_c(pos, np.int32)), _p(_c(y, np.uint16)),
                     _p(None if w_in is None else _c(w_in, np.float32)),
                     _p(out), _p(out_w))
    return out, out_w


def dispatch_prequant(wl, x8, scales, w, idx, num_tokens, pos, cap):
    """Dispatch of pre-quantised FP8 input (codes + block scales copied)."""
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    nb = H // 128
    out = np.zeros((W, cap, H), np.uint8)
    osc = np.zeros((W, cap, nb), np.float32)
    ow = np.zeros((W, cap, k), np.float32)
    oi = np.zeros((W, cap, k), np.int32)
    sp = np.zeros((W, cap), np.int32)
    lib().or_dispatch_prequant(W, k, T, H, cap, _p(_c(x8, np.uint8)),
                               _p(_c(scales, np.float32)), _p(_c(w, np.float32)),
                               _p(_c(idx, np.int32)), _p(_c(num_tokens, np.int32)),
                               _p(_c(pos, np.int32)), _p(out), _p(osc), _p(ow),
                               _p(oi), _p(sp))
    return dict(out=out, out_scales=osc, out_w=ow, out_idx=oi, src_pos=sp)


def identity_expert_f32(wl, recv_count, payload, scales, out_w, out_idx, cap,
                        fp8=None):
    """Identity-expert output as fp32 rows [W][cap][H] (no bf16 rounding)."""
    W, H, k = wl.world_size, wl.hidden, wl.topk
    fp8 = wl.fp8 if fp8 is None else fp8
    y = np.zeros((W, cap, H), np.float32)
    sc = (_c(scales, np.float32) if fp8 else np.zeros((W, cap, 1), np.float32))
    pl = _c(payload, np.uint8 if fp8 else np.uint16)
    lib().or_identity_expert_f32(W, wl.num_experts, k, H, cap, int(fp8),
                                 _p(_c(recv_count, np.int32)), _p(pl), _p(sc),
                                 _p(_c(out_w, np.float32)),
                                 _p(_c(out_idx, np.int32)), _p(y))
    return y


def combine_f32(wl, num_tokens, pos, y, w_in, cap):
    """Combine of fp32 expert rows y [W][cap][H] -> bf16 out [W][T][H]."""
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    out = np.zeros((W, T, H), np.uint16)
    out_w = np.zeros((W, T, k), np.float32) if w_in is not None else None
    lib().or_combine_f32(W, k, T, H, cap, _p(_c(num_tokens, np.int32)),
                         _p(_c(pos, np.int32)), _p(_c(y, np.float32)),
                         _p(None if w_in is None else _c(w_in, np.float32)),
                         _p(out), _p(out_w))
    return out, out_w


def expert_layout(wl, recv_count, out_idx, cap):
    """Standard-MoE grouping layout: (count [W][Er], offset [W][Er],
    entry_slot [W][cap][k])."""
    W, k, Er = wl.world_size, wl.topk, wl.experts_per_rank
    count = np.zeros((W, Er), np.int32)
    offset = np.zeros((W, Er), np.int32)
    slot = np.zeros((W, cap, k), np.int32)
    lib().or_expert_layout(W, wl.num_experts, k, cap, _p(_c(recv_count, np.int32)),
                           _p(_c(out_idx, np.int32)), _p(count), _p(offset), _p(slot))
    return count, offset, slot


def group_rows(wl, recv_count, out, out_scales, out_w, entry_slot, cap, gcap):
    """Grouped copy: (xg [W][gcap][H], xg_scales [W][gcap][nb], g_src, g_w);
    slots never written stay zero."""
    W, H, k = wl.world_size, wl.hidden, wl.topk
    fp8 = out.dtype == np.uint8
    nb = H // 128 if fp8 else 0
    xg = np.zeros((W, gcap, H), out.dtype)
    xs = np.zeros((W, gcap, max(nb, 1)), np.float32)
    src = np.zeros((W, gcap), np.int32)
    gw = np.zeros((W, gcap), np.float32)
    osc = _c(out_scales, np.float32) if fp8 else np.zeros((W, cap, 1), np.float32)
    lib().or_group_rows(W, k, H, 1 if fp8 else 2, nb, cap, gcap,
                        _p(_c(recv_count, np.int32)), _p(_c(out, out.dtype)), _p(osc),
                        _p(_c(out_w, np.float32)), _p(_c(entry_slot, np.int32)),
                        _p(xg), _p(xs), _p(src), _p(gw))
    return xg, xs[..., :nb], src, gw


def ungroup(wl, recv_count, out_w, entry_slot, yg, cap, gcap):
    """Weighted per-row sum of the grouped expert outputs: y [W][cap][H]."""
    W, H, k = wl.world_size, wl.hidden, wl.topk
    y = np.zeros((W, cap, H), np.uint16)
    lib().or_ungroup(W, k, H, cap, gcap, _p(_c(recv_count, np.int32)),
                     _p(_c(out_w, np.float32)), _p(_c(entry_slot, np.int32)),
                     _p(_c(yg, np.uint16)), _p(y))
    return y


def quant_rows_f32(v):
    """Per-128-element-block FP8 quantisation of fp32 rows [n][H]."""
    v = _c(v, np.float32)
    n, H = v.shape
    q = np.empty((n, H), np.uint8)
    sc = np.empty((n, H // 128), np.float32)
    for i in range(n):
        for b in range(H // 128):
            lib().or_quant_block_f32(v[i, b * 128:].ctypes.data_as(ctypes.c_void_p), 128,
                                     q[i, b * 128:].ctypes.data_as(ctypes.c_void_p),
                                     sc[i, b:].ctypes.data_as(ctypes.c_void_p))
    return q, sc


def identity_expert_fp8(wl, recv_count, payload, scales, out_w, out_idx, cap, fp8=None):
    """Identity expert with an FP8 combine payload: (yq [W][cap][H],
    ysc [W][cap][H/128]); rows past the count are zero."""
    W, H, k = wl.world_size, wl.hidden, wl.topk
    fp8 = wl.fp8 if fp8 is None else fp8
    yq = np.zeros((W, cap, H), np.uint8)
    ysc = np.zeros((W, cap, H // 128), np.float32)
    sc = (_c(scales, np.float32) if fp8 else np.zeros((W, cap, 1), np.float32))
    pl = _c(payload, np.uint8 if fp8 else np.uint16)
    tmp = np.empty(H, np.float32)
    lib().or_identity_expert_fp8(W, wl.num_experts, k, H, cap, int(fp8),
                                 _p(_c(recv_count, np.int32)), _p(pl), _p(sc),
                                 _p(_c(out_w, np.float32)), _p(_c(out_idx, np.int32)),
                                 _p(tmp), _p(yq), _p(ysc))
    return yq, ysc


def combine_fp8(wl, num_tokens, pos, yq, ysc, w_in, cap):
    """Combine of an FP8 expert payload -> bf16 out [W][T][H]."""
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    out = np.zeros((W, T, H), np.uint16)
    out_w = np.zeros((W, T, k), np.float32) if w_in is not None else None
    lib().or_combine_fp8(W, k, T, H, cap, _p(_c(num_tokens, np.int32)),
                         _p(_c(pos, np.int32)), _p(_c(yq, np.uint8)), _p(_c(ysc, np.float32)),
                         _p(None if w_in is None else _c(w_in, np.float32)),
                         _p(out), _p(out_w))
    return out, out_w


def run_all(inp, cap=None):
    """Layout, dispatch, identity expert and combine of one batch.
    Returns a dict with every intermediate (small workloads only)."""
    wl = inp.wl
    cap = wl.world_size * wl.max_tokens_per_rank if cap is None else cap
    pos, C, rc = layout(wl, inp.indices, inp.num_tokens)
    d = dispatch(wl, inp.x_bits, inp.weights, inp.indices, inp.num_tokens,
                 pos, cap)
    y = identity_expert(wl, rc, d["out"], d["out_scales"], d["out_w"],
                        d["out_idx"], cap)
    out, out_w = combine(wl, inp.num_tokens, pos, y, d["out_w"], cap)
    return dict(pos=pos, C=C, recv_count=rc, cap=cap, y=y, combined=out,
                combined_w=out_w, **d)


# ------------------------------------------- into preallocated buffers, by range
# The timed CPU baseline: the same C functions, run over disjoint slices of
# independent tokens (dispatch, combine) or receive rows (identity expert) on
# several host threads; ctypes releases the GIL for the duration of each call.

def run_ranges(fn, n, threads):
    """fn(lo, hi) over `threads` contiguous slices of [0, n), one thread each."""
    import concurrent.futures as cf
    threads = max(1, min(int(threads), n)) if n > 0 else 1
    bounds = [n * i // threads for i in range(threads + 1)]
    if threads == 1:
        fn(0, n)
        return
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda i: fn(bounds[i], bounds[i + 1]), range(threads)))


def dispatch_buffers(wl, cap, fp8=None):
    """Receive buffers [W][cap][...] for dispatch_into (contents unspecified)."""
    W, H, k = wl.world_size, wl.hidden, wl.topk
    fp8 = wl.fp8 if fp8 is None else fp8
    nb = H // 128 if fp8 else 0
    return dict(out=np.empty((W, cap, H), np.uint8 if fp8 else np.uint16),
                out_scales=np.empty((W, cap, max(nb, 1)), np.float32),
                out_w=np.empty((W, cap, k), np.float32),
                out_idx=np.empty((W, cap, k), np.int32),
                src_pos=np.empty((W, cap), np.int32))


def dispatch_into(wl, x_bits, w, idx, num_tokens, pos, cap, bufs, g0, g1, fp8=None):
    """Dispatch of source tokens g0 <= s*T + t < g1 into preallocated buffers
    (arrays must be C-contiguous of the dispatch_buffers types)."""
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    fp8 = wl.fp8 if fp8 is None else fp8
    lib().or_dispatch_range(W, k, T, H, cap, int(fp8), _p(x_bits), _p(w), _p(idx),
                            _p(num_tokens), _p(pos), _p(bufs["out"]),
                            _p(bufs["out_scales"]), _p(bufs["out_w"]),
                            _p(bufs["out_idx"]), _p(bufs["src_pos"]), int(g0), int(g1))


def identity_expert_into(wl, recv_count, bufs, cap, y, i0, i1, fp8=None):
    """Identity expert of receive rows i0 <= r*cap + p < i1 into y [W][cap][H]."""
    W, H, k = wl.world_size, wl.hidden, wl.topk
    fp8 = wl.fp8 if fp8 is None else fp8
    lib().or_identity_expert_range(W, wl.num_experts, k, H, cap, int(fp8),
                                   _p(recv_count), _p(bufs["out"]),
                                   _p(bufs["out_scales"]), _p(bufs["out_w"]),
                                   _p(bufs["out_idx"]), _p(y), int(i0), int(i1))


def combine_into(wl, num_tokens, pos, y, w_in, cap, out, out_w, g0, g1):
    """Combine of source tokens g0 <= s*T + t < g1 into out [W][T][H] (and
    out_w [W][T][k] when w_in is given)."""
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    lib().or_combine_range(W, k, T, H, cap, _p(num_tokens), _p(pos), _p(y),
                           _p(w_in), _p(out), _p(out_w), int(g0), int(g1))
