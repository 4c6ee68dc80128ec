"""Python face of the library: ``EpDispatchCombineConfig`` and
``EpDispatchCombineOp`` with the method set of the MORI-EP op (ROCm MORI
"Communication APIs", "MORI-EP (Expert Parallelism)", table
"EpDispatchCombineOp methods").

Marshalling only: every step runs in the CUDA kernels of libep_gb300.so.
PyTorch provides device memory, streams and tensor views.  All W logical
ranks live on one GPU, so per-rank tensors carry a leading [W] dimension.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import EpError, check


@dataclasses.dataclass
class EpDispatchCombineConfig:
    world_size: int
    num_experts: int
    topk: int
    hidden: int
    max_tokens_per_rank: int
    max_recv_tokens_per_rank: int = 0        # 0 -> W*T
    dispatch_dtype: str = "bf16"             # "bf16" | "fp8_e4m3"
    early_notify: bool = False
    fused_recv: bool = False
    wait_timeout_ns: int = 0                 # 0 -> 1 s
    combine_dtype: str = "bf16"              # expert rows combine reads: "bf16" | "fp32" | "fp8_e4m3"
    max_grouped_rows_per_rank: int = 0       # standard-MoE grouping (0: off)
    combine_mode: str = "gather"             # "gather" | "scatter"

    def to_c(self) -> _lib.EpConfigC:
        dt = {"bf16": _lib.EP_DT_BF16, "fp8_e4m3": _lib.EP_DT_FP8_E4M3}
        ct = {"bf16": _lib.EP_DT_BF16, "fp32": _lib.EP_DT_FP32,
              "fp8_e4m3": _lib.EP_DT_FP8_E4M3}
        if self.dispatch_dtype not in dt:
            raise ValueError(f"dispatch_dtype {self.dispatch_dtype!r}")
        if self.combine_dtype not in ct:
            raise ValueError(f"combine_dtype {self.combine_dtype!r}")
        return _lib.EpConfigC(
            self.world_size, self.num_experts, self.topk, self.hidden,
            self.max_tokens_per_rank, self.max_recv_tokens_per_rank,
            dt[self.dispatch_dtype], int(self.early_notify),
            int(self.fused_recv), ct[self.combine_dtype],
            int(self.wait_timeout_ns), int(self.max_grouped_rows_per_rank),
            {"gather": 0, "scatter": 1}[self.combine_mode])


def workspace_size(cfg: EpDispatchCombineConfig) -> int:
    n = ctypes.c_size_t(0)
    c = cfg.to_c()
    check(_lib.load().ep_workspace_size(ctypes.byref(c), ctypes.byref(n)),
          "ep_workspace_size")
    return n.value


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class EpDispatchCombineOp:
    """Stateful dispatch/combine op over W logical ranks on one GPU."""

    def __init__(self, config: EpDispatchCombineConfig,
                 device: Optional[torch.device] = None):
        self.config = config
        self.L = _lib.load()
        self.device = torch.device("cuda", torch.cuda.current_device()) \
            if device is None else torch.device(device)
        nbytes = workspace_size(config)
        with torch.cuda.device(self.device):
            self.workspace = torch.empty(nbytes, dtype=torch.uint8,
                                         device=self.device)
            h = ctypes.c_void_p()
            c = config.to_c()
            check(self.L.ep_create(ctypes.byref(c), _ptr(self.workspace),
                                   nbytes, ctypes.byref(h)), "ep_create")
        self.h = h
        self._views()

    # ----------------------------------------------------------- views
    def _views(self):
        o = _lib.EpDispatchOutC()
        check(self.L.ep_dispatch_outputs(self.h, ctypes.byref(o)),
              "ep_dispatch_outputs")
        c = self.config
        W, T, H, k = c.world_size, c.max_tokens_per_rank, c.hidden, c.topk
        cap = o.cap
        self.cap = cap
        base = self.workspace.data_ptr()
        rs = o.rank_stride_bytes
        fp8 = c.dispatch_dtype == "fp8_e4m3"

        def view(ptr, dtype, shape, strides_elems):
            esz = torch.empty((), dtype=dtype).element_size()
            off = ptr - base
            assert off % esz == 0
            flat = self.workspace.view(dtype)
            return torch.as_strided(flat, shape, strides_elems, off // esz)

        self.out = view(o.out, torch.uint8 if fp8 else torch.bfloat16,
                        (W, cap, H), (rs // (1 if fp8 else 2), H, 1))
        nb = H // 128
        self.out_scales = (view(o.out_scales, torch.float32, (W, cap, nb),
                                (rs // 4, nb, 1)) if fp8 else None)
        self.out_w = view(o.out_w, torch.float32, (W, cap, k), (rs // 4, k, 1))
        self.out_idx = view(o.out_idx, torch.int32, (W, cap, k), (rs // 4, k, 1))
        self.src_pos = view(o.src_pos, torch.int32, (W, cap), (rs // 4, 1))
        self.recv_count = view(o.recv_count, torch.int32, (W,), (1,))
        self.send_counts = view(o.send_counts, torch.int32, (W, W), (W, 1))
        self.pos = view(o.pos, torch.int32, (W, T, W), (T * W, W, 1))
        self.combine_stage = None
        if o.combine_stage:
            md = o.max_dest
            self.combine_stage = view(o.combine_stage, torch.bfloat16, (W, T, md, H),
                                      (T * md * H, md * H, H, 1))
        self.dispatch_flags = view(o.dispatch_flags, torch.int32, (W, W), (W, 1))
        self.combine_flags = view(o.combine_flags, torch.int32, (W, W), (W, 1))
        p = ctypes.c_void_p()
        s = ctypes.c_int64()
        ydt = {"bf16": (_lib.EP_DT_BF16, torch.bfloat16, 2),
               "fp32": (_lib.EP_DT_FP32, torch.float32, 4),
               "fp8_e4m3": (_lib.EP_DT_FP8_E4M3, torch.uint8, 1)}[c.combine_dtype]
        check(self.L.ep_get_combine_input_buffer(self.h, ydt[0], ctypes.byref(p),
                                                 ctypes.byref(s)),
              "ep_get_combine_input_buffer")
        self.y_dtype = ydt[1]
        self.combine_input = view(p.value, self.y_dtype, (W, cap, H),
                                  (s.value // ydt[2], H, 1))
        self.combine_input_scales = None
        if c.combine_dtype == "fp8_e4m3":
            ps = ctypes.c_void_p()
            check(self.L.ep_get_combine_input_scales(self.h, ctypes.byref(ps), ctypes.byref(s)),
                  "ep_get_combine_input_scales")
            self.combine_input_scales = view(ps.value, torch.float32, (W, cap, nb),
                                             (s.value // 4, nb, 1))
        self.rank_stride_bytes = rs
        if c.max_grouped_rows_per_rank > 0:
            m = _lib.EpMoeOutC()
            check(self.L.ep_moe_outputs(self.h, ctypes.byref(m)), "ep_moe_outputs")
            g, Er = m.gcap, m.experts_per_rank
            self.moe_x = view(m.xg, torch.uint8 if fp8 else torch.bfloat16, (W, g, H),
                              (rs // (1 if fp8 else 2), H, 1))
            self.moe_x_scales = (view(m.xg_scales, torch.float32, (W, g, nb),
                                      (rs // 4, nb, 1)) if fp8 else None)
            self.moe_src = view(m.g_src, torch.int32, (W, g), (rs // 4, 1))
            self.moe_w = view(m.g_w, torch.float32, (W, g), (rs // 4, 1))
            self.moe_y = view(m.yg, torch.bfloat16, (W, g, H), (rs // 2, H, 1))
            self.moe_entry_slot = view(m.entry_slot, torch.int32, (W, cap, k), (rs // 4, k, 1))
            self.moe_count = view(m.count, torch.int32, (W, Er), (Er, 1))
            self.moe_offset = view(m.offset, torch.int32, (W, Er), (Er, 1))

    def epochs(self):
        o = _lib.EpDispatchOutC()
        check(self.L.ep_dispatch_outputs(self.h, ctypes.byref(o)),
              "ep_dispatch_outputs")
        return o.dispatch_epoch, o.combine_epoch

    # ------------------------------------------------------- helpers
    def _counts(self, num_tokens):
        c = self.config
        if num_tokens is None:
            num_tokens = [c.max_tokens_per_rank] * c.world_size
        arr = (ctypes.c_int32 * c.world_size)(*[int(n) for n in num_tokens])
        return arr

    def _check_inputs(self, x, w, idx, scales=None):
        c = self.config
        W, T, H, k = c.world_size, c.max_tokens_per_rank, c.hidden, c.topk
        if scales is not None:
            # pre-quantised input: E4M3 codes (uint8 or float8_e4m3fn) + scales
            if c.dispatch_dtype != "fp8_e4m3":
                raise ValueError("scales (pre-quantised input) need an fp8_e4m3 dispatch")
            if x.element_size() != 1 or tuple(x.shape) != (W, T, H) or not x.is_contiguous():
                raise ValueError(f"pre-quantised input must be contiguous 1-byte [{W},{T},{H}]")
            if scales.dtype != torch.float32 or tuple(scales.shape) != (W, T, H // 128) \
                    or not scales.is_contiguous() or scales.device != self.device:
                raise ValueError(f"scales must be contiguous fp32 [{W},{T},{H // 128}]")
        elif x.dtype != torch.bfloat16 or tuple(x.shape) != (W, T, H) or not x.is_contiguous():
            raise ValueError(f"input must be contiguous bf16 [{W},{T},{H}]")
        if w.dtype != torch.float32 or tuple(w.shape) != (W, T, k) or not w.is_contiguous():
            raise ValueError(f"weights must be contiguous fp32 [{W},{T},{k}]")
        if idx.dtype != torch.int32 or tuple(idx.shape) != (W, T, k) or not idx.is_contiguous():
            raise ValueError(f"indices must be contiguous int32 [{W},{T},{k}]")
        for t in (x, w, idx):
            if t.device != self.device:
                raise ValueError("inputs must be on the op's device")

    def _dispatch_result(self):
        return (self.out, self.out_w, self.out_scales, self.out_idx,
                self.recv_count)

    # ------------------------------------------------------- methods
    def layout(self, indices, num_tokens=None, stream=None):
        check(self.L.ep_layout(self.h, _ptr(indices), self._counts(num_tokens),
                               _stream(stream)), "ep_layout")

    def dispatch(self, input, weights, scales=None, indices=None,
                 num_tokens: Optional[Sequence[int]] = None, stream=None):
        """Send each token to the ranks that hold its experts.  Returns
        (output, weights, scales, indices, recv_count): per-rank views
        [W][cap][...] into the receive segments (valid until the next
        dispatch / reset) and recv_count [W].
        Rows p >= recv_count[r] of rank r are unspecified."""
        self._check_inputs(input, weights, indices, scales)
        check(self.L.ep_dispatch(self.h, _ptr(input), _ptr(weights),
                                 _ptr(scales), _ptr(indices),
                                 self._counts(num_tokens), _stream(stream)),
              "ep_dispatch")
        return self._dispatch_result()

    def dispatch_send(self, input, weights, scales=None, indices=None,
                      num_tokens=None, stream=None):
        self._check_inputs(input, weights, indices, scales)
        check(self.L.ep_dispatch_send(self.h, _ptr(input), _ptr(weights),
                                      _ptr(scales), _ptr(indices),
                                      self._counts(num_tokens), _stream(stream)),
              "ep_dispatch_send")

    def dispatch_send_replay(self, input, weights, indices, num_tokens=None,
                             stream=None, scales=None):
        """Routing replay: copy with the cached layout of the last call."""
        self._check_inputs(input, weights, indices, scales)
        check(self.L.ep_dispatch_send_replay(self.h, _ptr(input), _ptr(weights),
                                             _ptr(scales), _ptr(indices),
                                             self._counts(num_tokens),
                                             _stream(stream)),
              "ep_dispatch_send_replay")

    def dispatch_recv(self, stream=None):
        check(self.L.ep_dispatch_recv(self.h, _stream(stream)), "ep_dispatch_recv")
        return self._dispatch_result()

    def _combine_call(self, fn, input, weights, indices, out, out_weights,
                      stream, what):
        c = self.config
        W, T, H, k = c.world_size, c.max_tokens_per_rank, c.hidden, c.topk
        if out is None:
            out = torch.empty((W, T, H), dtype=torch.bfloat16, device=self.device)
        if weights is not None and out_weights is None:
            out_weights = torch.empty((W, T, k), dtype=torch.float32,
                                      device=self.device)
        ys = 0
        if input is not None and self.config.combine_dtype == "fp8_e4m3":
            raise ValueError("an FP8 combine payload is read from the registered buffer")
        if input is not None:
            if input.dtype != self.y_dtype or input.dim() != 3 or \
                    input.shape[0] != W or input.shape[2] != H or input.stride(2) != 1 \
                    or input.stride(1) != H:
                raise ValueError(f"combine input must be {self.y_dtype} [W][>=cap][H] "
                                 "with dense rows")
            ys = input.stride(0) * input.element_size()
        ws = 0
        if weights is not None:
            if weights.dtype != torch.float32 or weights.dim() != 3 or \
                    weights.shape[2] != k or weights.stride(2) != 1 or weights.stride(1) != k:
                raise ValueError("combine weights must be fp32 [W][>=cap][k] with dense rows")
            ws = weights.stride(0) * 4
        check(fn(self.h, _ptr(input), ys, _ptr(weights), ws, _ptr(indices),
                 _ptr(out), _ptr(out_weights), _stream(stream)), what)
        return out, out_weights

    def combine(self, input=None, weights=None, indices=None, out=None,
                out_weights=None, stream=None):
        """Bring the experts' results back to the source tokens.  input: None
        for the registered combine buffer, else bf16 [W][cap][H] expert rows
        per rank.  Returns
        (output [W][T][H] bf16, weights [W][T][k] fp32 or None)."""
        return self._combine_call(self.L.ep_combine, input, weights, indices,
                                  out, out_weights, stream, "ep_combine")

    def combine_send(self, stream=None):
        check(self.L.ep_combine_send(self.h, _stream(stream)), "ep_combine_send")

    def combine_recv(self, input=None, weights=None, indices=None, out=None,
                     out_weights=None, stream=None):
        return self._combine_call(self.L.ep_combine_recv, input, weights,
                                  indices, out, out_weights, stream,
                                  "ep_combine_recv")

    def moe_group(self, stream=None):
        """Standard-MoE conversion: group the received rows per local expert.
        Returns (grouped payload [W][gcap][H], grouped scales or None,
        counts [W][Er], offsets [W][Er])."""
        check(self.L.ep_moe_group(self.h, _stream(stream)), "ep_moe_group")
        return self.moe_x, self.moe_x_scales, self.moe_count, self.moe_offset

    def moe_ungroup(self, y=None, stream=None):
        """Weighted per-row sums of the grouped expert outputs (y: None for the
        registered moe_y buffer) into the registered combine input buffer."""
        ys = 0 if y is None else y.stride(0) * 2
        check(self.L.ep_moe_ungroup(self.h, _ptr(y), ys, _stream(stream)), "ep_moe_ungroup")
        return self.combine_input

    def reset(self, stream=None):
        check(self.L.ep_reset(self.h, _stream(stream)), "ep_reset")

    def get_dispatch_src_token_pos(self):
        """Source position s*T + t of every received row, int32 [W][cap]."""
        return self.src_pos

    def get_registered_combine_input_buffer(self, dtype=None):
        if dtype is not None and dtype != self.y_dtype:
            raise EpError(4, "get_registered_combine_input_buffer")
        return self.combine_input

    def get_error(self, stream=None):
        """Synchronise and read/clear the device error word: (status, mask)."""
        m = ctypes.c_uint32(0)
        st = self.L.ep_get_error(self.h, ctypes.byref(m), _stream(stream))
        if st == _lib.EP_ERR_GPU_OP:
            raise EpError(st, "ep_get_error")
        return st, m.value

    def identity_expert(self, y=None, stream=None):
        """Test harness: y_r = rows scaled by their rank-local weight sum."""
        ys = 0 if y is None else y.stride(0) * y.element_size()
        check(self.L.ep_test_identity_expert(self.h, _ptr(y), ys, _stream(stream)),
              "ep_test_identity_expert")
        return self.combine_input if y is None else y

    def close(self):
        if getattr(self, "h", None):
            self.L.ep_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
