// Host side of the C ABI declared in include/ep_api.h: config validation,
// workspace carving into W symmetric rank segments, the send/receive state
// machine, argument checks and kernel launches.  Nothing here allocates
// device memory; the caller owns the workspace.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "ep_internal.cuh"

using namespace ep;

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxHidden = 1 << 24;
size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool aligned(const void *p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

int env_flag(const char *name, int dflt) {
    const char *v = std::getenv(name);
    if (!v || !*v) return dflt;
    return std::atoi(v) != 0 ? 1 : 0;
}

ep_status_t make_config(const ep_config_t *in, Config *c) {
    if (!in || !c) return EP_ERR_INVALID_ARGS;
    const int W = in->world_size, E = in->num_experts, k = in->topk;
    const int H = in->hidden, T = in->max_tokens_per_rank;
    if (W < 1 || W > EP_MAX_WORLD) return EP_ERR_INVALID_ARGS;
    if (E < W || E % W != 0) return EP_ERR_INVALID_ARGS;
    if (k < 1 || k > EP_MAX_TOPK) return EP_ERR_INVALID_ARGS;
    // H <= 2^24 keeps a row's byte count (up to 4 H for fp32 rows) in an int
    if (H < 8 || H % 8 != 0 || H > kMaxHidden) return EP_ERR_INVALID_ARGS;
    if (T < 1) return EP_ERR_INVALID_ARGS;
    if (in->dispatch_dtype != EP_DT_BF16 && in->dispatch_dtype != EP_DT_FP8_E4M3)
        return EP_ERR_INVALID_ARGS;
    const bool fp8 = in->dispatch_dtype == EP_DT_FP8_E4M3;
    if (in->combine_dtype != EP_DT_BF16 && in->combine_dtype != EP_DT_FP32 &&
        in->combine_dtype != EP_DT_FP8_E4M3)
        return EP_ERR_INVALID_ARGS;
    if (in->combine_dtype == EP_DT_FP8_E4M3 && H % EP_QUANT_BLOCK != 0)
        return EP_ERR_INVALID_ARGS;
    if (fp8 && (H % EP_QUANT_BLOCK != 0 || H > 16384)) return EP_ERR_INVALID_ARGS;
    const int64_t cap = in->max_recv_tokens_per_rank > 0
                            ? in->max_recv_tokens_per_rank
                            : (int64_t)W * T;
    if (in->max_recv_tokens_per_rank < 0 || cap > (int64_t)1 << 30 ||
        (int64_t)W * T > (int64_t)1 << 30)
        return EP_ERR_INVALID_ARGS;
    c->W = W; c->E = E; c->Er = E / W; c->k = k; c->H = H; c->T = T;
    c->cap = (int)cap;
    c->fp8 = fp8;
    c->y_f32 = in->combine_dtype == EP_DT_FP32;
    c->y_fp8 = in->combine_dtype == EP_DT_FP8_E4M3;
    c->nch = (T + kChunk - 1) / kChunk;
    c->G = W * c->nch;
    c->Q = (c->G + kGroup - 1) / kGroup;
    c->nvec = H / 8;
    c->nb = fp8 ? H / EP_QUANT_BLOCK : 0;
    c->early_notify = env_flag("EP_EARLY_NOTIFY", in->early_notify ? 1 : 0) != 0;
    c->fused_recv = env_flag("EP_FUSED_RECV", in->fused_recv ? 1 : 0) != 0;
    if (c->fused_recv && !c->early_notify) return EP_ERR_INVALID_ARGS;
    c->timeout_ns = in->wait_timeout_ns > 0 ? in->wait_timeout_ns : 1000000000LL;
    if (in->max_grouped_rows_per_rank < 0 ||
        (int64_t)in->max_grouped_rows_per_rank > (int64_t)1 << 30)
        return EP_ERR_INVALID_ARGS;
    c->gcap = in->max_grouped_rows_per_rank;
    if (in->combine_mode != EP_COMBINE_GATHER && in->combine_mode != EP_COMBINE_SCATTER)
        return EP_ERR_INVALID_ARGS;
    c->scatter = in->combine_mode == EP_COMBINE_SCATTER;
    if (c->scatter && (c->y_f32 || c->y_fp8)) return EP_ERR_INVALID_ARGS;
    c->maxd = W < k ? W : k;
    c->nrc = (c->cap + kChunk - 1) / kChunk;
    return EP_SUCCESS;
}

bool read_counts(const ep_handle_t *h, const int32_t *h_nt, TokenCounts *nt) {
    if (!h_nt) return false;
    std::memset(nt, 0, sizeof(*nt));
    for (int s = 0; s < h->cfg.W; ++s) {
        if (h_nt[s] < 0 || h_nt[s] > h->cfg.T) return false;
        nt->n[s] = h_nt[s];
    }
    return true;
}

ep_status_t gpu(ep_handle_t *h, cudaError_t e, const char *what) {
    if (e == cudaSuccess) return EP_SUCCESS;
    if (!h || h->log_level >= 1)
        std::fprintf(stderr, "[ep] %s: %s\n", what, cudaGetErrorString(e));
    return EP_ERR_GPU_OP;
}

}  // namespace

namespace ep {

void plan_workspace(const Config &c, char *base, Workspace *ws) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes);
        return base ? base + o : nullptr;
    };
    const size_t W = c.W, T = c.T, G = c.G;
    ws->words = reinterpret_cast<uint32_t *>(take(kCounterWords * 4));
    ws->dflags = reinterpret_cast<uint32_t *>(take(W * W * 4));
    ws->cflags = reinterpret_cast<uint32_t *>(take(W * W * 4));
    const size_t Q = c.Q;
    ws->chunk_local = reinterpret_cast<int32_t *>(take(G * W * 4));
    ws->group_tot = reinterpret_cast<int32_t *>(take(Q * W * 4));
    ws->group_base = reinterpret_cast<int32_t *>(take((Q + 1) * W * 4));
    ws->send_counts = reinterpret_cast<int32_t *>(take(W * W * 4));
    ws->recv_count = reinterpret_cast<int32_t *>(take(W * 4));
    ws->masks = reinterpret_cast<uint32_t *>(take(W * T * 4));
    ws->pos = reinterpret_cast<int32_t *>(take(W * T * W * 4));
    const size_t Er = c.Er, nrc = c.gcap ? c.nrc : 0;
    const bool moe = c.gcap > 0;
    ws->moe_cnt = reinterpret_cast<int32_t *>(take(W * nrc * Er * 4));
    ws->moe_base = reinterpret_cast<int32_t *>(take(W * nrc * Er * 4));
    ws->moe_count = reinterpret_cast<int32_t *>(take(moe ? W * Er * 4 : 0));
    ws->moe_offset = reinterpret_cast<int32_t *>(take(moe ? W * Er * 4 : 0));
    ws->stage = take(c.scatter ? W * T * (size_t)c.maxd * c.H * 2 : 0);
    // one rank segment
    const size_t cap = c.cap, H = c.H, k = c.k;
    size_t so = 0;
    auto seg_take = [&](size_t bytes) {
        const size_t o = so;
        so = align_up(so + bytes);
        return (int64_t)o;
    };
    ws->off_out = seg_take(cap * H * (c.fp8 ? 1 : 2));
    ws->off_scales = seg_take(c.fp8 ? cap * c.nb * 4 : 0);
    ws->off_w = seg_take(cap * k * 4);
    ws->off_idx = seg_take(cap * k * 4);
    ws->off_src = seg_take(cap * 4);
    ws->off_comb = seg_take(cap * H * (c.y_f32 ? 4 : (c.y_fp8 ? 1 : 2)));
    ws->off_comb_sc = seg_take(c.y_fp8 ? cap * (H / EP_QUANT_BLOCK) * 4 : 0);
    const size_t gc = c.gcap;
    ws->off_xg = seg_take(gc * H * (c.fp8 ? 1 : 2));
    ws->off_xgs = seg_take(c.fp8 ? gc * c.nb * 4 : 0);
    ws->off_gsrc = seg_take(gc * 4);
    ws->off_gw = seg_take(gc * 4);
    ws->off_yg = seg_take(gc * H * 2);
    ws->off_eslot = seg_take(moe ? cap * k * 4 : 0);
    ws->seg_stride = (int64_t)so;
    ws->seg0 = base ? base + off : nullptr;
    ws->total_bytes = off + so * W;
}

}  // namespace ep

extern "C" {

const char *ep_status_str(ep_status_t s) {
    switch (s) {
        case EP_SUCCESS: return "EP_SUCCESS";
        case EP_INIT: return "EP_INIT";
        case EP_IN_PROGRESS: return "EP_IN_PROGRESS";
        case EP_ERR_INVALID_ARGS: return "EP_ERR_INVALID_ARGS";
        case EP_ERR_NOT_FOUND: return "EP_ERR_NOT_FOUND";
        case EP_ERR_RDMA_OP: return "EP_ERR_RDMA_OP";
        case EP_ERR_BAD_STATE: return "EP_ERR_BAD_STATE";
        case EP_ERR_GPU_OP: return "EP_ERR_GPU_OP";
        case EP_ERR_TIMEOUT: return "EP_ERR_TIMEOUT";
        case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY";
        case EP_ERR_BAD_INDEX: return "EP_ERR_BAD_INDEX";
    }
    return "EP_UNKNOWN";
}

ep_status_t ep_workspace_size(const ep_config_t *cfg, size_t *bytes) {
    if (!bytes) return EP_ERR_INVALID_ARGS;
    Config c;
    const ep_status_t st = make_config(cfg, &c);
    if (st != EP_SUCCESS) return st;
    Workspace ws;
    plan_workspace(c, nullptr, &ws);
    *bytes = ws.total_bytes;
    return EP_SUCCESS;
}

ep_status_t ep_create(const ep_config_t *cfg, void *d_workspace, size_t bytes,
                      ep_handle_t **out) {
    EP_RANGE("ep_create");
    if (!out || !d_workspace || !aligned(d_workspace, kAlign))
        return EP_ERR_INVALID_ARGS;
    *out = nullptr;
    Config c;
    ep_status_t st = make_config(cfg, &c);
    if (st != EP_SUCCESS) return st;
    Workspace ws;
    plan_workspace(c, static_cast<char *>(d_workspace), &ws);
    if (bytes < ws.total_bytes) return EP_ERR_INVALID_ARGS;
    ep_handle_t *h = new (std::nothrow) ep_handle_t();
    if (!h) return EP_ERR_INVALID_ARGS;
    h->cfg = c;
    h->ws = ws;
    h->log_level = 0;
    if (const char *lv = std::getenv("EP_LOG_LEVEL")) h->log_level = std::atoi(lv);
    cudaGetDevice(&h->device);
    st = gpu(h, cudaEventCreateWithFlags(&h->ev_dispatch_sent, cudaEventDisableTiming),
             "cudaEventCreate");
    if (st == EP_SUCCESS)
        st = gpu(h, cudaEventCreateWithFlags(&h->ev_combine_sent, cudaEventDisableTiming),
                 "cudaEventCreate");
    // one pinned host word for ep_get_error's stream-ordered read
    if (st == EP_SUCCESS)
        st = gpu(h, cudaHostAlloc(reinterpret_cast<void **>(&h->h_err), sizeof(uint32_t),
                                  cudaHostAllocDefault),
                 "cudaHostAlloc");
    // zero the counters, flags and error word (everything before chunk_local)
    if (st == EP_SUCCESS)
        st = gpu(h, cudaMemset(ws.words, 0,
                               reinterpret_cast<char *>(ws.chunk_local) -
                                   reinterpret_cast<char *>(ws.words)),
                 "cudaMemset");
    if (st == EP_SUCCESS) st = gpu(h, cudaDeviceSynchronize(), "cudaDeviceSynchronize");
    if (st != EP_SUCCESS) {
        ep_destroy(h);
        return st;
    }
    if (h->log_level >= 2)
        std::fprintf(stderr,
                     "[ep] create W=%d E=%d k=%d H=%d T=%d cap=%d fp8=%d "
                     "early_notify=%d fused_recv=%d workspace=%zu B\n",
                     c.W, c.E, c.k, c.H, c.T, c.cap, (int)c.fp8,
                     (int)c.early_notify, (int)c.fused_recv, ws.total_bytes);
    *out = h;
    return EP_SUCCESS;
}

ep_status_t ep_destroy(ep_handle_t *h) {
    EP_RANGE("ep_destroy");
    if (!h) return EP_ERR_INVALID_ARGS;
    if (h->ev_dispatch_sent) cudaEventDestroy(h->ev_dispatch_sent);
    if (h->ev_combine_sent) cudaEventDestroy(h->ev_combine_sent);
    if (h->h_err) cudaFreeHost(h->h_err);
    delete h;
    return EP_SUCCESS;
}

ep_status_t ep_layout(ep_handle_t *h, const int32_t *d_idx,
                      const int32_t *h_num_tokens, void *stream) {
    EP_RANGE("ep_layout");
    if (!h || !d_idx || !aligned(d_idx, 4)) return EP_ERR_INVALID_ARGS;
    TokenCounts nt;
    if (!read_counts(h, h_num_tokens, &nt)) return EP_ERR_INVALID_ARGS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const ep_status_t s = gpu(h, launch_layout(h->cfg, h->ws, d_idx, nt, st, true),
                              "layout");
    if (s != EP_SUCCESS) return s;
    h->layout_valid = true;
    h->layout_nt = nt;
    return EP_SUCCESS;
}

static ep_status_t check_dispatch_args(ep_handle_t *h, const void *d_x,
                                       const float *d_w, const float *d_scales,
                                       const int32_t *d_idx) {
    if (!h || !d_x || !d_w || !d_idx) return EP_ERR_INVALID_ARGS;
    // pre-quantised input (codes + block scales) needs an FP8 dispatch
    if (d_scales && (!h->cfg.fp8 || !aligned(d_scales, 16))) return EP_ERR_INVALID_ARGS;
    if (!aligned(d_x, 16) || !aligned(d_w, 4) || !aligned(d_idx, 4))
        return EP_ERR_INVALID_ARGS;
    return EP_SUCCESS;
}

static ep_status_t dispatch_send_impl(ep_handle_t *h, const void *d_x,
                                      const float *d_w, const float *d_scales,
                                      const int32_t *d_idx,
                                      const TokenCounts &nt, bool run_layout,
                                      bool publish, cudaStream_t st) {
    if (h->cfg.early_notify) ++h->dispatch_epoch;
    h->moe_valid = false;             // a grouping belongs to one dispatch
    // few chunks: the copy kernel computes the layout itself (no layout kernel)
    const bool self_layout = run_layout && h->cfg.G <= self_layout_chunks();
    if (run_layout && !self_layout) {
        const ep_status_t s =
            gpu(h, launch_layout(h->cfg, h->ws, d_idx, nt, st, publish), "layout");
        if (s != EP_SUCCESS) return s;
    }
    DispatchArgs a;
    a.x = d_x;
    a.scales_in = d_scales;
    a.w = d_w;
    a.idx = d_idx;
    a.nt = nt;
    a.epoch = h->dispatch_epoch;
    a.after_layout = run_layout && !self_layout;
    a.self_layout = self_layout;
    a.publish = publish;
    const ep_status_t s = gpu(h, launch_dispatch(h->cfg, h->ws, a, st), "dispatch");
    if (s != EP_SUCCESS) return s;
    if (run_layout) {
        h->layout_valid = true;
        h->layout_nt = nt;
    }
    return EP_SUCCESS;
}

ep_status_t ep_dispatch_send(ep_handle_t *h, const void *d_x, const float *d_w,
                             const float *d_scales, const int32_t *d_idx,
                             const int32_t *h_num_tokens, void *stream) {
    EP_RANGE("ep_dispatch_send");
    ep_status_t s = check_dispatch_args(h, d_x, d_w, d_scales, d_idx);
    if (s != EP_SUCCESS) return s;
    TokenCounts nt;
    if (!read_counts(h, h_num_tokens, &nt)) return EP_ERR_INVALID_ARGS;
    if (h->dispatch_pending) return EP_ERR_BAD_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Without early notification the layout kernel produces recv_count
    // itself and the receive phase is stream order alone; with it, the
    // receive step checks the ready flags and then writes the count.
    s = dispatch_send_impl(h, d_x, d_w, d_scales, d_idx, nt, true,
                           !h->cfg.early_notify, st);
    if (s != EP_SUCCESS) return s;
    s = gpu(h, cudaEventRecord(h->ev_dispatch_sent, st), "cudaEventRecord");
    if (s != EP_SUCCESS) return s;
    h->dispatch_pending = true;
    return EP_SUCCESS;
}

ep_status_t ep_dispatch_send_replay(ep_handle_t *h, const void *d_x,
                                    const float *d_w, const float *d_scales,
                                    const int32_t *d_idx,
                                    const int32_t *h_num_tokens, void *stream) {
    EP_RANGE("ep_dispatch_send_replay");
    ep_status_t s = check_dispatch_args(h, d_x, d_w, d_scales, d_idx);
    if (s != EP_SUCCESS) return s;
    TokenCounts nt;
    if (!read_counts(h, h_num_tokens, &nt)) return EP_ERR_INVALID_ARGS;
    if (!h->layout_valid || h->dispatch_pending) return EP_ERR_BAD_STATE;
    if (std::memcmp(&nt, &h->layout_nt, sizeof(nt)) != 0) return EP_ERR_BAD_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = dispatch_send_impl(h, d_x, d_w, d_scales, d_idx, nt, false, false, st);
    if (s != EP_SUCCESS) return s;
    s = gpu(h, cudaEventRecord(h->ev_dispatch_sent, st), "cudaEventRecord");
    if (s != EP_SUCCESS) return s;
    h->dispatch_pending = true;
    return EP_SUCCESS;
}

ep_status_t ep_dispatch_recv(ep_handle_t *h, void *stream) {
    EP_RANGE("ep_dispatch_recv");
    if (!h) return EP_ERR_INVALID_ARGS;
    if (!h->dispatch_pending) return EP_ERR_BAD_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ep_status_t s = gpu(h, cudaStreamWaitEvent(st, h->ev_dispatch_sent, 0),
                        "cudaStreamWaitEvent");
    if (s != EP_SUCCESS) return s;
    if (h->cfg.early_notify) {
        s = gpu(h, launch_dispatch_recv(h->cfg, h->ws, true, h->dispatch_epoch, st),
                "dispatch_recv");
        if (s != EP_SUCCESS) return s;
    }
    h->dispatch_pending = false;
    return EP_SUCCESS;
}

ep_status_t ep_dispatch(ep_handle_t *h, const void *d_x, const float *d_w,
                        const float *d_scales, const int32_t *d_idx,
                        const int32_t *h_num_tokens, void *stream) {
    EP_RANGE("ep_dispatch");
    ep_status_t s = check_dispatch_args(h, d_x, d_w, d_scales, d_idx);
    if (s != EP_SUCCESS) return s;
    TokenCounts nt;
    if (!read_counts(h, h_num_tokens, &nt)) return EP_ERR_INVALID_ARGS;
    if (h->dispatch_pending) return EP_ERR_BAD_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // One stream: the layout publishes recv_count itself unless the ready
    // flags must be checked by a receive step.
    const bool notify = h->cfg.early_notify;
    s = dispatch_send_impl(h, d_x, d_w, d_scales, d_idx, nt, true, !notify, st);
    if (s != EP_SUCCESS) return s;
    if (notify)
        s = gpu(h, launch_dispatch_recv(h->cfg, h->ws, true, h->dispatch_epoch, st),
                "dispatch_recv");
    return s;
}

ep_status_t ep_dispatch_outputs(const ep_handle_t *h, ep_dispatch_out_t *o) {
    if (!h || !o) return EP_ERR_INVALID_ARGS;
    const Workspace &ws = h->ws;
    o->out = ws.seg0 + ws.off_out;
    o->out_scales = h->cfg.fp8 ? reinterpret_cast<float *>(ws.seg0 + ws.off_scales) : nullptr;
    o->out_w = reinterpret_cast<float *>(ws.seg0 + ws.off_w);
    o->out_idx = reinterpret_cast<int32_t *>(ws.seg0 + ws.off_idx);
    o->src_pos = reinterpret_cast<int32_t *>(ws.seg0 + ws.off_src);
    o->rank_stride_bytes = ws.seg_stride;
    o->recv_count = ws.recv_count;
    o->send_counts = ws.send_counts;
    o->pos = ws.pos;
    o->dispatch_flags = ws.dflags;
    o->combine_flags = ws.cflags;
    o->dispatch_epoch = h->dispatch_epoch;
    o->combine_epoch = h->combine_epoch;
    o->cap = h->cfg.cap;
    o->max_dest = h->cfg.maxd;
    o->combine_stage = h->cfg.scatter ? ws.stage : nullptr;
    return EP_SUCCESS;
}

ep_status_t ep_get_combine_input_buffer(const ep_handle_t *h, int32_t dtype,
                                        void **d_ptr, int64_t *rank_stride_bytes) {
    if (!h || !d_ptr || !rank_stride_bytes) return EP_ERR_INVALID_ARGS;
    if (dtype != (h->cfg.y_f32 ? EP_DT_FP32 : (h->cfg.y_fp8 ? EP_DT_FP8_E4M3 : EP_DT_BF16)))
        return EP_ERR_NOT_FOUND;
    *d_ptr = h->ws.seg0 + h->ws.off_comb;
    *rank_stride_bytes = h->ws.seg_stride;
    return EP_SUCCESS;
}

ep_status_t ep_get_combine_input_scales(const ep_handle_t *h, float **d_ptr,
                                        int64_t *rank_stride_bytes) {
    if (!h || !d_ptr || !rank_stride_bytes) return EP_ERR_INVALID_ARGS;
    if (!h->cfg.y_fp8) return EP_ERR_NOT_FOUND;
    *d_ptr = reinterpret_cast<float *>(h->ws.seg0 + h->ws.off_comb_sc);
    *rank_stride_bytes = h->ws.seg_stride;
    return EP_SUCCESS;
}

ep_status_t ep_combine_send(ep_handle_t *h, void *stream) {
    EP_RANGE("ep_combine_send");
    if (!h) return EP_ERR_INVALID_ARGS;
    // the dispatch's receive phase must be enqueued first: it orders the
    // expert side after the send's layout and copy
    if (!h->layout_valid || h->dispatch_pending || h->combine_pending)
        return EP_ERR_BAD_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (h->cfg.scatter) {
        const ep_status_t s = gpu(h, launch_scatter_send(h->cfg, h->ws, st), "scatter_send");
        if (s != EP_SUCCESS) return s;
    }
    if (h->cfg.early_notify) {
        ++h->combine_epoch;
        const ep_status_t s = gpu(h, launch_combine_notify(h->cfg, h->ws, h->combine_epoch, st),
                                  "combine_notify");
        if (s != EP_SUCCESS) return s;
    }
    const ep_status_t s = gpu(h, cudaEventRecord(h->ev_combine_sent, st), "cudaEventRecord");
    if (s != EP_SUCCESS) return s;
    h->combine_pending = true;
    return EP_SUCCESS;
}

static ep_status_t combine_args(ep_handle_t *h, const void *d_y, int64_t y_stride,
                                const float *d_w_in, int64_t w_stride,
                                const int32_t *d_idx, void *d_out, float *d_out_w,
                                CombineArgs *a) {
    const Config &c = h->cfg;
    if (!d_out || !aligned(d_out, 16)) return EP_ERR_INVALID_ARGS;
    if (d_idx && !aligned(d_idx, 4)) return EP_ERR_INVALID_ARGS;
    if ((d_w_in == nullptr) != (d_out_w == nullptr)) return EP_ERR_INVALID_ARGS;
    const int64_t row_bytes = (int64_t)c.cap * c.H * (c.y_f32 ? 4 : 2);
    a->ysc = h->ws.seg0 + h->ws.off_comb_sc;
    a->stage = c.scatter ? h->ws.stage : nullptr;
    // FP8 payload and scatter mode: the registered buffer only
    if (d_y && (c.y_fp8 || c.scatter)) return EP_ERR_INVALID_ARGS;
    if (d_y) {
        if (y_stride == 0) y_stride = row_bytes;
        if (!aligned(d_y, 16) || y_stride % 16 != 0 || y_stride < row_bytes)
            return EP_ERR_INVALID_ARGS;
        a->y = static_cast<const char *>(d_y);
        a->y_stride = y_stride;
    } else {
        a->y = h->ws.seg0 + h->ws.off_comb;
        a->y_stride = h->ws.seg_stride;
    }
    if (d_w_in) {
        const int64_t wrow = (int64_t)c.cap * c.k * 4;
        if (w_stride == 0) w_stride = wrow;
        if (!aligned(d_w_in, 4) || !aligned(d_out_w, 4) || w_stride % 4 != 0 ||
            w_stride < wrow)
            return EP_ERR_INVALID_ARGS;
    }
    a->w_in = reinterpret_cast<const char *>(d_w_in);
    a->w_stride = w_stride;
    a->idx = d_idx;
    a->out = static_cast<uint16_t *>(d_out);
    a->out_w = d_out_w;
    a->nt = h->layout_nt;
    a->fused_wait = false;
    a->epoch = h->combine_epoch;
    return EP_SUCCESS;
}

ep_status_t ep_combine_recv(ep_handle_t *h, const void *d_y,
                            int64_t y_rank_stride_bytes, const float *d_w_in,
                            int64_t w_rank_stride_bytes, const int32_t *d_idx,
                            void *d_out, float *d_out_w, void *stream) {
    EP_RANGE("ep_combine_recv");
    if (!h) return EP_ERR_INVALID_ARGS;
    CombineArgs a;
    ep_status_t s = combine_args(h, d_y, y_rank_stride_bytes, d_w_in,
                                 w_rank_stride_bytes, d_idx, d_out, d_out_w, &a);
    if (s != EP_SUCCESS) return s;
    if (!h->layout_valid || !h->combine_pending) return EP_ERR_BAD_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = gpu(h, cudaStreamWaitEvent(st, h->ev_combine_sent, 0), "cudaStreamWaitEvent");
    if (s != EP_SUCCESS) return s;
    if (h->cfg.early_notify && !h->cfg.fused_recv) {
        s = gpu(h, launch_combine_wait(h->cfg, h->ws, h->combine_epoch, st), "combine_wait");
        if (s != EP_SUCCESS) return s;
    }
    a.fused_wait = h->cfg.early_notify && h->cfg.fused_recv;
    s = gpu(h, launch_combine(h->cfg, h->ws, a, st), "combine");
    if (s != EP_SUCCESS) return s;
    h->combine_pending = false;
    return EP_SUCCESS;
}

ep_status_t ep_combine(ep_handle_t *h, const void *d_y, int64_t y_rank_stride_bytes,
                       const float *d_w_in, int64_t w_rank_stride_bytes,
                       const int32_t *d_idx, void *d_out, float *d_out_w,
                       void *stream) {
    EP_RANGE("ep_combine");
    if (!h) return EP_ERR_INVALID_ARGS;
    CombineArgs a;
    ep_status_t s = combine_args(h, d_y, y_rank_stride_bytes, d_w_in,
                                 w_rank_stride_bytes, d_idx, d_out, d_out_w, &a);
    if (s != EP_SUCCESS) return s;
    if (!h->layout_valid || h->dispatch_pending || h->combine_pending)
        return EP_ERR_BAD_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (h->cfg.scatter) {
        s = gpu(h, launch_scatter_send(h->cfg, h->ws, st), "scatter_send");
        if (s != EP_SUCCESS) return s;
    }
    if (h->cfg.early_notify) {
        ++h->combine_epoch;
        a.epoch = h->combine_epoch;
        s = gpu(h, launch_combine_notify(h->cfg, h->ws, h->combine_epoch, st),
                "combine_notify");
        if (s != EP_SUCCESS) return s;
        if (!h->cfg.fused_recv) {
            s = gpu(h, launch_combine_wait(h->cfg, h->ws, h->combine_epoch, st),
                    "combine_wait");
            if (s != EP_SUCCESS) return s;
        }
        a.fused_wait = h->cfg.fused_recv;
    }
    return gpu(h, launch_combine(h->cfg, h->ws, a, st), "combine");
}

ep_status_t ep_moe_group(ep_handle_t *h, void *stream) {
    EP_RANGE("ep_moe_group");
    if (!h) return EP_ERR_INVALID_ARGS;
    if (h->cfg.gcap <= 0) return EP_ERR_INVALID_ARGS;
    if (!h->layout_valid || h->dispatch_pending) return EP_ERR_BAD_STATE;
    const ep_status_t s = gpu(h, launch_moe_group(h->cfg, h->ws, static_cast<cudaStream_t>(stream)),
                              "moe_group");
    if (s == EP_SUCCESS) h->moe_valid = true;
    return s;
}

ep_status_t ep_moe_outputs(const ep_handle_t *h, ep_moe_out_t *o) {
    if (!h || !o) return EP_ERR_INVALID_ARGS;
    if (h->cfg.gcap <= 0) return EP_ERR_INVALID_ARGS;
    const Workspace &ws = h->ws;
    o->xg = ws.seg0 + ws.off_xg;
    o->xg_scales = h->cfg.fp8 ? reinterpret_cast<float *>(ws.seg0 + ws.off_xgs) : nullptr;
    o->g_src = reinterpret_cast<int32_t *>(ws.seg0 + ws.off_gsrc);
    o->g_w = reinterpret_cast<float *>(ws.seg0 + ws.off_gw);
    o->yg = ws.seg0 + ws.off_yg;
    o->entry_slot = reinterpret_cast<int32_t *>(ws.seg0 + ws.off_eslot);
    o->rank_stride_bytes = ws.seg_stride;
    o->count = ws.moe_count;
    o->offset = ws.moe_offset;
    o->gcap = h->cfg.gcap;
    o->experts_per_rank = h->cfg.Er;
    return EP_SUCCESS;
}

ep_status_t ep_moe_ungroup(ep_handle_t *h, const void *d_yg, int64_t yg_stride,
                           void *stream) {
    EP_RANGE("ep_moe_ungroup");
    if (!h) return EP_ERR_INVALID_ARGS;
    const Config &c = h->cfg;
    if (c.gcap <= 0 || c.y_f32 || c.y_fp8) return EP_ERR_INVALID_ARGS;
    const int64_t rows = (int64_t)c.gcap * c.H * 2;
    const char *yg;
    if (d_yg) {
        if (yg_stride == 0) yg_stride = rows;
        if (!aligned(d_yg, 16) || yg_stride % 16 != 0 || yg_stride < rows)
            return EP_ERR_INVALID_ARGS;
        yg = static_cast<const char *>(d_yg);
    } else {
        yg = h->ws.seg0 + h->ws.off_yg;
        yg_stride = h->ws.seg_stride;
    }
    if (!h->moe_valid || !h->layout_valid) return EP_ERR_BAD_STATE;
    return gpu(h, launch_moe_ungroup(c, h->ws, yg, yg_stride, static_cast<cudaStream_t>(stream)),
               "moe_ungroup");
}

ep_status_t ep_reset(ep_handle_t *h, void *stream) {
    EP_RANGE("ep_reset");
    if (!h) return EP_ERR_INVALID_ARGS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const ep_status_t s = gpu(
        h, cudaMemsetAsync(h->ws.words, 0,
                           reinterpret_cast<char *>(h->ws.chunk_local) -
                               reinterpret_cast<char *>(h->ws.words),
                           st),
        "cudaMemsetAsync");
    if (s != EP_SUCCESS) return s;
    h->dispatch_epoch = 0;
    h->combine_epoch = 0;
    h->layout_valid = false;
    h->dispatch_pending = false;
    h->combine_pending = false;
    h->moe_valid = false;
    return EP_SUCCESS;
}

ep_status_t ep_get_error(ep_handle_t *h, uint32_t *mask, void *stream) {
    EP_RANGE("ep_get_error");
    if (!h || !mask) return EP_ERR_INVALID_ARGS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Stream-ordered: one atomic exchange takes the word and clears it, the
    // taken value is copied to the handle's pinned host word, and only this
    // stream is waited for (work on other streams keeps running; a bit it
    // sets later is reported by a later call).
    ep_status_t s = gpu(h, launch_take_error(h->ws, st), "take_error");
    if (s != EP_SUCCESS) return s;
    s = gpu(h, cudaMemcpyAsync(h->h_err, h->ws.words + kWordErrTaken, 4,
                               cudaMemcpyDeviceToHost, st),
            "cudaMemcpyAsync");
    if (s != EP_SUCCESS) return s;
    s = gpu(h, cudaStreamSynchronize(st), "cudaStreamSynchronize");
    if (s != EP_SUCCESS) return s;
    const uint32_t word = *h->h_err;
    *mask = word;
    if (word & EP_DEVERR_BAD_INDEX) return EP_ERR_BAD_INDEX;
    if (word & EP_DEVERR_CAPACITY) return EP_ERR_CAPACITY;
    if (word & EP_DEVERR_TIMEOUT) return EP_ERR_TIMEOUT;
    if (word & EP_DEVERR_COMBINE_MISMATCH) return EP_ERR_BAD_STATE;
    return EP_SUCCESS;
}

ep_status_t ep_test_identity_expert(ep_handle_t *h, void *d_y,
                                    int64_t y_rank_stride_bytes, void *stream) {
    EP_RANGE("ep_test_identity_expert");
    if (!h) return EP_ERR_INVALID_ARGS;
    if (!h->layout_valid) return EP_ERR_BAD_STATE;
    const int64_t row_bytes = (int64_t)h->cfg.cap * h->cfg.H * (h->cfg.y_f32 ? 4 : 2);
    if (d_y && h->cfg.y_fp8) return EP_ERR_INVALID_ARGS;
    char *y;
    int64_t ys;
    if (d_y) {
        ys = y_rank_stride_bytes ? y_rank_stride_bytes : row_bytes;
        if (!aligned(d_y, 16) || ys % 16 != 0 || ys < row_bytes) return EP_ERR_INVALID_ARGS;
        y = static_cast<char *>(d_y);
    } else {
        y = h->ws.seg0 + h->ws.off_comb;
        ys = h->ws.seg_stride;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return gpu(h, launch_identity_expert(h->cfg, h->ws, y, ys, st), "identity_expert");
}

ep_status_t ep_test_fp8_quotient_check(uint64_t *d_counts, void *stream) {
    EP_RANGE("ep_test_fp8_quotient_check");
    if (!d_counts || !aligned(d_counts, 8)) return EP_ERR_INVALID_ARGS;
    return gpu(nullptr,
               launch_fp8_quotient_check(reinterpret_cast<unsigned long long *>(d_counts),
                                         static_cast<cudaStream_t>(stream)),
               "fp8_quotient_check");
}

}  // extern "C"
