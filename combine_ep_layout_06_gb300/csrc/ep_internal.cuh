// Internal definitions shared by the CUDA translation units of the library:
// the handle, the workspace map and the kernel launch wrappers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ep_api.h"

// NVTX ranges around every entry point, for timelines and for `ncu --nvtx`
// range filters: compiled in with -DEP_NVTX=1 (the build's EP_NVTX=1
// environment switch), absent otherwise, so the timed build carries none.
#ifndef EP_NVTX
#define EP_NVTX 0
#endif
#if EP_NVTX
#include <nvtx3/nvToolsExt.h>
namespace ep {
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
}  // namespace ep
#define EP_RANGE(name) ::ep::NvtxRange ep_nvtx_range_(name)
#else
#define EP_RANGE(name) ((void)0)
#endif

namespace ep {

// Tokens per layout chunk: one warp ballots over 32 tokens, so a chunk's
// per-destination counts come from one __ballot_sync + __popc each.
constexpr int kChunk = 32;
// Chunks per layout group (one layout CTA of 8 warps): the group prefix is
// computed inside the CTA, so the one global scan runs over groups only.
constexpr int kGroup = 8;

// Offsets of the small counters at the start of the workspace (u32 words).
constexpr int kWordErr = 0;        // sticky device error word
constexpr int kWordLayoutDone = 1; // "last CTA" ticket of the layout kernel
constexpr int kWordSrcDone = 8;    // [W] per-source ticket of the dispatch copy
constexpr int kWordMoeDone = 40;   // "last CTA" ticket of the grouping scan
constexpr int kWordErrTaken = 41;  // the error word as ep_get_error last took it
constexpr int kCounterWords = 64;  // 256 bytes

struct Workspace {
    // layout state
    uint32_t *words;       // kCounterWords u32
    uint32_t *dflags;      // [W dst][W src]
    uint32_t *cflags;      // [W src][W dst]
    int32_t *chunk_local;  // [G][W]   exclusive prefix of a chunk within its group
    int32_t *group_tot;    // [Q][W]   destination counts of each group
    int32_t *group_base;   // [Q+1][W] exclusive prefix over groups; row Q = totals
    int32_t *send_counts;  // [W][W]
    int32_t *recv_count;   // [W] published by the receive step
    uint32_t *masks;       // [W][T]   destination-rank bit mask per token
    int32_t *pos;          // [W][T][W]
    // standard-MoE grouping (when gcap > 0)
    int32_t *moe_cnt;      // [W][nrc][Er] entries per (rank, 32-row chunk, expert)
    int32_t *moe_base;     // [W][nrc][Er] exclusive prefix over chunks
    int32_t *moe_count;    // [W][Er]
    int32_t *moe_offset;   // [W][Er]
    char *stage;           // scatter combine: [W][T][maxd][H] bf16 staged rows
    // rank-0 segment; rank r's copy is at + r * seg_stride bytes
    char *seg0;
    int64_t seg_stride;
    int64_t off_out, off_scales, off_w, off_idx, off_src, off_comb, off_comb_sc;
    int64_t off_xg, off_xgs, off_gsrc, off_gw, off_yg, off_eslot;   // grouping
    size_t total_bytes;
};

struct Config {
    int W, E, Er, k, H, T, cap;
    bool fp8;
    bool y_f32;  // combine reads fp32 expert rows
    bool y_fp8;  // combine reads E4M3 expert rows + block scales (else bf16)
    int nch;     // chunks per source rank = ceil(T / kChunk)
    int G;       // W * nch
    int Q;       // layout groups = ceil(G / kGroup)
    int gcap;    // grouped rows per rank (0: no standard-MoE grouping)
    bool scatter;  // scatter combine (staging on the source side)
    int maxd;    // min(W, k): destinations per token at most
    int nrc;     // 32-row chunks of received rows per rank = ceil(cap / 32)
    int nvec;    // 16-byte vectors per bf16 row = H / 8
    int nb;      // FP8 blocks per row = H / 128 (0 for bf16)
    bool early_notify, fused_recv;
    int64_t timeout_ns;
};

// Plan the workspace of a config; base may be null (sizing only).
void plan_workspace(const Config &c, char *base, Workspace *ws);

// Per-call token counts, passed by value to kernels.
struct TokenCounts {
    int32_t n[EP_MAX_WORLD];
};

// ---------------------------------------------------------------- kernels
// Each launcher enqueues on `st` and returns cudaGetLastError().

// publish: also write recv_count (when no separate receive step follows).
cudaError_t launch_layout(const Config &c, const Workspace &ws,
                          const int32_t *idx, const TokenCounts &nt,
                          cudaStream_t st, bool publish);

struct DispatchArgs {
    const void *x;         // [W][T][H] bf16, or E4M3 codes with scales_in
    const float *scales_in;  // [W][T][H/128] pre-quantised block scales, or null
    const float *w;        // [W][T][k]
    const int32_t *idx;    // [W][T][k]
    TokenCounts nt;
    uint32_t epoch;        // flag value when early_notify
    bool after_layout;     // launched right after the layout kernel on the same stream
    bool self_layout;      // no layout kernel: the copy computes the layout (few chunks)
    bool publish;          // with self_layout: also write recv_count
};

// Chunks (W * ceil(T/32)) up to which the copy computes the layout itself.
int self_layout_chunks();
cudaError_t launch_dispatch(const Config &c, const Workspace &ws,
                            const DispatchArgs &a, cudaStream_t st);

// Receive step: optional bounded flag check, then publish recv_count.
cudaError_t launch_dispatch_recv(const Config &c, const Workspace &ws,
                                 bool check_flags, uint32_t epoch,
                                 cudaStream_t st);

cudaError_t launch_combine_notify(const Config &c, const Workspace &ws,
                                  uint32_t epoch, cudaStream_t st);
cudaError_t launch_combine_wait(const Config &c, const Workspace &ws,
                                uint32_t epoch, cudaStream_t st);

struct CombineArgs {
    const char *y;          // rank 0 rows; rank r at + r*y_stride
    const char *ysc;        // FP8 payload: rank 0 block scales, same stride
    const char *stage;      // scatter combine: staged rows instead of y
    int64_t y_stride;
    const char *w_in;       // nullable
    int64_t w_stride;
    const int32_t *idx;     // nullable
    uint16_t *out;          // [W][T][H]
    float *out_w;           // nullable
    TokenCounts nt;
    bool fused_wait;        // fused receive: each CTA waits on the flags
    uint32_t epoch;
};
cudaError_t launch_combine(const Config &c, const Workspace &ws,
                           const CombineArgs &a, cudaStream_t st);

// Scatter combine, send side: every received row's expert output to its
// token's staging slot.
cudaError_t launch_scatter_send(const Config &c, const Workspace &ws, cudaStream_t st);

cudaError_t launch_moe_group(const Config &c, const Workspace &ws, cudaStream_t st);
cudaError_t launch_moe_ungroup(const Config &c, const Workspace &ws, const char *yg,
                               int64_t yg_stride, cudaStream_t st);

cudaError_t launch_identity_expert(const Config &c, const Workspace &ws,
                                   char *y, int64_t y_stride, cudaStream_t st);

// Read and clear the error word in one atomic exchange (kWordErrTaken gets
// the old value), so that a bit set meanwhile by work on another stream is
// either taken now or left for the next call, never lost.
cudaError_t launch_take_error(const Workspace &ws, cudaStream_t st);

// Test harness: the FP8 quotient and scale identities over every bf16 pair.
cudaError_t launch_fp8_quotient_check(unsigned long long *d_counts, cudaStream_t st);

}  // namespace ep

// Host handle.
struct ep_handle {
    ep::Config cfg;
    ep::Workspace ws;
    int device;
    cudaEvent_t ev_dispatch_sent;
    cudaEvent_t ev_combine_sent;
    uint32_t dispatch_epoch;
    uint32_t combine_epoch;
    bool layout_valid;      // a layout exists for combine / replay
    bool dispatch_pending;  // sent, not yet received
    bool combine_pending;   // combine sent, not yet received
    bool moe_valid;         // a standard-MoE grouping exists for ungroup
    ep::TokenCounts layout_nt;
    int log_level;
    uint32_t *h_err;        // pinned host word for ep_get_error
};
