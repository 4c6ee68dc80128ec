// Routing layout (the step behind dispatch's recv_count and the receive
// order): per-token destination-rank masks, per-chunk destination counts by
// warp ballot, and -- in the last CTA to finish -- the exclusive prefix over
// chunks in (source rank, chunk) order that fixes every receive position.
//
// Definition (ROCm MORI "Communication APIs", MORI-EP, "EpDispatchCombineOp
// methods": dispatch routes each token to its expert ranks and returns
// recv_count): D(s,t) = { idx[s][t][j] / Er }, C[s][r] = #{t < n_s : r in
// D(s,t)}, recv_count[r] = sum_s C[s][r]; rows on rank r are ordered by
// (source rank, source token).  The chunk bases computed here plus the
// within-chunk ballot prefix (recomputed by the dispatch kernel) give
// pos[s][t][r] = sum_{s'<s} C[s'][r] + #{t' < t : r in D(s,t')}.
#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kLayoutThreads = 256;            // 8 warps = 8 chunks per CTA
constexpr int kLayoutWarps = kLayoutThreads / 32;

struct LayoutParams {
    const int32_t *idx;
    uint32_t *masks;
    int32_t *chunk_cnt;
    int32_t *chunk_base;
    int32_t *send_counts;
    int32_t *recv_count;
    uint32_t *words;
    int W, E, Er, k, T, nch, G, cap;
    int publish;             // also write recv_count (one-stream dispatch)
    TokenCounts nt;
};

__global__ void __launch_bounds__(kLayoutThreads)
layout_kernel(const LayoutParams p) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = blockIdx.x * kLayoutWarps + warp;

    if (g < p.G) {
        const int s = g / p.nch;
        const int t = (g - s * p.nch) * kChunk + lane;
        const bool present = t < p.nt.n[s];
        uint32_t mask = 0;
        bool bad = false;
        if (present) {
            const int32_t *row = p.idx + ((int64_t)s * p.T + t) * p.k;
            for (int j = 0; j < p.k; ++j) {
                const int32_t e = __ldg(row + j);
                if ((uint32_t)e < (uint32_t)p.E)
                    mask |= 1u << (e / p.Er);
                else
                    bad = true;
            }
        }
        if (bad) set_error(p.words, EP_DEVERR_BAD_INDEX);
        if (t < p.T) p.masks[(int64_t)s * p.T + t] = mask;
        int my_count = 0;
        for (int r = 0; r < p.W; ++r) {
            const uint32_t b = __ballot_sync(0xffffffffu, (mask >> r) & 1u);
            if (lane == r) my_count = __popc(b);
        }
        if (lane < p.W) p.chunk_cnt[(int64_t)g * p.W + lane] = my_count;
    }

    // Last CTA to arrive turns the chunk counts into chunk bases.
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = atom_add_acq_rel_gpu(p.words + kWordLayoutDone, 1u) ==
                 gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // Warp `warp` scans destinations r = warp, warp + 8, ...  Each lane owns
    // a contiguous run of chunks; a warp shuffle scan joins the runs.
    const int per = (p.G + 31) / 32;
    const int g0 = min(p.G, lane * per);
    const int g1 = min(p.G, g0 + per);
    for (int r = warp; r < p.W; r += kLayoutWarps) {
        int sum = 0;
        for (int gg = g0; gg < g1; ++gg)
            sum += __ldcg(p.chunk_cnt + (int64_t)gg * p.W + r);
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int gg = g0; gg < g1; ++gg) {
            p.chunk_base[(int64_t)gg * p.W + r] = run;
            run += __ldcg(p.chunk_cnt + (int64_t)gg * p.W + r);
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (lane == 0) {
            p.chunk_base[(int64_t)p.G * p.W + r] = total;
            if (total > p.cap) set_error(p.words, EP_DEVERR_CAPACITY);
            if (p.publish) p.recv_count[r] = total;
        }
        __syncwarp();
        // C[s][r] = base of the first chunk of s+1 minus that of s.
        for (int s = lane; s < p.W; s += 32) {
            const int b0 = __ldcg(p.chunk_base + (int64_t)s * p.nch * p.W + r);
            const int b1 = __ldcg(p.chunk_base + (int64_t)(s + 1) * p.nch * p.W + r);
            p.send_counts[s * p.W + r] = b1 - b0;
        }
    }
    if (threadIdx.x == 0) p.words[kWordLayoutDone] = 0;   // for the next call
}

}  // namespace

cudaError_t launch_layout(const Config &c, const Workspace &ws,
                          const int32_t *idx, const TokenCounts &nt,
                          cudaStream_t st, bool publish) {
    LayoutParams p;
    p.idx = idx;
    p.masks = ws.masks;
    p.chunk_cnt = ws.chunk_cnt;
    p.chunk_base = ws.chunk_base;
    p.send_counts = ws.send_counts;
    p.recv_count = ws.recv_count;
    p.words = ws.words;
    p.W = c.W; p.E = c.E; p.Er = c.Er; p.k = c.k; p.T = c.T;
    p.nch = c.nch; p.G = c.G; p.cap = c.cap;
    p.publish = publish ? 1 : 0;
    p.nt = nt;
    const int blocks = (c.G + kLayoutWarps - 1) / kLayoutWarps;
    layout_kernel<<<blocks, kLayoutThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
