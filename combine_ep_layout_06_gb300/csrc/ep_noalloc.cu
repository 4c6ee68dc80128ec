// Routing layout for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// that runs inside another framework's memory pool without access to its
// allocator (a plugin or custom op that only receives raw tensor pointers),
// and serving loops that forbid allocation on the request path because
// cudaMalloc can synchronise the device and can fail under memory pressure.
// ep_layout_noalloc gives them the routing layout with no allocation at
// all: its scratch (per-chunk offsets inside groups of 8 chunks, group
// totals and bases, a CTA ticket) lives in the file-scope device array
// below, which every GPU that loads this library holds until the process
// exits.
//
// Sharing rules: every call on a device uses the same array and leaves its
// contents behind.  The ticket that must start at zero is cleared at the
// start of each call.  Calls whose kernels overlap on the GPU (two streams,
// no ordering between them) race on the array and give wrong results;
// order them on one stream or with events.
#include <cstring>

#include "ep_device.cuh"

namespace ep {
namespace {

// Largest layout this entry point accepts: W <= 32 ranks and at most
// kNoAllocMaxChunks = 4128 32-token chunks in total (W * ceil(T/32)).  Any
// W * T <= 131072 fits whatever T is (ceil adds at most one chunk per rank,
// 32 in all); with T a multiple of 32 up to 132096 tokens fit.  Scratch:
// 256 B of counters, then per-chunk offsets inside their group of 8 chunks
// [kNoAllocMaxChunks][32], group totals [kNoAllocMaxGroups][32] and group
// bases [kNoAllocMaxGroups+1][32], int32 -- about 0.66 MB.
constexpr int kNoAllocMaxChunks = 4096 + EP_MAX_WORLD;
constexpr int kNoAllocGroup = 8;                       // chunks per CTA
constexpr int kNoAllocMaxGroups = (kNoAllocMaxChunks + kNoAllocGroup - 1) / kNoAllocGroup;
constexpr size_t kNoAllocCounterBytes = 256;
constexpr size_t kNoAllocLocalInts = (size_t)kNoAllocMaxChunks * EP_MAX_WORLD;
constexpr size_t kNoAllocTotInts = (size_t)kNoAllocMaxGroups * EP_MAX_WORLD;
constexpr size_t kNoAllocBaseInts = (size_t)(kNoAllocMaxGroups + 1) * EP_MAX_WORLD;
constexpr size_t kNoAllocScratchBytes =
    kNoAllocCounterBytes + 4 * (kNoAllocLocalInts + kNoAllocTotInts + kNoAllocBaseInts);

static __device__ __align__(256) unsigned char g_layout_scratch[kNoAllocScratchBytes];

constexpr int kWarps = kNoAllocGroup;
constexpr int kThreads = kWarps * 32;
constexpr int kBatch = 8;                             // group totals in registers per lane

struct NoAllocParams {
    const int32_t *idx;
    int32_t *pos;
    int32_t *send_counts;
    int32_t *recv_count;
    uint32_t *error;          // nullable
    uint32_t *ticket;         // in the scratch array
    int32_t *local;           // [G][W]   offset of a chunk inside its group
    int32_t *gtot;            // [Q][W]   group totals
    int32_t *gbase;           // [Q+1][W] exclusive prefix over groups; row Q = totals
    int W, E, Er, k, T, nch, G, Q;
    TokenCounts nt;
};

// Destination mask of token t of source s (0 past n_s); all k ids are
// loaded before the first is used.
__device__ __forceinline__ uint32_t chunk_mask(const NoAllocParams &p, int s,
                                               int t, bool *bad) {
    uint32_t mask = 0;
    if (t < p.nt.n[s]) {
        const int32_t *row = p.idx + ((int64_t)s * p.T + t) * p.k;
        int32_t e[EP_MAX_TOPK];
#pragma unroll
        for (int j = 0; j < EP_MAX_TOPK; ++j)
            if (j < p.k) e[j] = __ldg(row + j);
#pragma unroll
        for (int j = 0; j < EP_MAX_TOPK; ++j) {
            if (j < p.k) {
                if ((uint32_t)e[j] < (uint32_t)p.E)
                    mask |= 1u << (e[j] / p.Er);
                else
                    *bad = true;
            }
        }
    }
    return mask;
}

// Start of chunk g in its destinations' receive order once the group bases
// are final (g == G gives the totals).
__device__ __forceinline__ int chunk_start(const NoAllocParams &p, int g, int r) {
    if (g >= p.G) return __ldcg(p.gbase + (int64_t)p.Q * p.W + r);
    return __ldcg(p.gbase + (int64_t)(g / kNoAllocGroup) * p.W + r) +
           __ldcg(p.local + (int64_t)g * p.W + r);
}

// Pass 1: a CTA per group of 8 chunks counts each chunk's destinations
// (warp ballot) and prefixes them inside the group; the last CTA to finish
// scans the group totals (order: source rank, then chunk) into group bases
// and writes send_counts / recv_count.
__global__ void __launch_bounds__(kThreads) noalloc_count_kernel(const NoAllocParams p) {
    __shared__ int s_cnt[kWarps][EP_MAX_WORLD];
    __shared__ int s_last;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int q = blockIdx.x;
    const int g = q * kNoAllocGroup + warp;
    int my_count = 0;
    if (g < p.G) {
        const int s = g / p.nch;
        const int t = (g - s * p.nch) * kChunk + lane;
        bool bad = false;
        const uint32_t mask = chunk_mask(p, s, t, &bad);
        if (bad && p.error) atomicOr(p.error, EP_DEVERR_BAD_INDEX);
        for (int r = 0; r < p.W; ++r) {
            const uint32_t b = __ballot_sync(0xffffffffu, (mask >> r) & 1u);
            if (lane == r) my_count = __popc(b);
        }
    }
    s_cnt[warp][lane] = my_count;
    __syncthreads();
    if (warp == 0 && lane < p.W) {
        int run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int gg = q * kNoAllocGroup + w;
            if (gg < p.G) p.local[(int64_t)gg * p.W + lane] = run;
            run += s_cnt[w][lane];
        }
        p.gtot[(int64_t)q * p.W + lane] = run;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = atom_add_acq_rel_gpu(p.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // warp w scans destinations r = w, w + 8, ...; lane l owns a contiguous
    // run of groups, read kBatch at a time into registers
    const int per = (p.Q + 31) / 32;
    const int q0 = min(p.Q, lane * per);
    const int q1 = min(p.Q, q0 + per);
    for (int r = warp; r < p.W; r += kWarps) {
        int sum = 0;
        for (int b0 = q0; b0 < q1; b0 += kBatch) {
            int v[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                v[i] = (b0 + i < q1) ? __ldcg(p.gtot + (int64_t)(b0 + i) * p.W + r) : 0;
#pragma unroll
            for (int i = 0; i < kBatch; ++i) sum += v[i];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        int run = incl - sum;
        for (int b0 = q0; b0 < q1; b0 += kBatch) {
            int v[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                v[i] = (b0 + i < q1) ? __ldcg(p.gtot + (int64_t)(b0 + i) * p.W + r) : 0;
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (b0 + i < q1) p.gbase[(int64_t)(b0 + i) * p.W + r] = run;
                run += v[i];
            }
        }
        if (lane == 31) {
            p.gbase[(int64_t)p.Q * p.W + r] = incl;
            p.recv_count[r] = incl;
        }
    }
    __syncthreads();
    // C[s][r] = start of the first chunk of s+1 minus that of s
    for (int i = threadIdx.x; i < p.W * p.W; i += kThreads) {
        const int s = i / p.W, r = i - s * p.W;
        p.send_counts[i] = chunk_start(p, (s + 1) * p.nch, r) - chunk_start(p, s * p.nch, r);
    }
    if (threadIdx.x == 0) *p.ticket = 0u;
}

// Pass 2: pos[s][t][r] = the chunk's start + the number of earlier tokens of
// the chunk routed to r, or -1.
__global__ void __launch_bounds__(kThreads) noalloc_pos_kernel(const NoAllocParams p) {
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (g >= p.G) return;
    const int s = g / p.nch;
    const int t = (g - s * p.nch) * kChunk + lane;
    bool bad = false;
    const uint32_t mask = chunk_mask(p, s, t, &bad);
    const int my_base = (lane < p.W) ? chunk_start(p, g, lane) : 0;
    const uint32_t below = lanemask_lt();
    int32_t *dst = p.pos + ((int64_t)s * p.T + t) * p.W;
    for (int r = 0; r < p.W; ++r) {
        const uint32_t b = __ballot_sync(0xffffffffu, (mask >> r) & 1u);
        const int bs = __shfl_sync(0xffffffffu, my_base, r);
        if (t < p.T) dst[r] = ((mask >> r) & 1u) ? bs + __popc(b & below) : -1;
    }
}

}  // namespace
}  // namespace ep

extern "C" ep_status_t ep_layout_noalloc(
    int32_t world_size, int32_t num_experts, int32_t topk,
    int32_t max_tokens_per_rank, const int32_t *d_idx,
    const int32_t *h_num_tokens, int32_t *d_pos, int32_t *d_send_counts,
    int32_t *d_recv_count, uint32_t *d_error, void *stream) {
    using namespace ep;
    EP_RANGE("ep_layout_noalloc");
    const int W = world_size, E = num_experts, k = topk, T = max_tokens_per_rank;
    if (W < 1 || W > EP_MAX_WORLD || E < W || E % W != 0 || k < 1 ||
        k > EP_MAX_TOPK || T < 1)
        return EP_ERR_INVALID_ARGS;
    const int64_t nch = (T + kChunk - 1) / kChunk;
    if ((int64_t)W * nch > kNoAllocMaxChunks) return EP_ERR_INVALID_ARGS;
    if (!d_idx || !h_num_tokens || !d_pos || !d_send_counts || !d_recv_count)
        return EP_ERR_INVALID_ARGS;
    NoAllocParams p;
    std::memset(&p.nt, 0, sizeof(p.nt));
    for (int s = 0; s < W; ++s) {
        if (h_num_tokens[s] < 0 || h_num_tokens[s] > T) return EP_ERR_INVALID_ARGS;
        p.nt.n[s] = h_num_tokens[s];
    }
    // The array's name is only a host-side handle; its device address comes
    // from the runtime, looked up on every call with the caller's device
    // current (a host-side lookup once the module is loaded; never cached, so
    // a context torn down and recreated, as by cudaDeviceReset, is followed).
    // The first call on a device may load the module: make it before any
    // stream capture.
    void *scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_layout_scratch) != cudaSuccess || !scratch)
        return EP_ERR_GPU_OP;
    char *base = static_cast<char *>(scratch);
    p.idx = d_idx;
    p.pos = d_pos;
    p.send_counts = d_send_counts;
    p.recv_count = d_recv_count;
    p.error = d_error;
    p.ticket = reinterpret_cast<uint32_t *>(base);
    p.local = reinterpret_cast<int32_t *>(base + kNoAllocCounterBytes);
    p.gtot = p.local + kNoAllocLocalInts;
    p.gbase = p.gtot + kNoAllocTotInts;
    p.W = W; p.E = E; p.Er = E / W; p.k = k; p.T = T;
    p.nch = (int)nch;
    p.G = (int)(W * nch);
    p.Q = (p.G + kNoAllocGroup - 1) / kNoAllocGroup;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(p.ticket, 0, sizeof(uint32_t), st) != cudaSuccess)
        return EP_ERR_GPU_OP;
    noalloc_count_kernel<<<p.Q, kThreads, 0, st>>>(p);
    noalloc_pos_kernel<<<p.Q, kThreads, 0, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? EP_SUCCESS : EP_ERR_GPU_OP;
}
