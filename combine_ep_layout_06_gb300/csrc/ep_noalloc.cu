// Routing layout for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// that runs inside another framework's memory pool without access to its
// allocator (a plugin or custom op that only receives raw tensor pointers),
// and serving loops that forbid allocation on the request path because
// cudaMalloc can synchronise the device and can fail under memory pressure.
// ep_layout_noalloc gives them the routing layout with no allocation at
// all: its scratch (per-chunk destination counts, chunk bases and a CTA
// ticket) lives in the file-scope device array below, which every GPU that
// loads this library holds until the process exits.
//
// Sharing rules: every call on a device uses the same array and leaves its
// contents behind.  The ticket that must start at zero is cleared at the
// start of each call.  Calls whose kernels overlap on the GPU (two streams,
// no ordering between them) race on the array and give wrong results;
// order them on one stream or with events.
#include <cstring>
#include <mutex>

#include "ep_device.cuh"

namespace ep {
namespace {

// Largest layout this entry point accepts: W <= 32 ranks and at most
// kNoAllocMaxChunks 32-token chunks in total (W * ceil(T/32)), e.g.
// 131072 tokens when T is a multiple of 32.  Scratch: 256 B of counters,
// then counts [kNoAllocMaxChunks][32] and bases [kNoAllocMaxChunks+1][32]
// int32 -- about 1.06 MB.
constexpr int kNoAllocMaxChunks = 4096 + EP_MAX_WORLD;
constexpr size_t kNoAllocCounterBytes = 256;
constexpr size_t kNoAllocCountInts = (size_t)kNoAllocMaxChunks * EP_MAX_WORLD;
constexpr size_t kNoAllocBaseInts = (size_t)(kNoAllocMaxChunks + 1) * EP_MAX_WORLD;
constexpr size_t kNoAllocScratchBytes =
    kNoAllocCounterBytes + 4 * (kNoAllocCountInts + kNoAllocBaseInts);

static __device__ __align__(256) unsigned char g_layout_scratch[kNoAllocScratchBytes];

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct NoAllocParams {
    const int32_t *idx;
    int32_t *pos;
    int32_t *send_counts;
    int32_t *recv_count;
    uint32_t *error;          // nullable
    uint32_t *ticket;         // in the scratch array
    int32_t *cnt;             // [G][W]
    int32_t *base;            // [G+1][W]
    int W, E, Er, k, T, nch, G;
    TokenCounts nt;
};

__device__ __forceinline__ uint32_t chunk_mask(const NoAllocParams &p, int s,
                                               int t, bool *bad) {
    uint32_t mask = 0;
    if (t < p.nt.n[s]) {
        const int32_t *row = p.idx + ((int64_t)s * p.T + t) * p.k;
        for (int j = 0; j < p.k; ++j) {
            const int32_t e = __ldg(row + j);
            if ((uint32_t)e < (uint32_t)p.E)
                mask |= 1u << (e / p.Er);
            else
                *bad = true;
        }
    }
    return mask;
}

// Pass 1: per-chunk destination counts; the last CTA scans them into chunk
// bases (order: source rank, then chunk) and writes send_counts/recv_count.
__global__ void __launch_bounds__(kThreads) noalloc_count_kernel(const NoAllocParams p) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = blockIdx.x * kWarps + warp;
    if (g < p.G) {
        const int s = g / p.nch;
        const int t = (g - s * p.nch) * kChunk + lane;
        bool bad = false;
        const uint32_t mask = chunk_mask(p, s, t, &bad);
        if (bad && p.error) atomicOr(p.error, EP_DEVERR_BAD_INDEX);
        int my_count = 0;
        for (int r = 0; r < p.W; ++r) {
            const uint32_t b = __ballot_sync(0xffffffffu, (mask >> r) & 1u);
            if (lane == r) my_count = __popc(b);
        }
        if (lane < p.W) p.cnt[(int64_t)g * p.W + lane] = my_count;
    }
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = atom_add_acq_rel_gpu(p.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int per = (p.G + 31) / 32;
    const int g0 = min(p.G, lane * per);
    const int g1 = min(p.G, g0 + per);
    for (int r = warp; r < p.W; r += kWarps) {
        int sum = 0;
        for (int gg = g0; gg < g1; ++gg) sum += __ldcg(p.cnt + (int64_t)gg * p.W + r);
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int gg = g0; gg < g1; ++gg) {
            p.base[(int64_t)gg * p.W + r] = run;
            run += __ldcg(p.cnt + (int64_t)gg * p.W + r);
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (lane == 0) {
            p.base[(int64_t)p.G * p.W + r] = total;
            p.recv_count[r] = total;
        }
        __syncwarp();
        for (int s = lane; s < p.W; s += 32)
            p.send_counts[s * p.W + r] =
                __ldcg(p.base + (int64_t)(s + 1) * p.nch * p.W + r) -
                __ldcg(p.base + (int64_t)s * p.nch * p.W + r);
    }
    if (threadIdx.x == 0) *p.ticket = 0u;
}

// Pass 2: pos[s][t][r] = chunk base + number of earlier tokens of the chunk
// routed to r, or -1.
__global__ void __launch_bounds__(kThreads) noalloc_pos_kernel(const NoAllocParams p) {
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (g >= p.G) return;
    const int s = g / p.nch;
    const int t = (g - s * p.nch) * kChunk + lane;
    bool bad = false;
    const uint32_t mask = chunk_mask(p, s, t, &bad);
    const int my_base = (lane < p.W) ? p.base[(int64_t)g * p.W + lane] : 0;
    const uint32_t below = lanemask_lt();
    int32_t *dst = p.pos + ((int64_t)s * p.T + t) * p.W;
    for (int r = 0; r < p.W; ++r) {
        const uint32_t b = __ballot_sync(0xffffffffu, (mask >> r) & 1u);
        const int bs = __shfl_sync(0xffffffffu, my_base, r);
        if (t < p.T) dst[r] = ((mask >> r) & 1u) ? bs + __popc(b & below) : -1;
    }
}

std::mutex g_setup_mutex;
void *g_scratch_ptr[256] = {};

}  // namespace
}  // namespace ep

extern "C" ep_status_t ep_layout_noalloc(
    int32_t world_size, int32_t num_experts, int32_t topk,
    int32_t max_tokens_per_rank, const int32_t *d_idx,
    const int32_t *h_num_tokens, int32_t *d_pos, int32_t *d_send_counts,
    int32_t *d_recv_count, uint32_t *d_error, void *stream) {
    using namespace ep;
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
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256)
        return EP_ERR_GPU_OP;
    void *scratch = nullptr;
    {
        // Set-up, once per device, with that device current: the array's
        // name is only a host-side handle; its device address comes from the
        // runtime.  This may load the module, so make the first call on a
        // device before any stream capture.
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (!g_scratch_ptr[dev]) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_layout_scratch) != cudaSuccess || !ptr)
                return EP_ERR_GPU_OP;
            g_scratch_ptr[dev] = ptr;
        }
        scratch = g_scratch_ptr[dev];
    }
    char *base = static_cast<char *>(scratch);
    p.idx = d_idx;
    p.pos = d_pos;
    p.send_counts = d_send_counts;
    p.recv_count = d_recv_count;
    p.error = d_error;
    p.ticket = reinterpret_cast<uint32_t *>(base);
    p.cnt = reinterpret_cast<int32_t *>(base + kNoAllocCounterBytes);
    p.base = p.cnt + kNoAllocCountInts;
    p.W = W; p.E = E; p.Er = E / W; p.k = k; p.T = T;
    p.nch = (int)nch;
    p.G = (int)(W * nch);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(p.ticket, 0, sizeof(uint32_t), st) != cudaSuccess)
        return EP_ERR_GPU_OP;
    const int blocks = (p.G + kWarps - 1) / kWarps;
    noalloc_count_kernel<<<blocks, kThreads, 0, st>>>(p);
    noalloc_pos_kernel<<<blocks, kThreads, 0, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? EP_SUCCESS : EP_ERR_GPU_OP;
}
