// Dispatch copy: every present token row goes, once per distinct destination
// rank, to its receive slot in that rank's segment, with its k weights, k
// expert ids and its source position; optionally the row is quantised to
// OCP FP8 E4M3 with one fp32 scale per 128 elements on the way.
//
// Definition (ROCm MORI "Communication APIs", MORI-EP, "EpDispatchCombineOp
// methods": dispatch(input, weights, scales, indices) -> (output, weights,
// scales, indices, recv_count); get_dispatch_src_token_pos()).  FP8 is OCP
// E4M3 ("EPv2 configuration and lifecycle"); per block a = max|x|,
// scale = fl32(a/448), q = RNE-satfinite(fl32(x/scale)), a == 0 -> scale 0,
// codes 0.
//
// GB300 mapping.  A CTA takes a few tokens (TPC) of one 32-token layout
// chunk.  Warp 0 turns the chunk's masks and base into receive slots
// (ballot + popc of the lanes below) and writes pos.  Then either
//  - the register path: each warp streams whole token rows, reading the
//    source row ONCE from HBM (16-byte non-allocating loads, U vectors in
//    flight per lane) and storing it to each destination row with 16-byte
//    evict-first stores, 512 contiguous bytes per warp instruction (the FP8
//    path quantises on the way: 16 elements per lane, 8 lanes per block);
//  - the bulk path (bf16): one thread drives the Tensor Memory Accelerator
//    with 1-D cp.async.bulk row copies through a ring of shared-memory
//    stages, one load per source row and one bulk store per destination.
#include <cuda_fp8.h>

#include <atomic>
#include <mutex>

#include "ep_device.cuh"

namespace ep {
namespace {

#ifndef EP_DISPATCH_WARPS
#define EP_DISPATCH_WARPS 4
#endif
#ifndef EP_DISPATCH_UNROLL
#define EP_DISPATCH_UNROLL 4           // 16-byte vectors in flight per lane
#endif
#ifndef EP_DISPATCH_FP8_UNROLL
#define EP_DISPATCH_FP8_UNROLL 1       // 32-byte element pairs per lane (FP8)
#endif
#ifndef EP_DISPATCH_BULK_STAGES
#define EP_DISPATCH_BULK_STAGES 4      // 0: register path for bf16 rows too
#endif
#ifndef EP_DISPATCH_BULK_CTAS_PER_SM
#define EP_DISPATCH_BULK_CTAS_PER_SM 2 // resident bulk CTAs per SM (0: no cap)
#endif
#ifndef EP_DISPATCH_BULK_CAP_MIN_WAVES
#define EP_DISPATCH_BULK_CAP_MIN_WAVES 4 // cap residency only for grids of >= this many capped waves
#endif
#ifndef EP_DISPATCH_TPC
#define EP_DISPATCH_TPC 2              // tokens per CTA, bulk path (divides 32)
#endif
#ifndef EP_DISPATCH_FP8_PREFETCH
#define EP_DISPATCH_FP8_PREFETCH 1     // FP8: load the next element pair while quantising
#endif
#ifndef EP_FP8_RECIP_QUOT
#define EP_FP8_RECIP_QUOT 1            // FP8: quotients by reciprocal + one FMA correction
#endif
#ifndef EP_DISPATCH_PDL
#define EP_DISPATCH_PDL 1              // launch the copy programmatically after the layout
#endif
#ifndef EP_DISPATCH_SELF_LAYOUT_CHUNKS
#define EP_DISPATCH_SELF_LAYOUT_CHUNKS 8   // up to this many chunks the copy computes the layout
#endif
#ifndef EP_DISPATCH_REG_TPC
#define EP_DISPATCH_REG_TPC 4          // tokens per CTA, register / FP8 path
#endif

constexpr int kDispatchWarps = EP_DISPATCH_WARPS;
constexpr int kDispatchThreads = kDispatchWarps * 32;
constexpr int kMaxFp8Blocks = 128;   // H <= 16384 for FP8
static_assert(kChunk % EP_DISPATCH_TPC == 0 && kChunk % EP_DISPATCH_REG_TPC == 0,
              "tokens per CTA must divide the chunk");

struct DispatchParams {
    const uint4 *x;
    const float *scales_in;   // pre-quantised block scales [W][T][nb], or null
    const float *w;
    const int32_t *idx;
    const uint32_t *masks;
    const int32_t *chunk_local;
    const int32_t *group_base;
    int32_t *pos;
    char *seg0;
    int64_t seg_stride, off_out, off_scales, off_w, off_idx, off_src;
    uint32_t *words;
    uint32_t *dflags;
    int W, k, T, H, nch, cap, nvec, nb;
    int row_bytes;            // payload bytes per row on both sides (bulk path)
    int notify;
    uint32_t epoch;
    int64_t timeout_ns;
    TokenCounts nt;
    // the whole layout computed by every CTA (G <= kSelfChunks); CTA 0 also
    // writes the layout state that replay, the receive step and combine read
    int self_layout;
    int E, Er, G, publish;
    uint32_t *masks_w;
    int32_t *chunk_local_w, *group_tot_w, *group_base_w, *send_counts, *recv_count;
};

struct DispatchSmem {
    int32_t pos[kChunk][EP_MAX_WORLD];
    uint32_t mask[kChunk];
    float scales[kDispatchWarps][kMaxFp8Blocks];
};

struct BulkSmem {
    int32_t pos[kChunk][EP_MAX_WORLD];
    uint32_t mask[kChunk];
    int32_t list[kChunk];
};

// Receive slots of a chunk's tokens (the within-chunk part of the layout),
// one warp: lane l holds token t0 + l with destination mask m and, in lanes
// r < W, the chunk's start my_base on rank r.  A token's slot on rank r is
// the chunk's start plus the number of lanes below it that also go to r.
// Fills spos / smask for all 32 tokens and writes pos for the CTA's own
// tokens [i0, i0 + TPC).
template <int TPC>
__device__ __forceinline__ void slots_from(const DispatchParams &p, int s, int t0, int i0,
                                           uint32_t m, int my_base,
                                           int32_t (*spos)[EP_MAX_WORLD], uint32_t *smask) {
    const int lane = threadIdx.x & 31;
    const int t = t0 + lane;
    const uint32_t below = lanemask_lt();
    for (int r = 0; r < p.W; ++r) {
        const uint32_t b = __ballot_sync(0xffffffffu, (m >> r) & 1u);
        const int base = __shfl_sync(0xffffffffu, my_base, r);
        spos[lane][r] = ((m >> r) & 1u) ? base + __popc(b & below) : -1;
    }
    smask[lane] = m;
    if (t < p.T && lane >= i0 && lane < i0 + TPC) {
        int32_t *dst = p.pos + ((int64_t)s * p.T + t) * p.W;
        for (int r = 0; r < p.W; ++r) dst[r] = spos[lane][r];
    }
}

// The same from the layout kernel's results (warp 0): the masks, and the
// chunk's start = its group's base + its offset inside the group.
template <int TPC>
__device__ __forceinline__ void chunk_slots(const DispatchParams &p, int g, int s,
                                            int t0, int n_s, int i0,
                                            int32_t (*spos)[EP_MAX_WORLD],
                                            uint32_t *smask) {
    const int lane = threadIdx.x & 31;
    const int t = t0 + lane;
    const uint32_t m = (t < n_s) ? p.masks[(int64_t)s * p.T + t] : 0u;
    const int my_base = (lane < p.W) ? p.group_base[(int64_t)(g / kGroup) * p.W + lane] +
                                           p.chunk_local[(int64_t)g * p.W + lane]
                                     : 0;
    slots_from<TPC>(p, s, t0, i0, m, my_base, spos, smask);
}

// Up to kSelfChunks chunks (at most 256 tokens in all) every CTA computes
// the whole layout itself -- one round of id loads, then ballots -- instead
// of waiting for a layout kernel: the tiny workloads are pure latency, and
// one kernel fewer is the larger part of their step.  Warps take chunks
// c = warp, warp + kDispatchWarps, ...; CTA 0 writes the masks, chunk
// offsets, group totals and bases (one group), send counts and recv_count.
constexpr int kSelfChunks = EP_DISPATCH_SELF_LAYOUT_CHUNKS > 0 ? EP_DISPATCH_SELF_LAYOUT_CHUNKS : 1;
static_assert(kSelfChunks <= kGroup, "the self layout covers one layout group");

template <int TPC>
__device__ void self_layout_slots(const DispatchParams &p, int g, int s, int t0, int i0,
                                  int32_t (*spos)[EP_MAX_WORLD], uint32_t *smask,
                                  int (*s_cnt)[EP_MAX_WORLD], uint32_t *s_own) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    for (int c = warp; c < p.G; c += kDispatchWarps) {
        const int cs = c / p.nch;
        const int t = (c - cs * p.nch) * kChunk + lane;
        uint32_t mask = 0;
        bool bad = false;
        if (t < p.nt.n[cs]) {
            const int32_t *row = p.idx + ((int64_t)cs * p.T + t) * p.k;
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
                        bad = true;
                }
            }
        }
        if (blockIdx.x == 0) {
            if (bad) set_error(p.words, EP_DEVERR_BAD_INDEX);
            if (t < p.T) p.masks_w[(int64_t)cs * p.T + t] = mask;
        }
        int cnt = 0;
        for (int r = 0; r < p.W; ++r) {
            const uint32_t b = __ballot_sync(0xffffffffu, (mask >> r) & 1u);
            if (lane == r) cnt = __popc(b);
        }
        s_cnt[c][lane] = cnt;
        if (c == g) s_own[lane] = mask;
    }
    __syncthreads();
    if (warp == 0) {
        int my_base = 0;
        if (lane < p.W)
            for (int c = 0; c < g; ++c) my_base += s_cnt[c][lane];
        slots_from<TPC>(p, s, t0, i0, s_own[lane], my_base, spos, smask);
    } else if (warp == 1 && blockIdx.x == 0 && lane < p.W) {
        int run = 0;
        for (int c = 0; c < p.G; ++c) {
            p.chunk_local_w[(int64_t)c * p.W + lane] = run;
            run += s_cnt[c][lane];
        }
        p.group_tot_w[lane] = run;
        p.group_base_w[lane] = 0;
        p.group_base_w[p.W + lane] = run;              // row Q = 1: the totals
        if (run > p.cap) set_error(p.words, EP_DEVERR_CAPACITY);
        if (p.publish) p.recv_count[lane] = run;
        for (int sr = 0; sr < p.W; ++sr) {
            int cnt = 0;
            for (int c = sr * p.nch; c < (sr + 1) * p.nch; ++c) cnt += s_cnt[c][lane];
            p.send_counts[sr * p.W + lane] = cnt;
        }
    }
}

// Per-destination metadata of one token, written by one warp: all k
// weights, all k expert ids, src_pos, and for a pre-quantised input its
// block-scale row.
__device__ __forceinline__ void token_metadata(const DispatchParams &p, int s, int t,
                                               uint32_t m, const int32_t *slots) {
    const int lane = threadIdx.x & 31;
    const int64_t tok = (int64_t)s * p.T + t;
    float wv = 0.f;
    int32_t iv = 0;
    if (lane < p.k) {
        wv = __ldg(p.w + tok * p.k + lane);
        iv = __ldg(p.idx + tok * p.k + lane);
    }
    for (uint32_t mm = m; mm; mm &= mm - 1u) {
        const int r = __ffs(mm) - 1;
        const int slot = slots[r];
        if (slot >= p.cap) continue;
        char *seg = p.seg0 + (int64_t)r * p.seg_stride;
        if (lane < p.k) {
            reinterpret_cast<float *>(seg + p.off_w)[(int64_t)slot * p.k + lane] = wv;
            reinterpret_cast<int32_t *>(seg + p.off_idx)[(int64_t)slot * p.k + lane] = iv;
        }
        if (lane == 0)
            reinterpret_cast<int32_t *>(seg + p.off_src)[slot] = (int32_t)(s * p.T + t);
        if (p.scales_in) {
            float *dst = reinterpret_cast<float *>(seg + p.off_scales) + (int64_t)slot * p.nb;
            for (int b = lane; b < p.nb; b += 32) dst[b] = __ldg(p.scales_in + tok * p.nb + b);
        }
    }
}

// The last CTA of source s posts (s -> r) for every r, zero-count pairs
// included, after all of s's rows are stored.
template <int TPC>
__device__ __forceinline__ void notify_source_done(const DispatchParams &p, int s) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t tk = atom_add_acq_rel_gpu(p.words + kWordSrcDone + s, 1u);
        if (tk == (uint32_t)(p.nch * (kChunk / TPC)) - 1u) {
            p.words[kWordSrcDone + s] = 0u;
            for (int r = 0; r < p.W; ++r)
                st_release_gpu(p.dflags + r * p.W + s, p.epoch);
        }
    }
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 &v, float f[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// 4 values -> 4 E4M3 codes (byte i = element i) given the block scale.
__device__ __forceinline__ uint32_t quant4(const float *f, float scale) {
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float a = f[2 * i] / scale;
        const float b = f[2 * i + 1] / scale;
        const __nv_fp8x2_storage_t q =
            __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
        packed |= (uint32_t)q << (16 * i);
    }
    return packed;
}

// fl32(x / scale) from r = RN(1 / scale) and one FMA correction of the
// product (Markstein's division step: P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990).  For scale >= 2^-90 the residual x - q0*scale is exact
// for every quotient large enough to give a nonzero code, and the E4M3 code
// of the result equals that of the IEEE quotient for every bf16 x under every
// bf16 block maximum (fp8_quotient_check_kernel below compares the codes over
// all 1.07e9 pairs; ep_test_fp8_quotient_check runs it); smaller scales
// divide.  The
// residual is formed negated, q0*scale - x (the same magnitude: RN is
// symmetric), and applied with -r, so that for x = +-0 the sums of zeros
// keep the sign of x (the code of -0 is 0x80) with no sign fix-up.
__device__ __forceinline__ float quot_recip(float x, float scale, float r) {
    const float q0 = __fmul_rn(x, r);
    const float nres = __fmaf_rn(q0, scale, -x);
    return __fmaf_rn(nres, -r, q0);
}

// fl32(a / 448) for a block maximum a > 0 (a bf16 magnitude): the product
// with RN(1/448) and the same one-FMA correction.  Equal to the IEEE
// quotient for every finite non-negative bf16 a (proved on the host in exact
// rational arithmetic, and compared on the device for every positive finite
// a by fp8_quotient_check_kernel); a = inf gives inf.
__device__ __forceinline__ float block_scale(float a) {
#if EP_FP8_RECIP_QUOT
    constexpr float kInv448 = 0x1.24924ap-9f;   // RN(1/448)
    const float q0 = __fmul_rn(a, kInv448);
    const float e = __fmaf_rn(-q0, 448.0f, a);
    const float q = __fmaf_rn(e, kInv448, q0);
    return a <= 0x1.fffffep127f ? q : a;
#else
    return a / 448.0f;
#endif
}

__device__ __forceinline__ uint32_t quant4_recip(const float *f, float scale, float r) {
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float a = quot_recip(f[2 * i], scale, r);
        const float b = quot_recip(f[2 * i + 1], scale, r);
        const __nv_fp8x2_storage_t q =
            __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
        packed |= (uint32_t)q << (16 * i);
    }
    return packed;
}

// ------------------------------------------- quotient check (test harness)
// Every finite bf16 x under every positive finite bf16 block maximum a
// (|x| <= a, both signs): the block scale above against the IEEE quotient
// a / 448, and the codes of the dispatch's quotient (the reciprocal and one
// correction where the scale is >= 2^-90, as in dispatch_kernel) against the
// codes of the IEEE quotient x / scale.  One CTA per maximum; counts[0] =
// pairs, [1] = code mismatches, [2] = scale mismatches, [3] = pairs that took
// the reciprocal form.
constexpr int kQuotCheckThreads = 256;

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) {
    return __uint_as_float(b << 16);
}

__global__ void __launch_bounds__(kQuotCheckThreads)
fp8_quotient_check_kernel(unsigned long long *counts) {
    const uint32_t abits = blockIdx.x + 1u;          // 0x0001 .. 0x7F7F
    const float a = bf16_bits_to_float(abits);
    const float scale = block_scale(a);
    const float ieee_scale = a / 448.0f;
    const bool recip = EP_FP8_RECIP_QUOT && scale >= 0x1p-90f;
    const float r = __frcp_rn(scale);
    unsigned long long pairs = 0, bad = 0, fast = 0;
    // magnitudes 0..abits, four at a time, both signs
    for (uint32_t m0 = threadIdx.x * 4u; m0 <= abits; m0 += kQuotCheckThreads * 4u) {
        float f[4], g[4];
        int n = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t m = m0 + i;
            const bool in = m <= abits;
            n += in ? 1 : 0;
            f[i] = in ? bf16_bits_to_float(m) : 0.0f;
            g[i] = -f[i];
        }
        const uint32_t mask = n == 4 ? 0xffffffffu : ((1u << (8 * n)) - 1u);
        const uint32_t want_p = quant4(f, ieee_scale);
        const uint32_t want_n = quant4(g, ieee_scale);
        const uint32_t got_p = recip ? quant4_recip(f, scale, r) : quant4(f, scale);
        const uint32_t got_n = recip ? quant4_recip(g, scale, r) : quant4(g, scale);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t bm = 0xffu << (8 * i);
            if (bm & mask) {
                bad += ((want_p ^ got_p) & bm) ? 1 : 0;
                bad += ((want_n ^ got_n) & bm) ? 1 : 0;
            }
        }
        pairs += 2u * (unsigned)n;
        fast += recip ? 2u * (unsigned)n : 0u;
    }
    // block totals, then one atomic per counter
    __shared__ unsigned long long s_sum[3][kQuotCheckThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
        bad += __shfl_xor_sync(0xffffffffu, bad, o);
        fast += __shfl_xor_sync(0xffffffffu, fast, o);
    }
    if (lane == 0) {
        s_sum[0][warp] = pairs;
        s_sum[1][warp] = bad;
        s_sum[2][warp] = fast;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long t[3] = {0, 0, 0};
        for (int w = 0; w < kQuotCheckThreads / 32; ++w)
            for (int i = 0; i < 3; ++i) t[i] += s_sum[i][w];
        atomicAdd(counts + 0, t[0]);
        atomicAdd(counts + 1, t[1]);
        if (__float_as_uint(scale) != __float_as_uint(ieee_scale)) atomicAdd(counts + 2, 1ull);
        atomicAdd(counts + 3, t[2]);
    }
}

// ------------------------------------------------------------ register path

template <bool FP8, int U, int TPC>
__global__ void __launch_bounds__(kDispatchThreads)
dispatch_kernel(const DispatchParams p) {
    constexpr int kCtasPerChunk = kChunk / TPC;
    __shared__ DispatchSmem sm;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = blockIdx.x / kCtasPerChunk;
    const int i0 = (blockIdx.x - g * kCtasPerChunk) * TPC;
    const int s = g / p.nch;
    const int t0 = (g - s * p.nch) * kChunk;
    const int n_s = p.nt.n[s];

    grid_dependency_wait();
    if (p.self_layout) {
        __shared__ int s_cnt[kSelfChunks][EP_MAX_WORLD];
        __shared__ uint32_t s_own[kChunk];
        self_layout_slots<TPC>(p, g, s, t0, i0, sm.pos, sm.mask, s_cnt, s_own);
    } else if (warp == 0) {
        chunk_slots<TPC>(p, g, s, t0, n_s, i0, sm.pos, sm.mask);
    }
    __syncthreads();

    for (int i = i0 + warp; i < i0 + TPC; i += kDispatchWarps) {
        const int t = t0 + i;
        if (t >= n_s) break;
        const uint32_t m = sm.mask[i];
        if (m == 0u) continue;
        const int64_t tok = (int64_t)s * p.T + t;
        token_metadata(p, s, t, m, sm.pos[i]);

        const uint4 *src = p.x + tok * p.nvec;
        if constexpr (!FP8) {
            // The trip count is warp-uniform.
            for (int base = 0; base < p.nvec; base += 32 * U) {
                const int v0 = base + lane;
                uint4 buf[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + 32 * u;
                    if (v < p.nvec) buf[u] = ld_stream16(src + v);
                }
                for (uint32_t mm = m; mm; mm &= mm - 1u) {
                    const int r = __ffs(mm) - 1;
                    const int slot = sm.pos[i][r];
                    if (slot >= p.cap) continue;
                    uint4 *dst = reinterpret_cast<uint4 *>(
                                     p.seg0 + (int64_t)r * p.seg_stride + p.off_out) +
                                 (int64_t)slot * p.nvec;
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int v = v0 + 32 * u;
                        if (v < p.nvec) st_stream16(dst + v, buf[u]);
                    }
                }
            }
        } else {
            // A lane takes a pair of 16-byte vectors (16 elements); 8 lanes
            // hold one 128-element block; the warp covers 4 blocks per pair
            // index step.  npair = H/16 is a multiple of 8, so groups of 8
            // lanes are either wholly in range or wholly out of it, and the
            // trip count is warp-uniform (the amax shuffles need all lanes).
            const int npair = p.nvec >> 1;
#if EP_DISPATCH_FP8_PREFETCH
            static_assert(U == 1, "prefetch of the next pair is for one pair per lane");
            uint4 n0 = make_uint4(0u, 0u, 0u, 0u), n1 = n0;
            if (lane < npair) {
                n0 = ld_stream16(src + 2 * lane);
                n1 = ld_stream16(src + 2 * lane + 1);
            }
#endif
            for (int base = 0; base < npair; base += 32 * U) {
                uint4 q[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int pv = base + lane + 32 * u;
                    const bool active = pv < npair;
                    uint4 r0 = make_uint4(0u, 0u, 0u, 0u), r1 = r0;
#if EP_DISPATCH_FP8_PREFETCH
                    if (active) {
                        r0 = n0;
                        r1 = n1;
                    }
                    if (pv + 32 < npair) {
                        n0 = ld_stream16(src + 2 * (pv + 32));
                        n1 = ld_stream16(src + 2 * (pv + 32) + 1);
                    }
#else
                    if (active) {
                        r0 = ld_stream16(src + 2 * pv);
                        r1 = ld_stream16(src + 2 * pv + 1);
                    }
#endif
                    float f[16];
                    unpack_bf16x8(r0, f);
                    unpack_bf16x8(r1, f + 8);
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < 16; ++e) a = fmaxf(a, fabsf(f[e]));
#pragma unroll
                    for (int o = 4; o > 0; o >>= 1)
                        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
                    float scale = 0.f;
                    q[u] = make_uint4(0u, 0u, 0u, 0u);
                    if (a != 0.f) {
                        scale = block_scale(a);
#if EP_FP8_RECIP_QUOT
                        if (scale >= 0x1p-90f) {   // the same for the block's 8 lanes
                            const float r = __frcp_rn(scale);
                            q[u].x = quant4_recip(f, scale, r);
                            q[u].y = quant4_recip(f + 4, scale, r);
                            q[u].z = quant4_recip(f + 8, scale, r);
                            q[u].w = quant4_recip(f + 12, scale, r);
                        } else
#endif
                        {
                            q[u].x = quant4(f, scale);
                            q[u].y = quant4(f + 4, scale);
                            q[u].z = quant4(f + 8, scale);
                            q[u].w = quant4(f + 12, scale);
                        }
                    }
                    if (active && (lane & 7) == 0) sm.scales[warp][pv >> 3] = scale;
                }
                for (uint32_t mm = m; mm; mm &= mm - 1u) {
                    const int r = __ffs(mm) - 1;
                    const int slot = sm.pos[i][r];
                    if (slot >= p.cap) continue;
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        p.seg0 + (int64_t)r * p.seg_stride + p.off_out + (int64_t)slot * p.H);
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int pv = base + lane + 32 * u;
                        if (pv < npair) st_plain16(dst + pv, q[u]);
                    }
                }
            }
            __syncwarp();
            for (uint32_t mm = m; mm; mm &= mm - 1u) {
                const int r = __ffs(mm) - 1;
                const int slot = sm.pos[i][r];
                if (slot >= p.cap) continue;
                float *dst = reinterpret_cast<float *>(
                                 p.seg0 + (int64_t)r * p.seg_stride + p.off_scales) +
                             (int64_t)slot * p.nb;
                for (int b = lane; b < p.nb; b += 32) dst[b] = sm.scales[warp][b];
            }
            __syncwarp();
        }
    }

    if (p.notify) notify_source_done<TPC>(p, s);
}

// ---------------------------------------------------------------- bulk path
// Rows copied unchanged (bf16, or pre-quantised E4M3 codes whose scale rows
// the metadata warps copy) by the Tensor Memory Accelerator's bulk copies:
// thread 0 runs a
// ring of STAGES row buffers in shared memory.  Each source row is brought
// in ONCE by cp.async.bulk (completion counted on an mbarrier), then one
// bulk store per destination writes it out; a stage is refilled once the
// bulk stores that read it have finished reading.  Warps 1.. write the
// per-row metadata meanwhile.  Every mbarrier wait is bounded.

template <int STAGES, int TPC>
__global__ void __launch_bounds__(kDispatchThreads)
dispatch_bulk_kernel(const DispatchParams p) {
    constexpr int kCtasPerChunk = kChunk / TPC;
    extern __shared__ __align__(128) unsigned char stage_buf[];
    __shared__ BulkSmem sm;
    __shared__ __align__(8) uint64_t bar[STAGES];
    __shared__ int s_n;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = blockIdx.x / kCtasPerChunk;
    const int i0 = (blockIdx.x - g * kCtasPerChunk) * TPC;
    const int s = g / p.nch;
    const int t0 = (g - s * p.nch) * kChunk;
    const int n_s = p.nt.n[s];

    // The CTA's rows are its tokens below n_s.  Their loads do not depend on
    // the layout, so thread 0 issues them before waiting for it: launched
    // programmatically after the layout kernel, they overlap its tail.  (The
    // layout kernel waited for the kernel before it, so the rows are final.
    // With the self layout no layout kernel runs, and the loads follow the
    // wait instead.)
    const uint32_t bytes = (uint32_t)p.row_bytes;
    auto issue = [&](int j, uint64_t pol) {
        const int st = j % STAGES;
        const char *src = reinterpret_cast<const char *>(p.x) +
                          ((int64_t)s * p.T + t0 + sm.list[j]) * bytes;
        mbar_expect_tx(&bar[st], bytes);
        bulk_load(stage_buf + (size_t)st * bytes, src, bytes, &bar[st], pol);
    };
    if (threadIdx.x == 0) {
        int n = 0;
        for (int i = i0; i < i0 + TPC; ++i)
            if (t0 + i < n_s) sm.list[n++] = i;
        s_n = n;
        for (int i = 0; i < STAGES; ++i) mbar_init(&bar[i], 1);
        mbar_init_fence();
        if (!p.self_layout) {
            const uint64_t pol = l2_evict_first_policy();
            for (int j = 0; j < (n < STAGES ? n : STAGES); ++j) issue(j, pol);
        }
    }
    grid_dependency_wait();
    if (p.self_layout) {
        if (threadIdx.x == 0) {
            const uint64_t pol = l2_evict_first_policy();
            const int n0 = s_n;
            for (int j = 0; j < (n0 < STAGES ? n0 : STAGES); ++j) issue(j, pol);
        }
        __shared__ int s_cnt[kSelfChunks][EP_MAX_WORLD];
        __shared__ uint32_t s_own[kChunk];
        self_layout_slots<TPC>(p, g, s, t0, i0, sm.pos, sm.mask, s_cnt, s_own);
    } else if (warp == 0) {
        chunk_slots<TPC>(p, g, s, t0, n_s, i0, sm.pos, sm.mask);
    }
    __syncthreads();
    const int n = s_n;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int issued = n < STAGES ? n : STAGES;
            bool ok = true;
            for (int j = 0; j < n; ++j) {
                const int st = j % STAGES;
                if (!mbar_wait(&bar[st], (uint32_t)(j / STAGES) & 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const int i = sm.list[j];
                const uint32_t m = sm.mask[i];
                const unsigned char *src = stage_buf + (size_t)st * bytes;
                for (uint32_t mm = m; mm; mm &= mm - 1u) {
                    const int r = __ffs(mm) - 1;
                    const int slot = sm.pos[i][r];
                    if (slot >= p.cap) continue;
                    bulk_store(p.seg0 + (int64_t)r * p.seg_stride + p.off_out +
                                   (int64_t)slot * bytes,
                               src, bytes, pol);
                }
                bulk_commit();
                // refill the stage of token j-1: its stores were committed one
                // group ago, so waiting until at most the newest group is still
                // reading frees it
                if (j >= 1 && issued < n) {
                    bulk_wait_read1();
                    issue(issued, pol);
                    ++issued;
                }
            }
            if (!ok) {
                set_error(p.words, EP_DEVERR_TIMEOUT);
                // drain the loads still in flight (bounded), so no copy
                // writes shared memory after the CTA has gone
                for (int j = 0; j < issued; ++j)
                    mbar_wait(&bar[j % STAGES], (uint32_t)(j / STAGES) & 1u, p.timeout_ns);
            }
            bulk_wait_all();
            // order the bulk (async-proxy) row writes before the generic
            // release of the ready flags
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        __syncwarp();
    } else {
        for (int j = warp - 1; j < n; j += kDispatchWarps - 1) {
            const int i = sm.list[j];
            token_metadata(p, s, t0 + i, sm.mask[i], sm.pos[i]);
        }
    }

    if (p.notify) notify_source_done<TPC>(p, s);
}

__global__ void take_error_kernel(uint32_t *words) {
    words[kWordErrTaken] = atomicExch(words + kWordErr, 0u);
}

__global__ void dispatch_recv_kernel(uint32_t *dflags, uint32_t *words,
                                     const int32_t *totals, int32_t *recv_count,
                                     int W, int check, uint32_t epoch,
                                     int64_t timeout_ns) {
    const int tid = threadIdx.x;
    if (check && tid < W * W) {
        if (!wait_flag_eq(dflags + tid, epoch, timeout_ns))
            set_error(words, EP_DEVERR_TIMEOUT);
    }
    __syncthreads();
    if (tid < W) recv_count[tid] = totals[tid];
}

// Launch, programmatically dependent on the kernel before it when that is the
// layout kernel: the copy kernel's CTAs start while the layout finishes and
// wait for its results with griddepcontrol.wait.
template <typename Kernel>
cudaError_t launch_copy(Kernel kernel, int blocks, size_t dyn, bool after_layout,
                        const DispatchParams &p, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kDispatchThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = after_layout ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <bool FP8, int U, int TPC>
cudaError_t launch_dispatch_t(const Config &c, const DispatchParams &p, bool after_layout,
                              cudaStream_t st) {
    return launch_copy(dispatch_kernel<FP8, U, TPC>, c.G * (kChunk / TPC), 0, after_layout, p, st);
}

// The ring never needs more stages than the CTA has tokens.
constexpr int kBulkStages =
    EP_DISPATCH_BULK_STAGES < EP_DISPATCH_TPC ? EP_DISPATCH_BULK_STAGES : EP_DISPATCH_TPC;

// Residency cap: when a CTA moves a lot of data (its tokens x up to
// min(W,k) destinations x the row, >= 64 KB), fewer bulk-copy CTAs per SM --
// fewer concurrent row streams per SM -- measured faster than filling every
// slot, so the dynamic shared memory is padded until at most
// max(EP_DISPATCH_BULK_CTAS_PER_SM, kBulkStreamBytes / row) CTAs fit: two
// CTAs per SM for 14 KB rows, four for 7 KB E4M3 code rows.  Small rows or
// few destinations keep full residency (per-CTA set-up would dominate).
constexpr size_t kBulkStreamBytes = 2 * 14336;

template <int STAGES, int TPC>
cudaError_t launch_dispatch_bulk(const Config &c, const DispatchParams &p, bool after_layout,
                                 cudaStream_t st) {
    // Function attributes are per device: cache the opted-in size and the
    // shared-memory figures per device.
    constexpr int kMaxDevices = 64;
    // (atomics: handles on different host threads may launch at once)
    static std::atomic<size_t> configured[kMaxDevices];
    static std::atomic<long> per_sm[kMaxDevices];
    static std::atomic<long> fixed[kMaxDevices];   // reserved + static shared memory per CTA
    static std::atomic<int> sms[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const size_t row = (size_t)p.row_bytes;
    size_t dyn = (size_t)STAGES * row;
    const size_t per_cta = (size_t)TPC * (size_t)(c.W < c.k ? c.W : c.k) * row;
    const long blocks = (long)c.G * (kChunk / TPC);
    if (EP_DISPATCH_BULK_CTAS_PER_SM > 0 && per_cta >= 64 * 1024) {
        if (per_sm[dev].load(std::memory_order_acquire) == 0) {
            int sm_bytes = 0, reserved = 0, n_sm = 0;
            cudaFuncAttributes fa;
            if ((e = cudaDeviceGetAttribute(&sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                            dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock,
                                            dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) !=
                    cudaSuccess ||
                (e = cudaFuncGetAttributes(&fa, dispatch_bulk_kernel<STAGES, TPC>)) != cudaSuccess)
                return e;
            fixed[dev].store((long)reserved + (long)fa.sharedSizeBytes, std::memory_order_relaxed);
            sms[dev].store(n_sm, std::memory_order_relaxed);
            per_sm[dev].store(sm_bytes, std::memory_order_release);
        }
        long ctas = (long)(kBulkStreamBytes / row);
        if (ctas < EP_DISPATCH_BULK_CTAS_PER_SM) ctas = EP_DISPATCH_BULK_CTAS_PER_SM;
        // Short grids keep full residency: the 1024-CTA decode copy (3.4 capped
        // waves) measured 84.8 against 85.9 us uncapped, while 2048 CTAs (6.7
        // waves) measured 61.4 against 59.6 us capped.
        const long capped_wave = ctas * (long)sms[dev].load(std::memory_order_relaxed);
        if (blocks >= (long)EP_DISPATCH_BULK_CAP_MIN_WAVES * capped_wave) {
            const long share = (per_sm[dev].load(std::memory_order_acquire) / ctas -
                                fixed[dev].load(std::memory_order_relaxed)) &
                               ~127L;
            if (share > 0 && (size_t)share > dyn) dyn = (size_t)share;
        }
    }
    if (dyn > configured[dev].load(std::memory_order_acquire)) {   // opt in to the dynamic size
        // never lower the attribute under a concurrent launch that needs more
        static std::mutex mu;
        std::lock_guard<std::mutex> lock(mu);
        if (dyn > configured[dev].load(std::memory_order_relaxed)) {
            e = cudaFuncSetAttribute(dispatch_bulk_kernel<STAGES, TPC>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
            if (e != cudaSuccess) return e;
            configured[dev].store(dyn, std::memory_order_release);
        }
    }
    return launch_copy(dispatch_bulk_kernel<STAGES, TPC>, c.G * (kChunk / TPC), dyn, after_layout,
                       p, st);
}

}  // namespace

cudaError_t launch_dispatch(const Config &c, const Workspace &ws,
                            const DispatchArgs &a, cudaStream_t st) {
    DispatchParams p;
    p.x = reinterpret_cast<const uint4 *>(a.x);
    p.scales_in = a.scales_in;
    p.w = a.w;
    p.idx = a.idx;
    p.masks = ws.masks;
    p.chunk_local = ws.chunk_local;
    p.group_base = ws.group_base;
    p.pos = ws.pos;
    p.seg0 = ws.seg0;
    p.seg_stride = ws.seg_stride;
    p.off_out = ws.off_out;
    p.off_scales = ws.off_scales;
    p.off_w = ws.off_w;
    p.off_idx = ws.off_idx;
    p.off_src = ws.off_src;
    p.words = ws.words;
    p.dflags = ws.dflags;
    p.W = c.W; p.k = c.k; p.T = c.T; p.H = c.H; p.nch = c.nch; p.cap = c.cap;
    p.nvec = c.nvec; p.nb = c.nb;
    p.row_bytes = c.fp8 ? c.H : c.H * 2;
    p.notify = c.early_notify ? 1 : 0;
    p.epoch = a.epoch;
    p.timeout_ns = c.timeout_ns;
    p.nt = a.nt;
    p.self_layout = a.self_layout ? 1 : 0;
    p.E = c.E; p.Er = c.Er; p.G = c.G;
    p.publish = a.publish ? 1 : 0;
    p.masks_w = ws.masks;
    p.chunk_local_w = ws.chunk_local;
    p.group_tot_w = ws.group_tot;
    p.group_base_w = ws.group_base;
    p.send_counts = ws.send_counts;
    p.recv_count = ws.recv_count;
    // the self-layout copy is the step's first kernel: launched programmatically
    // after whatever precedes it, it waits for that kernel before any read
    const bool pdl = (a.after_layout || a.self_layout) && EP_DISPATCH_PDL;
    if (c.fp8 && !a.scales_in)      // fused quantisation
        return launch_dispatch_t<true, EP_DISPATCH_FP8_UNROLL, EP_DISPATCH_REG_TPC>(c, p, pdl, st);
    // rows copied unchanged: bf16, or pre-quantised codes (H <= 16384 bytes)
#if EP_DISPATCH_BULK_STAGES > 0
    if ((size_t)kBulkStages * p.row_bytes <= 160 * 1024)
        return launch_dispatch_bulk<kBulkStages, EP_DISPATCH_TPC>(c, p, pdl, st);
#endif
    if (c.fp8)   // the register path copies bf16-sized vectors: not for codes
        return cudaErrorInvalidValue;
    return launch_dispatch_t<false, EP_DISPATCH_UNROLL, EP_DISPATCH_REG_TPC>(c, p, pdl, st);
}

cudaError_t launch_dispatch_recv(const Config &c, const Workspace &ws,
                                 bool check_flags, uint32_t epoch,
                                 cudaStream_t st) {
    const int threads = ((c.W * c.W + 31) / 32) * 32;
    dispatch_recv_kernel<<<1, threads, 0, st>>>(
        ws.dflags, ws.words, ws.group_base + (int64_t)c.Q * c.W, ws.recv_count,
        c.W, check_flags ? 1 : 0, epoch, c.timeout_ns);
    return cudaGetLastError();
}

int self_layout_chunks() { return EP_DISPATCH_SELF_LAYOUT_CHUNKS; }

cudaError_t launch_take_error(const Workspace &ws, cudaStream_t st) {
    take_error_kernel<<<1, 1, 0, st>>>(ws.words);
    return cudaGetLastError();
}

cudaError_t launch_fp8_quotient_check(unsigned long long *d_counts, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(d_counts, 0, 4 * sizeof(unsigned long long), st);
    if (e != cudaSuccess) return e;
    fp8_quotient_check_kernel<<<0x7F7F, kQuotCheckThreads, 0, st>>>(d_counts);
    return cudaGetLastError();
}

}  // namespace ep
