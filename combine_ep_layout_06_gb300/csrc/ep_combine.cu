// Combine: gather each source token's expert-side rows back from its
// destination ranks and reduce them in fp32, ranks ascending, to one bf16
// row (and the same ordered sum of the expert-side weight rows).  Also the
// combine ready flags (send phase / receive wait) and the identity expert of
// the correctness harness.
//
// Definition (ROCm MORI "Communication APIs", MORI-EP, "EpDispatchCombineOp
// methods": combine(input, weights, indices) -> (output, weights), "combine
// expert outputs back"; combine_send()/combine_recv(); and the "AsyncLL v2
// SDMA overlap" section for the split receive): out[s][t] = bf16_rne(
// +0.0f + y_r0[p0] + y_r1[p1] + ...) over r in D(s,t) ascending, each '+' an
// fp32 add.
//
// GB300 mapping.  One warp per source token.  Lanes read the token's W
// slots; for each group of U 16-byte column vectors a lane issues the loads
// of ALL of the token's (<= MAXD) rows before it adds any, so up to
// U * MAXD independent 16-byte loads per lane are in flight, then it adds
// them in rank order and writes 16 bytes of bf16.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "ep_device.cuh"

namespace ep {
namespace {

#ifndef EP_COMBINE_WARPS
#define EP_COMBINE_WARPS 8
#endif
#ifndef EP_COMBINE_MIN_BLOCKS
#define EP_COMBINE_MIN_BLOCKS 3    // 3 CTAs of 8 warps per SM: <= 80 registers
#endif
#ifndef EP_COMBINE_UNROLL8
#define EP_COMBINE_UNROLL8 2       // column vectors in flight per row, <= 8 rows
#endif

constexpr int kCombineWarps = EP_COMBINE_WARPS;
constexpr int kCombineThreads = kCombineWarps * 32;

struct CombineParams {
    const char *y;
    int64_t y_stride;
    const char *w_in;
    int64_t w_stride;
    const int32_t *idx;
    const int32_t *pos;
    uint16_t *out;
    float *out_w;
    uint32_t *words;
    const uint32_t *cflags;
    int W, E, Er, k, T, cap, nvec;
    int fused_wait;
    uint32_t epoch;
    int64_t timeout_ns;
    TokenCounts nt;
};

__device__ __forceinline__ uint4 ld_coherent16(const void *p) {
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void add_bf16x8(float acc[8], const uint4 &v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = acc[2 * i] + __uint_as_float(w[i] << 16);
        acc[2 * i + 1] = acc[2 * i + 1] + __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return a | (b << 16);
}

// The fused receive: warp 0 of the CTA waits (bounded) for the combine
// ready flags of every source rank its tokens belong to; the CTA barrier
// then releases the gather warps.
__device__ void fused_receive_wait(const CombineParams &p) {
    if ((threadIdx.x >> 5) == 0) {
        const int lane = threadIdx.x & 31;
        const int64_t first = (int64_t)blockIdx.x * kCombineWarps;
        const int64_t last = min(first + kCombineWarps, (int64_t)p.W * p.T) - 1;
        const int s0 = (int)(first / p.T);
        const int s1 = (int)(last / p.T);
        bool ok = true;
        for (int s = s0; s <= s1; ++s)
            for (int r = lane; r < p.W; r += 32)
                ok &= wait_flag_eq(p.cflags + s * p.W + r, p.epoch, p.timeout_ns);
        if (!ok) set_error(p.words, EP_DEVERR_TIMEOUT);
    }
    __syncthreads();
}

__device__ __forceinline__ void add_f32x4(float *acc, const uint4 &v) {
    acc[0] = acc[0] + __uint_as_float(v.x);
    acc[1] = acc[1] + __uint_as_float(v.y);
    acc[2] = acc[2] + __uint_as_float(v.z);
    acc[3] = acc[3] + __uint_as_float(v.w);
}

// F32: the expert rows are fp32 (two 16-byte loads per 8 output elements).
template <int MAXD, int U, bool COHERENT, bool F32>
__global__ void __launch_bounds__(kCombineThreads, EP_COMBINE_MIN_BLOCKS)
combine_kernel(const CombineParams p) {
    constexpr int NL = F32 ? 2 : 1;       // 16-byte loads per output vector
    if (p.fused_wait) fused_receive_wait(p);

    const int lane = threadIdx.x & 31;
    const int64_t tok = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (tok >= (int64_t)p.W * p.T) return;
    const int s = (int)(tok / p.T);
    const int t = (int)(tok - (int64_t)s * p.T);
    if (t >= p.nt.n[s]) return;

    const int pr = (lane < p.W) ? p.pos[tok * p.W + lane] : -1;
    const uint32_t present = __ballot_sync(0xffffffffu, pr >= 0);
    const uint32_t dm = __ballot_sync(0xffffffffu, pr >= 0 && pr < p.cap);

    if (p.idx) {   // the indices must name the dispatch's destination set
        uint32_t rb = 0;
        if (lane < p.k) {
            const int32_t e = p.idx[tok * p.k + lane];
            if ((uint32_t)e < (uint32_t)p.E) rb = 1u << (e / p.Er);
        }
        rb = __reduce_or_sync(0xffffffffu, rb);
        if (rb != present && lane == 0) set_error(p.words, EP_DEVERR_COMBINE_MISMATCH);
    }

    // rows of this token, ranks ascending
    const char *rows[MAXD];
    int nd = 0;
    {
        uint32_t mm = dm;
#pragma unroll
        for (int j = 0; j < MAXD; ++j) {
            rows[j] = nullptr;
            if (mm) {
                const int r = __ffs(mm) - 1;
                mm &= mm - 1u;
                const int slot = __shfl_sync(0xffffffffu, pr, r);
                rows[j] = p.y + (int64_t)r * p.y_stride + (int64_t)slot * p.nvec * 16 * NL;
                nd = j + 1;
            }
        }
    }

    uint4 *out_row = reinterpret_cast<uint4 *>(p.out) + tok * p.nvec;
    for (int v0 = lane; v0 < p.nvec; v0 += 32 * U) {
        uint4 val[U][MAXD][NL];
#pragma unroll
        for (int j = 0; j < MAXD; ++j) {
            if (j < nd) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + 32 * u;
                    if (v < p.nvec) {
#pragma unroll
                        for (int l = 0; l < NL; ++l) {
                            const char *a = rows[j] + ((int64_t)v * NL + l) * 16;
                            val[u][j][l] = COHERENT ? ld_coherent16(a) : ld_stream16(a);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 32 * u;
            if (v >= p.nvec) continue;
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
            for (int j = 0; j < MAXD; ++j) {
                if (j < nd) {
                    if constexpr (F32) {
                        add_f32x4(acc, val[u][j][0]);
                        add_f32x4(acc + 4, val[u][j][1]);
                    } else {
                        add_bf16x8(acc, val[u][j][0]);
                    }
                }
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            st_stream16(out_row + v, o);
        }
    }

    if (p.w_in && p.out_w) {
        float aw = 0.0f;
        for (uint32_t mm = dm; mm; mm &= mm - 1u) {
            const int r = __ffs(mm) - 1;
            const int slot = __shfl_sync(0xffffffffu, pr, r);
            if (lane < p.k)
                aw = aw + reinterpret_cast<const float *>(
                              p.w_in + (int64_t)r * p.w_stride)[(int64_t)slot * p.k + lane];
        }
        if (lane < p.k) p.out_w[tok * p.k + lane] = aw;
    }
}

__global__ void flags_post_kernel(uint32_t *flags, int n, uint32_t epoch) {
    const int i = threadIdx.x;
    if (i < n) st_release_gpu(flags + i, epoch);
}

__global__ void flags_wait_kernel(const uint32_t *flags, uint32_t *words,
                                  int n, uint32_t epoch, int64_t timeout_ns) {
    const int i = threadIdx.x;
    if (i < n && !wait_flag_eq(flags + i, epoch, timeout_ns))
        set_error(words, EP_DEVERR_TIMEOUT);
}

// Identity expert: warp per received row.
__global__ void __launch_bounds__(256)
identity_expert_kernel(const char *seg0, int64_t seg_stride, int64_t off_out,
                       int64_t off_scales, int64_t off_w, int64_t off_idx,
                       const int32_t *totals, char *y, int64_t y_stride,
                       int W, int E, int Er, int k, int H, int cap, int fp8,
                       int y_f32) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int r = (int)(gw / cap);
    const int slot = (int)(gw - (int64_t)r * cap);
    if (r >= W) return;
    if (slot >= min(totals[r], cap)) return;
    const char *seg = seg0 + (int64_t)r * seg_stride;
    const float *wrow = reinterpret_cast<const float *>(seg + off_w) + (int64_t)slot * k;
    const int32_t *irow = reinterpret_cast<const int32_t *>(seg + off_idx) + (int64_t)slot * k;
    float alpha = 0.0f;
    for (int j = 0; j < k; ++j) {
        const int32_t e = irow[j];
        if ((uint32_t)e < (uint32_t)E && e / Er == r) alpha = alpha + wrow[j];
    }
    const int nvec = H / 8;
    uint4 *yrow = reinterpret_cast<uint4 *>(y + (int64_t)r * y_stride) +
                  (int64_t)slot * nvec * (y_f32 ? 2 : 1);
    for (int v = lane; v < nvec; v += 32) {
        float f[8];
        if (fp8) {
            const uint2 q = *reinterpret_cast<const uint2 *>(
                seg + off_out + (int64_t)slot * H + (int64_t)v * 8);
            const float sc = reinterpret_cast<const float *>(seg + off_scales)
                [(int64_t)slot * (H / 128) + (v >> 4)];
            const uint32_t qw[2] = {q.x, q.y};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const __nv_fp8_storage_t code = (qw[e >> 2] >> (8 * (e & 3))) & 0xffu;
                const __half_raw hr = __nv_cvt_fp8_to_halfraw(code, __NV_E4M3);
                const float val = __half2float(__half(hr));
                f[e] = val * sc;
            }
        } else {
            const uint4 raw = reinterpret_cast<const uint4 *>(seg + off_out)[(int64_t)slot * nvec + v];
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = __uint_as_float(w4[i] << 16);
                f[2 * i + 1] = __uint_as_float(w4[i] & 0xffff0000u);
            }
        }
        if (y_f32) {
            float g[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) g[e] = f[e] * alpha;
            yrow[2 * v] = make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]),
                                     __float_as_uint(g[2]), __float_as_uint(g[3]));
            yrow[2 * v + 1] = make_uint4(__float_as_uint(g[4]), __float_as_uint(g[5]),
                                         __float_as_uint(g[6]), __float_as_uint(g[7]));
        } else {
            uint4 o;
            o.x = pack_bf16x2(f[0] * alpha, f[1] * alpha);
            o.y = pack_bf16x2(f[2] * alpha, f[3] * alpha);
            o.z = pack_bf16x2(f[4] * alpha, f[5] * alpha);
            o.w = pack_bf16x2(f[6] * alpha, f[7] * alpha);
            yrow[v] = o;
        }
    }
}

template <int MAXD, int U, bool COH, bool F32>
cudaError_t launch_combine_t(const Config &c, const CombineParams &p,
                             cudaStream_t st) {
    const int64_t tokens = (int64_t)c.W * c.T;
    const int blocks = (int)((tokens + kCombineWarps - 1) / kCombineWarps);
    combine_kernel<MAXD, U, COH, F32><<<blocks, kCombineThreads, 0, st>>>(p);
    return cudaGetLastError();
}

template <int MAXD, int U>
cudaError_t launch_combine_m(const Config &c, const CombineParams &p,
                             cudaStream_t st) {
    if (c.y_f32) {
        constexpr int U32 = U > 1 ? U / 2 : 1;    // twice the bytes per vector
        if (p.fused_wait) return launch_combine_t<MAXD, U32, true, true>(c, p, st);
        return launch_combine_t<MAXD, U32, false, true>(c, p, st);
    }
    if (p.fused_wait) return launch_combine_t<MAXD, U, true, false>(c, p, st);
    return launch_combine_t<MAXD, U, false, false>(c, p, st);
}

}  // namespace

cudaError_t launch_combine(const Config &c, const Workspace &ws,
                           const CombineArgs &a, cudaStream_t st) {
    CombineParams p;
    p.y = a.y;
    p.y_stride = a.y_stride;
    p.w_in = a.w_in;
    p.w_stride = a.w_stride;
    p.idx = a.idx;
    p.pos = ws.pos;
    p.out = a.out;
    p.out_w = a.out_w;
    p.words = ws.words;
    p.cflags = ws.cflags;
    p.W = c.W; p.E = c.E; p.Er = c.Er; p.k = c.k; p.T = c.T; p.cap = c.cap;
    p.nvec = c.nvec;
    p.fused_wait = a.fused_wait ? 1 : 0;
    p.epoch = a.epoch;
    p.timeout_ns = c.timeout_ns;
    p.nt = a.nt;
    const int maxd = c.W < c.k ? c.W : c.k;   // |D(s,t)| <= min(W, k)
    if (maxd <= 2) return launch_combine_m<2, 4>(c, p, st);
    if (maxd <= 4) return launch_combine_m<4, 2>(c, p, st);
    if (maxd <= 8) return launch_combine_m<8, EP_COMBINE_UNROLL8>(c, p, st);
    if (maxd <= 16) return launch_combine_m<16, 1>(c, p, st);
    return launch_combine_m<32, 1>(c, p, st);
}

cudaError_t launch_combine_notify(const Config &c, const Workspace &ws,
                                  uint32_t epoch, cudaStream_t st) {
    const int n = c.W * c.W;
    flags_post_kernel<<<1, ((n + 31) / 32) * 32, 0, st>>>(ws.cflags, n, epoch);
    return cudaGetLastError();
}

cudaError_t launch_combine_wait(const Config &c, const Workspace &ws,
                                uint32_t epoch, cudaStream_t st) {
    const int n = c.W * c.W;
    flags_wait_kernel<<<1, ((n + 31) / 32) * 32, 0, st>>>(ws.cflags, ws.words, n,
                                                          epoch, c.timeout_ns);
    return cudaGetLastError();
}

cudaError_t launch_identity_expert(const Config &c, const Workspace &ws,
                                   char *y, int64_t y_stride, cudaStream_t st) {
    const int64_t rows = (int64_t)c.W * c.cap;
    const int blocks = (int)((rows + 7) / 8);
    identity_expert_kernel<<<blocks, 256, 0, st>>>(
        ws.seg0, ws.seg_stride, ws.off_out, ws.off_scales, ws.off_w, ws.off_idx,
        ws.group_base + (int64_t)c.Q * c.W, y, y_stride, c.W, c.E, c.Er, c.k,
        c.H, c.cap, c.fp8 ? 1 : 0, c.y_f32 ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace ep
