// Standard-MoE conversion of the received rows ("Choosing an EP API and
// backend", EPv2 feature list: "standard-MoE conversion"; reading: per-local-
// expert contiguous groups) and its inverse before combine.
//
// On rank r, the entries are the pairs (received row p < n_r, top-k slot j)
// whose expert lives on r; they are grouped per local expert e in e order,
// (p, j) ascending inside a group.  slot(p, j) = offset[r][e] + number of
// earlier entries of e.  The inverse writes, for every received row,
// bf16(+0 + sum over its entries, j ascending, of fl32(w_j * y[slot])) into
// the registered combine buffer.
//
// GB300 mapping, deterministic (scans, no atomics decide a slot):
//  count   one warp per 32-row chunk of a rank: per local expert, the warp
//          reduce-adds its lanes' entry counts;
//  scan    one warp per (rank, expert): exclusive prefix over the chunks; the
//          last CTA turns expert totals into per-rank offsets;
//  group   one CTA per chunk: warp 0 derives every entry's slot (per-expert
//          warp scan of the lanes' counts); then each payload row is read
//          ONCE and stored to each of its entry slots -- by TMA bulk copies
//          through a shared-memory ring, or (long rows) by 16-byte vectors;
//  ungroup one warp per received row: the loads of all its entries' rows for
//          several column vectors are in flight together (more vectors when
//          the row has fewer entries), then the weighted fp32 sum in slot
//          order (a rounded multiply, then a rounded add: no contraction).
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "ep_device.cuh"

namespace ep {
namespace {

#ifndef EP_MOE_GROUP_BULK_STAGES
#define EP_MOE_GROUP_BULK_STAGES 4    // grouping by TMA bulk copies (0: register path)
#endif
#ifndef EP_MOE_GROUP_EARLY_LOADS
#define EP_MOE_GROUP_EARLY_LOADS 1    // grouping: row loads issued before the slot scan
#endif

constexpr int kMoeWarps = 8;
constexpr int kGroupWarps = 4;

struct MoeParams {
    char *seg0;
    int64_t seg_stride;
    int64_t off_out, off_scales, off_w, off_idx, off_xg, off_xgs, off_gsrc, off_gw, off_eslot,
        off_comb;
    const int32_t *totals;      // [W] rows received per rank (layout totals)
    int32_t *cnt, *base, *count, *offset;
    uint32_t *words;
    int W, E, Er, k, H, cap, gcap, nrc, nb, row_bytes;
    int64_t timeout_ns;        // bound of every mbarrier wait
};

__device__ __forceinline__ int rank_rows(const MoeParams &p, int r) {
    return min(p.totals[r], p.cap);
}

// Local expert of each of the lane's k selections (-1 if not on rank r).
__device__ __forceinline__ void local_experts(const MoeParams &p, int r, int row, bool valid,
                                              int *lid) {
    const int32_t *ids = reinterpret_cast<const int32_t *>(
                             p.seg0 + (int64_t)r * p.seg_stride + p.off_idx) +
                         (int64_t)row * p.k;
    for (int j = 0; j < p.k; ++j) {
        int e = -1;
        if (valid) {
            const int32_t g = ids[j];
            if ((uint32_t)g < (uint32_t)p.E && g / p.Er == r) e = g - r * p.Er;
        }
        lid[j] = e;
    }
}

__global__ void __launch_bounds__(kMoeWarps * 32) moe_count_kernel(const MoeParams p) {
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kMoeWarps + (threadIdx.x >> 5);
    if (gw >= p.W * p.nrc) return;
    const int r = gw / p.nrc, c = gw - r * p.nrc;
    const int row = c * kChunk + lane;
    int lid[EP_MAX_TOPK];
    local_experts(p, r, row, row < rank_rows(p, r), lid);
    int32_t *dst = p.cnt + ((int64_t)r * p.nrc + c) * p.Er;
    for (int e0 = 0; e0 < p.Er; e0 += 32) {
        int mine = 0;
        for (int e = e0; e < min(p.Er, e0 + 32); ++e) {
            int ce = 0;
            for (int j = 0; j < p.k; ++j) ce += (lid[j] == e);
            const int tot = __reduce_add_sync(0xffffffffu, ce);
            if (lane == e - e0) mine = tot;
        }
        if (e0 + lane < p.Er) dst[e0 + lane] = mine;
    }
}

__global__ void __launch_bounds__(kMoeWarps * 32) moe_scan_kernel(const MoeParams p) {
    __shared__ int s_last;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int seq = blockIdx.x * kMoeWarps + warp;
    if (seq < p.W * p.Er) {
        const int r = seq / p.Er, e = seq - r * p.Er;
        const int per = (p.nrc + 31) / 32;
        const int c0 = min(p.nrc, lane * per), c1 = min(p.nrc, c0 + per);
        const int32_t *src = p.cnt + (int64_t)r * p.nrc * p.Er + e;
        int32_t *dst = p.base + (int64_t)r * p.nrc * p.Er + e;
        int sum = 0;
        for (int cc = c0; cc < c1; ++cc) sum += src[(int64_t)cc * p.Er];
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        int run = incl - sum;
        for (int cc = c0; cc < c1; ++cc) {
            dst[(int64_t)cc * p.Er] = run;
            run += src[(int64_t)cc * p.Er];
        }
        if (lane == 31) p.count[seq] = incl;
    }
    // the last CTA turns per-rank expert totals into offsets
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = atom_add_acq_rel_gpu(p.words + kWordMoeDone, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int r = warp; r < p.W; r += kMoeWarps) {
        int carry = 0;
        for (int e0 = 0; e0 < p.Er; e0 += 32) {
            const int e = e0 + lane;
            const int v = e < p.Er ? __ldcg(p.count + r * p.Er + e) : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += x;
            }
            if (e < p.Er) p.offset[r * p.Er + e] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0 && carry > p.gcap) set_error(p.words, EP_DEVERR_CAPACITY);
    }
    if (threadIdx.x == 0) p.words[kWordMoeDone] = 0;
}

struct GroupSmem {
    int32_t slot[kChunk][EP_MAX_TOPK];
};

// Warp 0: every entry slot of the chunk's 32 rows (per-expert warp scans
// of the lanes' counts) into smem, and the entry-slot rows (-1: no entry).
__device__ __forceinline__ void group_slots(const MoeParams &p, int r, int c, int n_r, char *seg,
                                            GroupSmem &sm) {
    const int lane = threadIdx.x & 31;
    const int row = c * kChunk + lane;
    int lid[EP_MAX_TOPK];
    int slot[EP_MAX_TOPK];
    local_experts(p, r, row, row < n_r, lid);
    for (int j = 0; j < p.k; ++j) slot[j] = -1;
    const int32_t *brow = p.base + ((int64_t)r * p.nrc + c) * p.Er;
    for (int e = 0; e < p.Er; ++e) {
        int ce = 0;
        for (int j = 0; j < p.k; ++j) ce += (lid[j] == e);
        if (!__any_sync(0xffffffffu, ce > 0)) continue;
        int incl = ce;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        int next = p.offset[r * p.Er + e] + brow[e] + incl - ce;
        for (int j = 0; j < p.k; ++j)
            if (lid[j] == e) slot[j] = next++;
    }
    for (int j = 0; j < p.k; ++j) sm.slot[lane][j] = slot[j];
    if (row < p.cap) {
        int32_t *es = reinterpret_cast<int32_t *>(seg + p.off_eslot) + (int64_t)row * p.k;
        for (int j = 0; j < p.k; ++j) es[j] = slot[j];
    }
}

// Metadata of row i's entries (one warp): source code p*k + j, weight, and
// the FP8 block scales.
__device__ __forceinline__ void group_metadata(const MoeParams &p, int row, int i, char *seg,
                                               const GroupSmem &sm) {
    const int lane = threadIdx.x & 31;
    if (lane < p.k) {
        const int q = sm.slot[i][lane];
        if (q >= 0 && q < p.gcap) {
            reinterpret_cast<int32_t *>(seg + p.off_gsrc)[q] = row * p.k + lane;
            reinterpret_cast<float *>(seg + p.off_gw)[q] =
                reinterpret_cast<const float *>(seg + p.off_w)[(int64_t)row * p.k + lane];
        }
    }
    if (p.nb) {
        const float *ssrc = reinterpret_cast<const float *>(seg + p.off_scales) + (int64_t)row * p.nb;
        for (int j = 0; j < p.k; ++j) {
            const int q = sm.slot[i][j];
            if (q < 0 || q >= p.gcap) continue;
            float *sdst = reinterpret_cast<float *>(seg + p.off_xgs) + (int64_t)q * p.nb;
            for (int b = lane; b < p.nb; b += 32) sdst[b] = ssrc[b];
        }
    }
}

// Register path: the warps read each payload row once (16-byte vectors,
// 4 in flight per lane) and store it to every entry slot.
__global__ void __launch_bounds__(kGroupWarps * 32) moe_group_kernel(const MoeParams p) {
    __shared__ GroupSmem sm;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x / p.nrc, c = blockIdx.x - r * p.nrc;
    const int n_r = rank_rows(p, r);
    char *seg = p.seg0 + (int64_t)r * p.seg_stride;
    if (warp == 0) group_slots(p, r, c, n_r, seg, sm);
    __syncthreads();

    const int nvec = p.row_bytes / 16;
    for (int i = warp; i < kChunk; i += kGroupWarps) {
        const int row = c * kChunk + i;
        if (row >= n_r) break;
        const uint4 *src = reinterpret_cast<const uint4 *>(seg + p.off_out) + (int64_t)row * nvec;
        group_metadata(p, row, i, seg, sm);
        // payload: read once, store to every entry slot
        for (int v0 = lane; v0 < nvec; v0 += 32 * 4) {
            uint4 buf[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v0 + 32 * u < nvec) buf[u] = ld_stream16(src + v0 + 32 * u);
            for (int j = 0; j < p.k; ++j) {
                const int q = sm.slot[i][j];
                if (q < 0 || q >= p.gcap) continue;
                uint4 *dst = reinterpret_cast<uint4 *>(seg + p.off_xg) + (int64_t)q * nvec;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (v0 + 32 * u < nvec) st_stream16(dst + v0 + 32 * u, buf[u]);
            }
        }
    }
}

// Bulk path: thread 0 runs a ring of STAGES row buffers in shared memory;
// each received row comes in once by cp.async.bulk (completion on an
// mbarrier, bounded waits), then one bulk store per entry slot writes it
// out, and a stage is refilled once the stores that read it are done
// reading.  Warps 1.. write the entries' metadata meanwhile.
template <int STAGES>
__global__ void __launch_bounds__(kGroupWarps * 32) moe_group_bulk_kernel(const MoeParams p) {
    extern __shared__ __align__(128) unsigned char gstage[];
    __shared__ GroupSmem sm;
    __shared__ __align__(8) uint64_t bar[STAGES];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x / p.nrc, c = blockIdx.x - r * p.nrc;
    const int n_r = rank_rows(p, r);
    char *seg = p.seg0 + (int64_t)r * p.seg_stride;
    const int rows = max(0, min(kChunk, n_r - c * kChunk));
    const uint32_t bytes = (uint32_t)p.row_bytes;
    const uint64_t pol = 0;   // these copies take no L2 cache hint
    auto issue = [&](int i) {
        const int st = i % STAGES;
        mbar_expect_tx(&bar[st], bytes);
        bulk_load<false>(gstage + (size_t)st * bytes,
                         seg + p.off_out + ((int64_t)c * kChunk + i) * bytes, bytes,
                         &bar[st], pol);
    };
    const int pre = rows < STAGES ? rows : STAGES;
    if (warp == 0) {
        if (lane == 0) {
            for (int i = 0; i < STAGES; ++i) mbar_init(&bar[i], 1);
            mbar_init_fence();
#if EP_MOE_GROUP_EARLY_LOADS
            // the rows do not depend on the slots: start them first
            // (990 against 994 us on the DeepSeek-V3 shape)
            for (int i = 0; i < pre; ++i) issue(i);
#endif
        }
        __syncwarp();
        group_slots(p, r, c, n_r, seg, sm);
    }
    __syncthreads();
    if (rows == 0) return;

    if (warp == 0) {
        if (lane == 0) {
#if !EP_MOE_GROUP_EARLY_LOADS
            for (int i = 0; i < pre; ++i) issue(i);
#endif
            int issued = pre;
            bool ok = true;
            for (int i = 0; i < rows; ++i) {
                const int st = i % STAGES;
                if (!mbar_wait(&bar[st], (uint32_t)(i / STAGES) & 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const unsigned char *src = gstage + (size_t)st * bytes;
                for (int j = 0; j < p.k; ++j) {
                    const int q = sm.slot[i][j];
                    if (q >= 0 && q < p.gcap)
                        bulk_store<false>(seg + p.off_xg + (int64_t)q * bytes, src, bytes, pol);
                }
                bulk_commit();
                // the stage of row i-1: its stores were committed one group ago
                if (i >= 1 && issued < rows) {
                    bulk_wait_read1();
                    issue(issued);
                    ++issued;
                }
            }
            if (!ok) {
                set_error(p.words, EP_DEVERR_TIMEOUT);
                for (int i = 0; i < issued; ++i)   // no copy may outlive the CTA
                    mbar_wait(&bar[i % STAGES], (uint32_t)(i / STAGES) & 1u, p.timeout_ns);
            }
            bulk_wait_all();
        }
        __syncwarp();
    } else {
        for (int i = warp - 1; i < rows; i += kGroupWarps - 1)
            group_metadata(p, c * kChunk + i, i, seg, sm);
    }
}

#ifndef EP_UNGROUP_PAIRS
#define EP_UNGROUP_PAIRS 1   // scalar products summed two at a time (952 -> 940 us, DeepSeek-V3 shape)
#endif

// Weighted fp32 sum of NE grouped rows (NE > 0 known: a fixed number of
// entries, U column vectors per lane per pass) or of up to NE rows (the
// general case, `ne` at run time).  Entries are taken in ascending top-k
// slot j; the sum starts from +0 and each term is fl(w_j * y) (no FMA): a
// scalar round-to-nearest product, added with add.rn.f32x2 (each half the
// scalar round-to-nearest add).
template <int NE, int U, bool EXACT>
__device__ __forceinline__ void ungroup_row(uint32_t em, int q, float w, const char *ybase,
                                            uint4 *out, int nvec, int lane) {
    const char *rows[NE];
    float ws[NE];
    int ne = 0;
#pragma unroll
    for (int i = 0; i < NE; ++i) {
        rows[i] = nullptr;
        ws[i] = 0.f;
        if (em) {
            const int j = __ffs(em) - 1;
            em &= em - 1u;
            const int qq = __shfl_sync(0xffffffffu, q, j);
            ws[i] = __shfl_sync(0xffffffffu, w, j);
            rows[i] = ybase + (int64_t)qq * nvec * 16;
            ne = i + 1;
        }
    }
    if (EXACT) ne = NE;
    for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
        uint4 val[U][NE];
#pragma unroll
        for (int i = 0; i < NE; ++i)
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (i < ne && v0 + 32 * u < nvec)
                    val[u][i] = ld_stream16(rows[i] + (int64_t)(v0 + 32 * u) * 16);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 32 * u;
            if (v >= nvec) continue;
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
            for (int i = 0; i < NE; ++i) {
                if (i < ne) {
                    const uint32_t wd[4] = {val[u][i].x, val[u][i].y, val[u][i].z, val[u][i].w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
#if EP_UNGROUP_PAIRS
                        // scalar round-to-nearest products, summed two at a time
                        const float2 r = add2_rn(
                            make_float2(acc[2 * h], acc[2 * h + 1]),
                            make_float2(__fmul_rn(ws[i], __uint_as_float(wd[h] << 16)),
                                        __fmul_rn(ws[i], __uint_as_float(wd[h] & 0xffff0000u))));
                        acc[2 * h] = r.x;
                        acc[2 * h + 1] = r.y;
#else
                        acc[2 * h] = __fadd_rn(acc[2 * h],
                                               __fmul_rn(ws[i], __uint_as_float(wd[h] << 16)));
                        acc[2 * h + 1] = __fadd_rn(
                            acc[2 * h + 1], __fmul_rn(ws[i], __uint_as_float(wd[h] & 0xffff0000u)));
#endif
                    }
                }
            }
            uint32_t pk[4];
#pragma unroll
            for (int h = 0; h < 4; ++h)
                pk[h] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * h])) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * h + 1])) << 16);
            st_stream16(out + v, make_uint4(pk[0], pk[1], pk[2], pk[3]));
        }
    }
}

// One warp per received row.  A row usually holds few entries (k over the
// number of distinct destination ranks: ~1.5 for top-8 of 256 experts on 8
// ranks), so the common counts get their own unrolled bodies with more
// column vectors per lane: about 16 loads of 16 bytes in flight per lane
// whatever the count.
template <int MAXE, int U>
__global__ void __launch_bounds__(kMoeWarps * 32) moe_ungroup_kernel(const MoeParams p,
                                                                     const char *yg,
                                                                     int64_t yg_stride) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kMoeWarps + (threadIdx.x >> 5);
    if (gw >= (int64_t)p.W * p.cap) return;
    const int r = (int)(gw / p.cap);
    const int row = (int)(gw - (int64_t)r * p.cap);
    if (row >= rank_rows(p, r)) return;
    const char *seg = p.seg0 + (int64_t)r * p.seg_stride;
    int q = -1;
    float w = 0.f;
    if (lane < p.k) {
        q = reinterpret_cast<const int32_t *>(seg + p.off_eslot)[(int64_t)row * p.k + lane];
        w = reinterpret_cast<const float *>(seg + p.off_w)[(int64_t)row * p.k + lane];
    }
    const uint32_t em = __ballot_sync(0xffffffffu, q >= 0 && q < p.gcap);
    const int nvec = p.H / 8;
    const char *ybase = yg + (int64_t)r * yg_stride;
    uint4 *out = reinterpret_cast<uint4 *>(const_cast<char *>(seg) + p.off_comb) + (int64_t)row * nvec;
    switch (__popc(em)) {
    case 1: ungroup_row<1, 16, true>(em, q, w, ybase, out, nvec, lane); break;
    case 2: ungroup_row<2, 8, true>(em, q, w, ybase, out, nvec, lane); break;
    case 3: ungroup_row<3, 5, true>(em, q, w, ybase, out, nvec, lane); break;
    case 4: ungroup_row<4, 4, true>(em, q, w, ybase, out, nvec, lane); break;
    default: ungroup_row<MAXE, U, false>(em, q, w, ybase, out, nvec, lane); break;
    }
}

MoeParams make_params(const Config &c, const Workspace &ws) {
    MoeParams p;
    p.seg0 = ws.seg0;
    p.seg_stride = ws.seg_stride;
    p.off_out = ws.off_out;
    p.off_scales = ws.off_scales;
    p.off_w = ws.off_w;
    p.off_idx = ws.off_idx;
    p.off_xg = ws.off_xg;
    p.off_xgs = ws.off_xgs;
    p.off_gsrc = ws.off_gsrc;
    p.off_gw = ws.off_gw;
    p.off_eslot = ws.off_eslot;
    p.off_comb = ws.off_comb;
    p.totals = ws.group_base + (int64_t)c.Q * c.W;
    p.cnt = ws.moe_cnt;
    p.base = ws.moe_base;
    p.count = ws.moe_count;
    p.offset = ws.moe_offset;
    p.words = ws.words;
    p.W = c.W; p.E = c.E; p.Er = c.Er; p.k = c.k; p.H = c.H; p.cap = c.cap;
    p.gcap = c.gcap; p.nrc = c.nrc; p.nb = c.nb;
    p.row_bytes = c.fp8 ? c.H : c.H * 2;
    p.timeout_ns = c.timeout_ns;
    return p;
}

}  // namespace

cudaError_t launch_moe_group(const Config &c, const Workspace &ws, cudaStream_t st) {
    const MoeParams p = make_params(c, ws);
    const int chunks = c.W * c.nrc;
    moe_count_kernel<<<(chunks + kMoeWarps - 1) / kMoeWarps, kMoeWarps * 32, 0, st>>>(p);
    const int seqs = c.W * c.Er;
    moe_scan_kernel<<<(seqs + kMoeWarps - 1) / kMoeWarps, kMoeWarps * 32, 0, st>>>(p);
#if EP_MOE_GROUP_BULK_STAGES > 0
    const size_t dyn = (size_t)EP_MOE_GROUP_BULK_STAGES * p.row_bytes;
    if (dyn <= 160 * 1024) {
        constexpr int kMaxDevices = 64;     // function attributes are per device
        static std::atomic<size_t> configured[kMaxDevices];   // launches may race
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        if (dyn > configured[dev].load(std::memory_order_acquire)) {
            // never lower the attribute under a concurrent launch that needs more
            static std::mutex mu;
            std::lock_guard<std::mutex> lock(mu);
            if (dyn > configured[dev].load(std::memory_order_relaxed)) {
                e = cudaFuncSetAttribute(moe_group_bulk_kernel<EP_MOE_GROUP_BULK_STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
                if (e != cudaSuccess) return e;
                configured[dev].store(dyn, std::memory_order_release);
            }
        }
        moe_group_bulk_kernel<EP_MOE_GROUP_BULK_STAGES><<<chunks, kGroupWarps * 32, dyn, st>>>(p);
        return cudaGetLastError();
    }
#endif
    moe_group_kernel<<<chunks, kGroupWarps * 32, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_moe_ungroup(const Config &c, const Workspace &ws, const char *yg,
                               int64_t yg_stride, cudaStream_t st) {
    const MoeParams p = make_params(c, ws);
    const int64_t rows = (int64_t)c.W * c.cap;
    const int blocks = (int)((rows + kMoeWarps - 1) / kMoeWarps);
    if (c.k <= 2) moe_ungroup_kernel<2, 4><<<blocks, kMoeWarps * 32, 0, st>>>(p, yg, yg_stride);
    else if (c.k <= 4) moe_ungroup_kernel<4, 4><<<blocks, kMoeWarps * 32, 0, st>>>(p, yg, yg_stride);
    else if (c.k <= 8) moe_ungroup_kernel<8, 2><<<blocks, kMoeWarps * 32, 0, st>>>(p, yg, yg_stride);
    else if (c.k <= 16) moe_ungroup_kernel<16, 1><<<blocks, kMoeWarps * 32, 0, st>>>(p, yg, yg_stride);
    else moe_ungroup_kernel<32, 1><<<blocks, kMoeWarps * 32, 0, st>>>(p, yg, yg_stride);
    return cudaGetLastError();
}

}  // namespace ep
