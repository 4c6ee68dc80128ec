/*
 * ep_api.h -- C ABI of the GB300 (sm_103a) MoE expert-parallel token
 * layout / dispatch / combine library (libep_gb300.so).
 *
 * What it computes follows the ROCm MORI documentation, "Communication APIs"
 * page, section "MORI-EP (Expert Parallelism)", table "EpDispatchCombineOp
 * methods":
 *   dispatch(input, weights, scales, indices)
 *       -> (output, weights, scales, indices, recv_count)   sends each token
 *          to the ranks that hold its experts
 *   combine(input, weights, indices) -> (output, weights)    brings the
 *          experts' results back to the source tokens
 *   dispatch_send()/dispatch_recv(), combine_send()/combine_recv()  split
 *          phases for overlapping independent work
 *   reset(), get_dispatch_src_token_pos(),
 *   get_registered_combine_input_buffer(dtype)
 * and the "AsyncLL v2 SDMA overlap" section of the same page (send posts the
 * payload, then a ready notification; receive waits, then data and counts
 * are ready on the stream; zero-token peers notify too; the receive step
 * writes the count, zero included; options are frozen at construction).
 *
 * Model.  All W logical EP ranks live in ONE GPU's HBM.  The caller passes
 * one device workspace; the library carves it into a layout-state region and
 * W identical per-rank segments (the symmetric-heap analogue).  A "send" to
 * rank r is a store into segment r.  There is no collective.
 *
 * Notation: W ranks (1..32), E experts (multiple of W), Er = E/W, k = top-k
 * (1..32), T = max tokens per source rank, n_s = tokens present on source
 * rank s in this call (0..T), H = hidden size, cap = receive rows per rank.
 * D(s,t) = { idx[s][t][j] / Er : j < k } is the set of distinct destination
 * ranks of token t on rank s; duplicate experts collapse.
 *
 * Results:
 *  - layout: C[s][r] = #{t < n_s : r in D(s,t)}; recv_count[r] = sum_s
 *    C[s][r]; rows on rank r are ordered by (source rank, source token);
 *    pos[s][t][r] = sum_{s'<s} C[s'][r] + #{t' < t : r in D(s,t')} when
 *    r in D(s,t), else -1.  Deterministic; no atomics decide any position.
 *  - dispatch: row p = pos[s][t][r] of rank r receives x[s][t] (bf16 bits,
 *    or FP8 E4M3 codes plus one fp32 scale per 128 elements with
 *    scale = fl32(amax/448) and q = RNE-satfinite(fl32(x/scale)); an
 *    all-zero block gives scale 0 and codes 0x00; the quantised input is
 *    taken to be finite: a block holding an infinity or a NaN gets an
 *    unspecified scale and codes), all k weights and all k expert ids
 *    unchanged, and src_pos = s*T + t.
 *  - combine: out[s][t] = bf16_rne( fp32 sum over r in D(s,t), r ascending,
 *    starting from +0.0f, of y_r[pos[s][t][r]] ); out_w the same ordered
 *    fp32 sum of the expert-side weight rows.  No weighting is applied.
 *
 * Conventions.
 *  - Pointers named d_* are device pointers, h_* host pointers.  Streams are
 *    cudaStream_t passed as void* (NULL = the legacy default stream).
 *  - Every call after ep_create is asynchronous on the given stream and
 *    allocates nothing (ep_create takes one pinned host word for
 *    ep_get_error).  ep_get_error synchronises the stream it is given.
 *  - Device-side problems (an expert id outside [0,E), a rank receiving more
 *    than cap rows, a wait that timed out, combine indices that differ from
 *    the dispatch's) set bits of a sticky device error word; the kernels skip
 *    the offending entry or row, never write out of bounds and never trap.
 *  - Host-detectable problems return a status at once and launch nothing.
 *
 * Status codes: the first eight mirror the StatusCode enum of the same
 * page's MORI-IO section (SUCCESS, INIT, IN_PROGRESS, ERR_INVALID_ARGS,
 * ERR_NOT_FOUND, ERR_RDMA_OP, ERR_BAD_STATE, ERR_GPU_OP), the only error
 * convention the pages give; EP_ERR_RDMA_OP is never returned here.
 */
#ifndef EP_API_H
#define EP_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EP_SUCCESS = 0,
    EP_INIT = 1,
    EP_IN_PROGRESS = 2,
    EP_ERR_INVALID_ARGS = 3,
    EP_ERR_NOT_FOUND = 4,
    EP_ERR_RDMA_OP = 5,       /* reserved: no RDMA on one GPU */
    EP_ERR_BAD_STATE = 6,     /* call out of order (recv w/o send, ...) */
    EP_ERR_GPU_OP = 7,        /* a CUDA runtime call failed */
    EP_ERR_TIMEOUT = 8,       /* a bounded device wait gave up */
    EP_ERR_CAPACITY = 9,      /* a rank would receive more than cap rows */
    EP_ERR_BAD_INDEX = 10     /* an expert id outside [0, E) */
} ep_status_t;

/* Bits of the device error word (ep_get_error). */
#define EP_DEVERR_BAD_INDEX        0x1u
#define EP_DEVERR_CAPACITY         0x2u
#define EP_DEVERR_TIMEOUT          0x4u
#define EP_DEVERR_COMBINE_MISMATCH 0x8u

typedef enum {
    EP_DT_BF16 = 0,
    EP_DT_FP8_E4M3 = 1,       /* OCP E4M3 ("fn"), max 448 */
    EP_DT_FP32 = 2
} ep_dtype_t;

#define EP_MAX_WORLD 32
#define EP_MAX_TOPK 32
#define EP_QUANT_BLOCK 128

/* Op configuration (the EpDispatchCombineConfig analogue).  Frozen into the
 * handle by ep_create; ops with different options coexist. */
typedef struct {
    int32_t world_size;               /* W, 1..32 */
    int32_t num_experts;              /* E, multiple of W */
    int32_t topk;                     /* k, 1..32 */
    int32_t hidden;                   /* H, multiple of 8 (of 128 for FP8),
                                         8..2^24 (16384 at most for the fused
                                         FP8 dispatch) */
    int32_t max_tokens_per_rank;      /* T >= 1 */
    int32_t max_recv_tokens_per_rank; /* cap; 0 selects W*T (exact worst case) */
    int32_t dispatch_dtype;           /* EP_DT_BF16, or EP_DT_FP8_E4M3 for the
                                         fused per-128-element quantisation */
    int32_t early_notify;             /* 1: the send phase posts per-(source,
                                         destination) ready flags after its
                                         payload, zero-token pairs included;
                                         the receive phase checks them */
    int32_t fused_recv;               /* 1 (needs early_notify): combine's
                                         gather kernel does the receive wait
                                         itself, one warp per CTA, then a CTA
                                         barrier releases the gather warps */
    int32_t combine_dtype;            /* element type of the expert rows that
                                         combine reads: EP_DT_BF16 (0),
                                         EP_DT_FP32, or EP_DT_FP8_E4M3 (codes
                                         + one fp32 scale per 128 elements,
                                         registered buffer only; H % 128 == 0);
                                         the output is bf16 */
    int64_t wait_timeout_ns;          /* bound of every device wait; 0 = 1 s */
    int32_t max_grouped_rows_per_rank;/* rows of the standard-MoE grouped
                                         buffers per rank (0: no grouping);
                                         cap * k is the exact worst case */
    int32_t combine_mode;             /* EP_COMBINE_GATHER (0): combine_recv
                                         gathers the expert rows from the
                                         destination segments.
                                         EP_COMBINE_SCATTER: combine_send pushes
                                         every received row's expert output to a
                                         per-token staging area on the source
                                         side (slot = the rank's order among the
                                         token's destinations) and combine_recv
                                         reduces the staged rows; bf16 rows from
                                         the registered buffer only */
} ep_config_t;

#define EP_COMBINE_GATHER 0
#define EP_COMBINE_SCATTER 1

/* A handle is not thread-safe: drive it from one host thread at a time. */
typedef struct ep_handle ep_handle_t;

/* Device views of the dispatch results (valid until the next dispatch,
 * reset or destroy).  Every per-rank buffer of rank r starts at
 * base + r * rank_stride_bytes; rows hold H payload elements (bf16 or u8),
 * H/128 scales, k weights, k expert ids, one src_pos. */
typedef struct {
    void     *out;            /* [W] x [cap][H]  bf16 or e4m3 codes */
    float    *out_scales;     /* [W] x [cap][H/128]; NULL unless FP8 */
    float    *out_w;          /* [W] x [cap][k] */
    int32_t  *out_idx;        /* [W] x [cap][k] global expert ids */
    int32_t  *src_pos;        /* [W] x [cap]   s*T + t */
    int64_t   rank_stride_bytes;
    int32_t  *recv_count;     /* [W], written by the receive step */
    int32_t  *send_counts;    /* [W][W], C[s][r] */
    int32_t  *pos;            /* [W][T][W], -1 where r is not in D(s,t) */
    uint32_t *dispatch_flags; /* [W dst][W src] ready epochs (early_notify) */
    uint32_t *combine_flags;  /* [W src][W dst] ready epochs (early_notify) */
    uint32_t  dispatch_epoch; /* value the flags carry for the last send */
    uint32_t  combine_epoch;
    int32_t   cap;
    int32_t   max_dest;       /* min(W, k) */
    void     *combine_stage;  /* scatter combine: [W][T][max_dest][H] bf16, or NULL */
} ep_dispatch_out_t;

const char *ep_status_str(ep_status_t s);

/* Bytes of device workspace ep_create needs for this config.
 * INVALID_ARGS if the config is outside the limits above. */
ep_status_t ep_workspace_size(const ep_config_t *cfg, size_t *bytes);

/* Validate cfg, carve d_workspace (>= ep_workspace_size bytes, 256-byte
 * aligned, owned by the caller and kept alive until ep_destroy), zero the
 * flags, counters and error word (synchronously), take one pinned host word
 * (cudaHostAlloc) for ep_get_error, and return a host handle.
 * Reads EP_EARLY_NOTIFY / EP_FUSED_RECV / EP_LOG_LEVEL from the environment
 * once, here.  Must be called with the workspace's device current. */
ep_status_t ep_create(const ep_config_t *cfg, void *d_workspace, size_t bytes,
                      ep_handle_t **out);

/* Free the host handle and its CUDA events (not the workspace). */
ep_status_t ep_destroy(ep_handle_t *h);

/* Layout only (step "routing layout"): from d_idx int32 [W][T][k] and the
 * per-call token counts h_num_tokens int32 [W] (host), compute per-token
 * destination masks, the W x W send counts, recv_count and the chunk bases
 * that fix every position.  Sets BAD_INDEX / CAPACITY device bits. */
ep_status_t ep_layout(ep_handle_t *h, const int32_t *d_idx,
                      const int32_t *h_num_tokens, void *stream);

/* Send phase of dispatch: layout, then the copy of every token row to each
 * of its destination ranks (with its k weights, k ids and src_pos), then
 * (early_notify) the ready flags.  d_w: [W][T][k] fp32; d_idx: [W][T][k]
 * int32.  d_x and d_scales, 16-byte aligned:
 *  - d_scales == NULL: d_x is [W][T][H] bf16; with an FP8 dispatch_dtype
 *    every row is quantised on the way (fused per-128-element E4M3);
 *  - d_scales != NULL (FP8 dispatch_dtype only; the pages' dispatch takes
 *    `scales` beside `input`, and a backend may pass FP8 input that is
 *    quantised already): d_x is [W][T][H] E4M3 codes and d_scales [W][T][H/128]
 *    fp32 block scales, both copied unchanged.
 * Inputs must stay unchanged until the receive phase has been enqueued.
 * The copy kernel is launched as a programmatic dependent of the layout
 * kernel just before it (both enqueued by this call), so stream capture
 * records a programmatic edge between them.  When the routing spans at most
 * 8 chunks of 32 tokens (W * ceil(T/32) <= 8), no layout kernel runs: the
 * copy computes the layout itself and is launched as a programmatic
 * dependent of whatever kernel precedes it.  Either way anything enqueued
 * earlier on the stream is complete before the first read of the inputs. */
ep_status_t ep_dispatch_send(ep_handle_t *h, const void *d_x, const float *d_w,
                             const float *d_scales, const int32_t *d_idx,
                             const int32_t *h_num_tokens, void *stream);

/* Receive phase of dispatch on `stream` (may differ from the send stream):
 * wait for the send (stream-ordered via an event the send recorded); with
 * early_notify, check the ready flags (bounded wait, TIMEOUT bit on expiry)
 * and then write recv_count (zero included).  Without early_notify the
 * send's layout kernel has produced recv_count and this phase launches no
 * kernel.  Either way the received rows and recv_count are ready on
 * `stream` once this call's work there is done.  BAD_STATE without a
 * pending send. */
ep_status_t ep_dispatch_recv(ep_handle_t *h, void *stream);

/* Send + receive on one stream. */
ep_status_t ep_dispatch(ep_handle_t *h, const void *d_x, const float *d_w,
                        const float *d_scales, const int32_t *d_idx,
                        const int32_t *h_num_tokens, void *stream);

/* Routing replay: the copy (and notify) of ep_dispatch_send, reusing the
 * layout of the last ep_layout / ep_dispatch_send call for the same indices
 * and token counts, without recomputing it.  d_x / d_scales as in
 * ep_dispatch_send; h_num_tokens must equal the layout's.  BAD_STATE
 * without a layout. */
ep_status_t ep_dispatch_send_replay(ep_handle_t *h, const void *d_x,
                                    const float *d_w, const float *d_scales,
                                    const int32_t *d_idx,
                                    const int32_t *h_num_tokens, void *stream);

ep_status_t ep_dispatch_outputs(const ep_handle_t *h, ep_dispatch_out_t *out);

/* The pre-registered combine input buffer of rank 0 (the expert writes
 * y_r rows here; rank r's rows start at *d_ptr + r * *rank_stride_bytes).
 * dtype must be the config's combine_dtype (else EP_ERR_NOT_FOUND). */
ep_status_t ep_get_combine_input_buffer(const ep_handle_t *h, int32_t dtype,
                                        void **d_ptr,
                                        int64_t *rank_stride_bytes);

/* FP8 combine payload (combine_dtype == EP_DT_FP8_E4M3): the block scales
 * of the registered combine buffer, rank r's [cap][H/128] fp32 rows at
 * *d_ptr + r * *rank_stride_bytes.  Combine dequantises each element as
 * fl32(e4m3_value(q) * scale) before its ordered fp32 sum.  NOT_FOUND for
 * other combine dtypes. */
ep_status_t ep_get_combine_input_scales(const ep_handle_t *h, float **d_ptr,
                                        int64_t *rank_stride_bytes);

/* Send phase of combine (expert side): records the completion of the
 * expert's work on `stream` and (early_notify) posts combine ready flags.
 * BAD_STATE without a dispatch, while a dispatch send waits for its receive
 * phase (the receive orders the expert side after the send's copy), or while
 * an earlier combine send waits for its receive. */
ep_status_t ep_combine_send(ep_handle_t *h, void *stream);

/* Receive phase of combine (source side): wait for the combine send, then
 * gather-reduce.  d_y: NULL for the registered buffer, else rank r's rows at
 * d_y + r*y_rank_stride_bytes ([cap][H] of combine_dtype, 16-byte aligned).
 * d_w_in: NULL, or rank r's expert-side weight rows [cap][k] fp32 at
 * d_w_in + r*w_rank_stride_bytes.  d_idx: NULL, or the [W][T][k] ids of the
 * dispatch (checked: a token whose destination set differs sets the
 * COMBINE_MISMATCH bit; the dispatch's layout is used).  d_out: [W][T][H]
 * bf16; d_out_w: [W][T][k] fp32 (written iff d_w_in).  Rows t >= n_s are
 * not written.  BAD_STATE without a dispatch or without a combine send.
 * The gather kernel is launched as a programmatic dependent of the kernel
 * before it on the stream and waits for that kernel's completion before
 * its first read, so it may be enqueued right after the expert's kernel. */
ep_status_t ep_combine_recv(ep_handle_t *h, const void *d_y,
                            int64_t y_rank_stride_bytes, const float *d_w_in,
                            int64_t w_rank_stride_bytes, const int32_t *d_idx,
                            void *d_out, float *d_out_w, void *stream);

/* Send + receive on one stream.  BAD_STATE without a dispatch, while a
 * dispatch send waits for its receive phase, or while a combine send waits
 * for its receive. */
ep_status_t ep_combine(ep_handle_t *h, const void *d_y,
                       int64_t y_rank_stride_bytes, const float *d_w_in,
                       int64_t w_rank_stride_bytes, const int32_t *d_idx,
                       void *d_out, float *d_out_w, void *stream);

/* Standard-MoE conversion ("Choosing an EP API and backend", EPv2 row:
 * "standard-MoE conversion"), needs max_grouped_rows_per_rank > 0.
 * After the receive phase of a dispatch, on every rank r the entries
 * (received row p < min(recv_count[r], cap), top-k slot j) whose expert
 * lives on r are grouped per local expert e = idx - r*Er: groups in e order,
 * entries in (p, j) order inside a group.  count[r][e], offset[r][e] (its
 * exclusive prefix) and entry_slot[r][p][j] (-1 if non-local) describe it;
 * slot q of rank r gets the payload row (and FP8 scale row), g_src = p*k + j
 * and g_w = the row's weight j.  Entries whose slot is >= the grouped
 * capacity are dropped and set the CAPACITY bit. */
typedef struct {
    void     *xg;             /* [W] x [gcap][H] payload (bf16 or e4m3) */
    float    *xg_scales;      /* [W] x [gcap][H/128] (FP8) or NULL */
    int32_t  *g_src;          /* [W] x [gcap] p*k + j */
    float    *g_w;            /* [W] x [gcap] routing weight of the entry */
    void     *yg;             /* [W] x [gcap][H] bf16: registered expert-output rows */
    int32_t  *entry_slot;     /* [W] x [cap][k] */
    int64_t   rank_stride_bytes;
    int32_t  *count;          /* [W][Er] */
    int32_t  *offset;         /* [W][Er] */
    int32_t   gcap;
    int32_t   experts_per_rank;
} ep_moe_out_t;

ep_status_t ep_moe_group(ep_handle_t *h, void *stream);
ep_status_t ep_moe_outputs(const ep_handle_t *h, ep_moe_out_t *out);

/* The inverse before combine: for every received row p of rank r,
 * y_r[p][h] = bf16_rne(+0.0f + sum over its entries j ascending of
 * fl32(g_w * fp32(yg[slot][h]))) written to the registered combine input
 * buffer (combine_dtype must be bf16).  d_yg: NULL for the registered
 * expert-output buffer, else rank r's [gcap][H] bf16 rows at
 * d_yg + r*yg_rank_stride_bytes.  BAD_STATE without a grouping. */
ep_status_t ep_moe_ungroup(ep_handle_t *h, const void *d_yg,
                           int64_t yg_rank_stride_bytes, void *stream);

/* Reset between iterations: zero the ready flags, epochs and error word on
 * `stream` and forget the layout (combine then needs a new dispatch). */
ep_status_t ep_reset(ep_handle_t *h, void *stream);

/* Read and clear the device error word in `stream` order (one atomic
 * exchange on the device, so no bit set concurrently is lost), then wait for
 * that stream alone (cudaStreamSynchronize; work on other streams keeps
 * running, and what it sets later shows in a later call).  *mask gets the
 * EP_DEVERR_* bits; the return is EP_SUCCESS for 0, else the status of the
 * lowest set bit (BAD_INDEX, CAPACITY, TIMEOUT, BAD_STATE for a combine
 * mismatch). */
ep_status_t ep_get_error(ep_handle_t *h, uint32_t *mask, void *stream);

/* Test harness, not part of the hot path: the identity expert of the
 * benchmark's correctness check ("Validation before tuning").  For each
 * received row p < min(recv_count[r], cap) of every rank r:
 * alpha = ordered fp32 sum of the row's weights whose expert lives on r,
 * y_r[p][h] = bf16_rne(fl32(v_h * alpha)) (fp32 rows: fl32(v_h * alpha);
 * FP8 payload: those fp32 products quantised per 128-element block with the
 * dispatch formula),
 * v = the bf16 payload, or fl32(e4m3_value(q) * scale) for FP8.  d_y as in
 * ep_combine_recv. */
ep_status_t ep_test_identity_expert(ep_handle_t *h, void *d_y,
                                    int64_t y_rank_stride_bytes, void *stream);

/* Test harness, not part of the hot path: checks the arithmetic behind the
 * fused FP8 quantisation of dispatch (per 128-element block a = max|x|,
 * scale = fl32(a/448), q = RNE-satfinite(fl32(x/scale)); OCP E4M3, "Choosing
 * an EP API and backend", "EPv2 configuration and lifecycle") over every
 * positive finite bf16 block maximum a and every finite bf16 x with
 * |x| <= a, both signs (1 065 402 238 pairs), using the dispatch kernel's
 * own device functions.  d_counts: 4 device uint64 (8-byte aligned), zeroed
 * here, then [0] = pairs checked, [1] = pairs whose E4M3 code differs from
 * the code of the IEEE quotient x / (a / 448), [2] = block maxima whose scale
 * differs from the IEEE quotient a / 448, [3] = pairs that took the
 * reciprocal-and-correction quotient.  Asynchronous on `stream`. */
ep_status_t ep_test_fp8_quotient_check(uint64_t *d_counts, void *stream);

/* Routing layout without any allocation, for callers that cannot allocate
 * device memory or pass a workspace: code living inside another
 * framework's memory pool that only sees raw tensor pointers, and serving
 * paths that forbid cudaMalloc (it can synchronise the device and can fail
 * under memory pressure).  The pages have no counterpart of this call; it
 * computes the same layout as ep_layout + ep_dispatch (pos, send counts,
 * recv_count) with no handle.
 *   d_idx [W][T][k] int32, h_num_tokens [W] host; outputs (caller-owned,
 *   device): d_pos [W][T][W] (-1 where r is not a destination),
 *   d_send_counts [W][W], d_recv_count [W]; d_error: NULL or a device u32
 *   that gets EP_DEVERR_BAD_INDEX OR-ed in (out-of-range ids contribute no
 *   destination).
 * Scratch is a fixed device array inside the library (about 0.66 MB, held
 * by every GPU that loads the library until the process exits); it limits
 * the layout to W <= 32 and W * ceil(T/32) <= 4128 32-token chunks: any
 * W * T <= 131072 is accepted whatever T is, and up to 132096 tokens when T
 * is a multiple of 32.  Larger sizes return EP_ERR_INVALID_ARGS.  Every call
 * looks the array's device address up with the caller's device current (a
 * host-side lookup once the library's device code is loaded, so a context
 * reset in between is harmless); the first call on a device may load that
 * code, so make it before any stream capture.  All calls share the array:
 * calls whose work overlaps on the GPU race; order them on one stream. */
ep_status_t ep_layout_noalloc(int32_t world_size, int32_t num_experts,
                              int32_t topk, int32_t max_tokens_per_rank,
                              const int32_t *d_idx, const int32_t *h_num_tokens,
                              int32_t *d_pos, int32_t *d_send_counts,
                              int32_t *d_recv_count, uint32_t *d_error,
                              void *stream);

#ifdef __cplusplus
}
#endif
#endif /* EP_API_H */
