/*
 * CPU oracle for MoE token layout, dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and
 * the CPU-baseline leg of the benchmark may load this file's library.  The
 * product path (the CUDA library and its Python binding) never calls it.
 *
 * Plain, slow, scalar C11.  Every function follows the definition of the
 * operation it computes, step by step, with no blocking, fusion or
 * reordering.  It shares no code, header or constant table with the CUDA
 * path.  Floating point: the method fixes fp32 (FP8 scale, quotient,
 * identity-expert product, combine accumulation) and bf16 (payload, combine
 * output); the oracle computes exactly those fp32 operations in the stated
 * order.  Build with -ffp-contract=off so that no product and sum are fused.
 *
 * Source: ROCm MORI documentation, "Communication APIs" page, section
 * "MORI-EP (Expert Parallelism)", table "EpDispatchCombineOp methods":
 *   dispatch(input, weights, scales, indices)
 *       -> (output, weights, scales, indices, recv_count)
 *   combine(input, weights, indices) -> (output, weights)
 *   get_dispatch_src_token_pos()
 * and "Choosing an EP API and backend", "EPv2 configuration and lifecycle"
 * (FP8 is OCP E4M3 on gfx950) and "Validation before tuning" (the
 * identity-expert correctness check).
 *
 * Notation: W ranks, E experts, Er = E/W experts per rank, k = top-k,
 * T = max tokens per rank, n_s = tokens present on source rank s (<= T),
 * H = hidden size, cap = receive rows per rank.
 * D(s,t) = { idx[s][t][j] / Er : j < k } (a set; duplicates collapse).
 *
 * Readings the pages leave open (taken as stated here):
 *  - receive order on rank r is (source rank, then source token) ascending;
 *  - src_pos of a received row is s*T + t;
 *  - combine is an unweighted fp32 sum over r in D(s,t), r ascending,
 *    started from +0.0f and rounded once to bf16; the returned weights are
 *    the same ordered sum over the expert-side weight rows;
 *  - carried weights / indices are all k entries, unchanged;
 *  - FP8: per 128-element block a = max|x|, scale = fl(a/448),
 *    q = E4M3_RNE_SATFINITE(fl(x/scale)); an all-zero block has scale 0 and
 *    all codes 0x00; the sign of a zero code is kept otherwise;
 *  - rows whose slot is >= cap are dropped by dispatch and skipped by
 *    combine.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define OR_OK 0
#define OR_EINVAL 1

/* ---------------------------------------------------------------- scalars */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 -> fp32 is exact: the bf16 pattern is the upper half of the fp32. */
float or_bf16_to_f32(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

/* fp32 -> bf16, round to nearest, ties to even (IEEE-754 roundTiesToEven).
 * The kept part is the upper 16 bits; the discarded lower 16 bits decide:
 * above one half ulp round up, below round down, exactly one half round to
 * the even kept pattern.  A carry out of the mantissa moves to the next
 * binade (or to infinity), which is the correct rounded value.  Inputs are
 * finite in this method. */
uint16_t or_bf16_rne(float f)
{
    uint32_t u = bits_from_f32(f);
    uint32_t kept = u >> 16;
    uint32_t rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double y)
{
    double f = floor(y);
    double d = y - f;
    if (d > 0.5) return f + 1.0;
    if (d < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* OCP 8-bit floating point, E4M3 ("fn"): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits.  Exponent field 0 holds subnormals m * 2^-9;
 * fields 1..15 hold (1 + m/8) * 2^(e-7); S.1111.111 is NaN, so the largest
 * finite magnitude is 1.75 * 2^8 = 448 (code 0x7E); there is no infinity.
 * Encoding: round to nearest, ties to even mantissa; "satfinite" clamps
 * magnitudes that round beyond 448 to 448.  The sign bit is always kept
 * (so a negative value that rounds to zero gives 0x80).
 *
 * Codes are monotone in magnitude: with quantum 2^-9 below 2^-6 and
 * 2^(e-3) in binade [2^e, 2^(e+1)), the code of n quanta is n in the
 * subnormal range and (e+6)*8 + n in binade e (n in [8,16]); n = 16 lands
 * on the first code of the next binade, which is the right rounding carry. */
uint8_t or_e4m3_encode(float v)
{
    uint8_t sign = (bits_from_f32(v) >> 31) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (isnan(v)) return (uint8_t)(sign | 0x7F);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int code;
    if (a < ldexp(1.0, -6)) {
        code = (int)round_half_even(a / ldexp(1.0, -9));      /* 0..8 */
    } else {
        int e2;
        frexp(a, &e2);            /* a = m * 2^e2, m in [0.5, 1) */
        int e = e2 - 1;           /* a in [2^e, 2^(e+1)), e in [-6, 8] */
        int n = (int)round_half_even(a / ldexp(1.0, e - 3));  /* 8..16 */
        code = (e + 6) * 8 + n;
    }
    if (code > 0x7E) code = 0x7E;  /* satfinite (a < 448 never exceeds it) */
    return (uint8_t)(sign | code);
}

/* Value of an E4M3 code (exact in fp32). */
float or_e4m3_value(uint8_t q)
{
    int s = q >> 7, e = (q >> 3) & 0xF, m = q & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return (float)(s ? -v : v);
}

/* One quantisation block of n bf16 values (n = 128 in this method):
 * a = max |x_i| (exact), scale = fl32(a / 448), codes q_i =
 * E4M3(fl32(x_i / scale)); a == 0 gives scale 0 and codes 0x00. */
void or_quant_block(const uint16_t *x, int n, uint8_t *q, float *scale)
{
    float a = 0.0f;
    for (int i = 0; i < n; ++i) {
        float v = fabsf(or_bf16_to_f32(x[i]));
        if (v > a) a = v;
    }
    if (a == 0.0f) {
        *scale = 0.0f;
        for (int i = 0; i < n; ++i) q[i] = 0x00;
        return;
    }
    float s = a / 448.0f;
    *scale = s;
    for (int i = 0; i < n; ++i) {
        float v = or_bf16_to_f32(x[i]) / s;
        q[i] = or_e4m3_encode(v);
    }
}

/* Element-wise forms of the scalars above, for testing over many values. */
void or_bf16_rne_array(const float *v, uint16_t *o, int64_t n)
{ for (int64_t i = 0; i < n; ++i) o[i] = or_bf16_rne(v[i]); }
void or_e4m3_encode_array(const float *v, uint8_t *o, int64_t n)
{ for (int64_t i = 0; i < n; ++i) o[i] = or_e4m3_encode(v[i]); }
void or_e4m3_value_array(const uint8_t *q, float *o, int64_t n)
{ for (int64_t i = 0; i < n; ++i) o[i] = or_e4m3_value(q[i]); }
void or_quant_rows(const uint16_t *x, int64_t rows, int H, uint8_t *q, float *scales)
{
    for (int64_t i = 0; i < rows; ++i)
        for (int b = 0; b < H / 128; ++b)
            or_quant_block(x + i * H + b * 128, 128, q + i * H + b * 128,
                           scales + i * (H / 128) + b);
}

/* ------------------------------------------------------------- validation */

int or_validate(int W, int E, int k, int T, int H, int fp8,
                const int32_t *idx, const int32_t *num_tokens)
{
    if (W < 1 || W > 64 || E < 1 || k < 1 || T < 0 || H < 1) return OR_EINVAL;
    if (E % W != 0) return OR_EINVAL;
    if (H % 8 != 0) return OR_EINVAL;
    if (fp8 && H % 128 != 0) return OR_EINVAL;
    for (int s = 0; s < W; ++s) {
        if (num_tokens[s] < 0 || num_tokens[s] > T) return OR_EINVAL;
        for (int t = 0; t < num_tokens[s]; ++t)
            for (int j = 0; j < k; ++j) {
                int32_t e = idx[((int64_t)s * T + t) * k + j];
                if (e < 0 || e >= E) return OR_EINVAL;
            }
    }
    return OR_OK;
}

/* ----------------------------------------------------------------- layout */

/* Routing layout of one batch.
 *   in_D[s][t][r]  = 1 iff r in D(s,t) and t < n_s
 *   C[s][r]        = #{t < n_s : r in D(s,t)}            (send counts)
 *   recv_count[r]  = sum_s C[s][r]
 *   pos[s][t][r]   = sum_{s'<s} C[s'][r] + #{t' < t : r in D(s,t')}
 *                    if r in D(s,t), else -1
 * pos is int32 [W][T][W]; C is int32 [W][W]; recv_count int32 [W].
 * in_D is caller scratch, uint8 [W][T][W]. */
int or_layout(int W, int E, int k, int T, const int32_t *idx,
              const int32_t *num_tokens, uint8_t *in_D,
              int32_t *pos, int32_t *C, int32_t *recv_count)
{
    int Er = E / W;
    memset(in_D, 0, (size_t)W * T * W);
    for (int s = 0; s < W; ++s)
        for (int t = 0; t < num_tokens[s]; ++t)
            for (int j = 0; j < k; ++j) {
                int r = idx[((int64_t)s * T + t) * k + j] / Er;
                in_D[((int64_t)s * T + t) * W + r] = 1;
            }
    for (int s = 0; s < W; ++s)
        for (int r = 0; r < W; ++r) {
            int32_t c = 0;
            for (int t = 0; t < T; ++t) c += in_D[((int64_t)s * T + t) * W + r];
            C[s * W + r] = c;
        }
    for (int r = 0; r < W; ++r) {
        int32_t tot = 0;
        for (int s = 0; s < W; ++s) tot += C[s * W + r];
        recv_count[r] = tot;
    }
    for (int s = 0; s < W; ++s)
        for (int r = 0; r < W; ++r) {
            int32_t base = 0;
            for (int sp = 0; sp < s; ++sp) base += C[sp * W + r];
            int32_t before = 0;   /* #{t' < t : r in D(s,t')} */
            for (int t = 0; t < T; ++t) {
                int64_t o = ((int64_t)s * T + t) * W + r;
                if (in_D[o]) { pos[o] = base + before; before += 1; }
                else pos[o] = -1;
            }
        }
    return OR_OK;
}

/* --------------------------------------------------------------- dispatch */

/* Dispatch, given the layout.  For every source token (s,t) with t < n_s and
 * every r in D(s,t) with p = pos[s][t][r] < cap, row p of rank r receives:
 *   out[r][p]        = x[s][t]                (bf16 bits), or the FP8 codes
 *   out_scales[r][p] = the H/128 block scales (FP8 only)
 *   out_w[r][p]      = w[s][t][0..k)
 *   out_idx[r][p]    = idx[s][t][0..k)
 *   src_pos[r][p]    = s*T + t
 * Outputs are dense [W][cap][...]; rows never written are left as they are.
 * out is uint16 [W][cap][H] for bf16, uint8 [W][cap][H] for FP8; with
 * out == NULL only the per-row metadata (scales excepted) is produced. */
/* Dispatch of the source tokens g = s*T + t with g0 <= g < g1 (t < n_s):
 * each goes to row pos[s][t][r] of every r in D(s,t).  Tokens are
 * independent, so disjoint ranges may run on different threads; the whole
 * method is the range [0, W*T). */
int or_dispatch_range(int W, int k, int T, int H, int cap, int fp8,
                      const uint16_t *x, const float *w, const int32_t *idx,
                      const int32_t *num_tokens, const int32_t *pos,
                      void *out, float *out_scales, float *out_w,
                      int32_t *out_idx, int32_t *src_pos, int64_t g0, int64_t g1)
{
    int nb = fp8 ? H / 128 : 0;
    for (int64_t g = g0; g < g1; ++g) {
        int s = (int)(g / T), t = (int)(g % T);
        if (t >= num_tokens[s]) continue;
        const uint16_t *row = x + ((int64_t)s * T + t) * H;
        for (int r = 0; r < W; ++r) {
            int32_t p = pos[((int64_t)s * T + t) * W + r];
            if (p < 0 || p >= cap) continue;
            int64_t rp = (int64_t)r * cap + p;
            if (!out) {
                /* metadata only */
            } else if (fp8) {
                uint8_t *o = (uint8_t *)out + rp * H;
                for (int b = 0; b < nb; ++b)
                    or_quant_block(row + b * 128, 128, o + b * 128,
                                   out_scales + rp * nb + b);
            } else {
                uint16_t *o = (uint16_t *)out + rp * H;
                for (int h = 0; h < H; ++h) o[h] = row[h];
            }
            for (int j = 0; j < k; ++j) {
                out_w[rp * k + j] = w[((int64_t)s * T + t) * k + j];
                out_idx[rp * k + j] = idx[((int64_t)s * T + t) * k + j];
            }
            src_pos[rp] = s * T + t;
        }
    }
    return OR_OK;
}

int or_dispatch(int W, int k, int T, int H, int cap, int fp8,
                const uint16_t *x, const float *w, const int32_t *idx,
                const int32_t *num_tokens, const int32_t *pos,
                void *out, float *out_scales, float *out_w,
                int32_t *out_idx, int32_t *src_pos)
{
    return or_dispatch_range(W, k, T, H, cap, fp8, x, w, idx, num_tokens, pos,
                             out, out_scales, out_w, out_idx, src_pos,
                             0, (int64_t)W * T);
}

int or_dispatch_rows(int W, int k, int T, int H, int fp8,
                     const uint16_t *x, const float *w, const int32_t *idx,
                     const int32_t *num_tokens, const int32_t *pos,
                     const int32_t *ranks, const int32_t *slots, int n,
                     void *out_rows, float *scale_rows, float *w_rows,
                     int32_t *idx_rows, int32_t *src_rows)
{
    int nb = fp8 ? H / 128 : 0;
    for (int i = 0; i < n; ++i) {
        int r = ranks[i], found = 0;
        for (int s = 0; s < W && !found; ++s)
            for (int t = 0; t < num_tokens[s] && !found; ++t) {
                if (pos[((int64_t)s * T + t) * W + r] != slots[i]) continue;
                found = 1;
                const uint16_t *row = x + ((int64_t)s * T + t) * H;
                if (fp8) {
                    for (int b = 0; b < nb; ++b)
                        or_quant_block(row + b * 128, 128,
                                       (uint8_t *)out_rows + (int64_t)i * H + b * 128,
                                       scale_rows + (int64_t)i * nb + b);
                } else {
                    for (int h = 0; h < H; ++h)
                        ((uint16_t *)out_rows)[(int64_t)i * H + h] = row[h];
                }
                for (int j = 0; j < k; ++j) {
                    w_rows[(int64_t)i * k + j] = w[((int64_t)s * T + t) * k + j];
                    idx_rows[(int64_t)i * k + j] = idx[((int64_t)s * T + t) * k + j];
                }
                src_rows[i] = s * T + t;
            }
        if (!found) return OR_EINVAL;
    }
    return OR_OK;
}

/* ------------------------------------------------------- identity expert */

/* The identity expert of the benchmark's correctness check, for one row
 * received on rank r:
 *   alpha = +0.0f, then alpha = fl32(alpha + w[j]) for the j in ascending
 *           order whose expert idx[j] lives on rank r;
 *   v_h   = the bf16 payload as fp32, or fl32(value(q_h) * scale of its
 *           block) for FP8;
 *   y[h]  = bf16_rne(fl32(v_h * alpha)). */
static void identity_row(int r, int Er, int k, int H, int fp8,
                         const void *payload, const float *scales,
                         const float *w, const int32_t *idx, uint16_t *y)
{
    float alpha = 0.0f;
    for (int j = 0; j < k; ++j)
        if (idx[j] / Er == r)
            alpha = alpha + w[j];
    for (int h = 0; h < H; ++h) {
        float v;
        if (fp8)
            v = or_e4m3_value(((const uint8_t *)payload)[h]) * scales[h / 128];
        else
            v = or_bf16_to_f32(((const uint16_t *)payload)[h]);
        float prod = v * alpha;
        y[h] = or_bf16_rne(prod);
    }
}

/* Identity expert over whole receive buffers: every received row
 * p < min(recv_count[r], cap) of every rank r.  y is uint16 [W][cap][H]. */
/* Identity expert over the receive rows i = r*cap + p with i0 <= i < i1
 * (p < min(recv_count[r], cap)); rows are independent. */
int or_identity_expert_range(int W, int E, int k, int H, int cap, int fp8,
                             const int32_t *recv_count, const void *payload,
                             const float *scales, const float *out_w,
                             const int32_t *out_idx, uint16_t *y,
                             int64_t i0, int64_t i1)
{
    int Er = E / W;
    int nb = fp8 ? H / 128 : 0;
    for (int64_t rp = i0; rp < i1; ++rp) {
        int r = (int)(rp / cap), p = (int)(rp % cap);
        int n = recv_count[r] < cap ? recv_count[r] : cap;
        if (p >= n) continue;
        const void *row = fp8 ? (const void *)((const uint8_t *)payload + rp * H)
                              : (const void *)((const uint16_t *)payload + rp * H);
        identity_row(r, Er, k, H, fp8, row, fp8 ? scales + rp * nb : 0,
                     out_w + rp * k, out_idx + rp * k, y + rp * H);
    }
    return OR_OK;
}

int or_identity_expert(int W, int E, int k, int H, int cap, int fp8,
                       const int32_t *recv_count, const void *payload,
                       const float *scales, const float *out_w,
                       const int32_t *out_idx, uint16_t *y)
{
    return or_identity_expert_range(W, E, k, H, cap, fp8, recv_count, payload,
                                    scales, out_w, out_idx, y, 0, (int64_t)W * cap);
}

int or_identity_rows(int W, int E, int k, int H, int fp8, const int32_t *ranks,
                     int n, const void *payload, const float *scales,
                     const float *w, const int32_t *idx, uint16_t *y)
{
    int Er = E / W;
    int nb = fp8 ? H / 128 : 0;
    for (int i = 0; i < n; ++i) {
        const void *row = fp8 ? (const void *)((const uint8_t *)payload + (int64_t)i * H)
                              : (const void *)((const uint16_t *)payload + (int64_t)i * H);
        identity_row(ranks[i], Er, k, H, fp8, row, fp8 ? scales + (int64_t)i * nb : 0,
                     w + (int64_t)i * k, idx + (int64_t)i * k, y + (int64_t)i * H);
    }
    return OR_OK;
}

/* ---------------------------------------------------------------- combine */

/* The combine sum of one token from its rows in ascending rank order:
 *   acc_h = +0.0f; acc_h = fl32(acc_h + fp32(rows[i][h])) for i = 0..nd-1;
 *   out_h = bf16_rne(acc_h). */
static void sum_rows(int nd, const uint16_t *const *rows, int H, uint16_t *out)
{
    for (int h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int i = 0; i < nd; ++i)
            acc = acc + or_bf16_to_f32(rows[i][h]);
        out[h] = or_bf16_rne(acc);
    }
}

/* Combine of one source token (s,t), given the layout: its rows are
 * y[r][pos[s][t][r]] for r = 0..W-1 ascending with the slot in [0, cap);
 * out_row = sum_rows of them and, if w_in is given, out_w_row[j] = the same
 * ordered fp32 sum of w_in[r][p][j] (no rounding at the end).  y is uint16
 * [W][cap][H], w_in float [W][cap][k]. */
static void combine_token(int W, int k, int T, int H, int cap, int s, int t,
                          const int32_t *pos, const uint16_t *y,
                          const float *w_in, uint16_t *out_row, float *out_w_row)
{
    const uint16_t *rows[64];
    int nd = 0;
    for (int r = 0; r < W; ++r) {
        int32_t p = pos[((int64_t)s * T + t) * W + r];
        if (p < 0 || p >= cap) continue;
        rows[nd++] = y + ((int64_t)r * cap + p) * H;
    }
    sum_rows(nd, rows, H, out_row);
    if (w_in && out_w_row) {
        for (int j = 0; j < k; ++j) {
            float acc = 0.0f;
            for (int r = 0; r < W; ++r) {
                int32_t p = pos[((int64_t)s * T + t) * W + r];
                if (p < 0 || p >= cap) continue;
                acc = acc + w_in[((int64_t)r * cap + p) * k + j];
            }
            out_w_row[j] = acc;
        }
    }
}

/* Combine of one token whose nd rows (ascending rank order) are given
 * gathered: rows [nd][H] -> out [H]. */
int or_combine_gathered(int nd, int H, const uint16_t *rows, uint16_t *out)
{
    const uint16_t *ptrs[64];
    if (nd < 0 || nd > 64) return OR_EINVAL;
    for (int i = 0; i < nd; ++i) ptrs[i] = rows + (int64_t)i * H;
    sum_rows(nd, ptrs, H, out);
    return OR_OK;
}

/* Combine of every present token: out uint16 [W][T][H], out_w float
 * [W][T][k] (nullable with w_in).  Rows t >= n_s are left as they are. */
/* Combine of the source tokens g = s*T + t with g0 <= g < g1 (t < n_s);
 * tokens are independent. */
int or_combine_range(int W, int k, int T, int H, int cap, const int32_t *num_tokens,
                     const int32_t *pos, const uint16_t *y, const float *w_in,
                     uint16_t *out, float *out_w, int64_t g0, int64_t g1)
{
    for (int64_t g = g0; g < g1; ++g) {
        int s = (int)(g / T), t = (int)(g % T);
        if (t >= num_tokens[s]) continue;
        combine_token(W, k, T, H, cap, s, t, pos, y, w_in,
                      out + ((int64_t)s * T + t) * H,
                      out_w ? out_w + ((int64_t)s * T + t) * k : 0);
    }
    return OR_OK;
}

int or_combine(int W, int k, int T, int H, int cap, const int32_t *num_tokens,
               const int32_t *pos, const uint16_t *y, const float *w_in,
               uint16_t *out, float *out_w)
{
    return or_combine_range(W, k, T, H, cap, num_tokens, pos, y, w_in, out, out_w,
                            0, (int64_t)W * T);
}

/* ------------------------------------------- pre-quantised FP8 dispatch */

/* Dispatch of an input that is already quantised (the pages' dispatch takes
 * `scales` next to `input`; the HIP backend accepts FP8 input
 * that is quantised already): the E4M3 codes x8[s][t][0..H) and the block scales
 * sc[s][t][0..H/128) of each present token are copied unchanged to every
 * destination slot p = pos[s][t][r] < cap, with the weights, ids and
 * src_pos as in or_dispatch.  out uint8 [W][cap][H], out_scales
 * [W][cap][H/128]. */
int or_dispatch_prequant(int W, int k, int T, int H, int cap,
                         const uint8_t *x8, const float *sc, const float *w,
                         const int32_t *idx, const int32_t *num_tokens,
                         const int32_t *pos, uint8_t *out, float *out_scales,
                         float *out_w, int32_t *out_idx, int32_t *src_pos)
{
    int nb = H / 128;
    for (int s = 0; s < W; ++s)
        for (int t = 0; t < num_tokens[s]; ++t) {
            int64_t tok = (int64_t)s * T + t;
            for (int r = 0; r < W; ++r) {
                int32_t p = pos[tok * W + r];
                if (p < 0 || p >= cap) continue;
                int64_t rp = (int64_t)r * cap + p;
                for (int h = 0; h < H; ++h) out[rp * H + h] = x8[tok * H + h];
                for (int b = 0; b < nb; ++b) out_scales[rp * nb + b] = sc[tok * nb + b];
                for (int j = 0; j < k; ++j) {
                    out_w[rp * k + j] = w[tok * k + j];
                    out_idx[rp * k + j] = idx[tok * k + j];
                }
                src_pos[rp] = s * T + t;
            }
        }
    return OR_OK;
}

/* ------------------------------------------------ FP32 combine input */

/* Identity expert with an fp32 output row (the expert hands combine fp32
 * rows): y[h] = fl32(v_h * alpha), alpha and v as in identity_row, with no
 * rounding to bf16.  y is float [W][cap][H]. */
int or_identity_expert_f32(int W, int E, int k, int H, int cap, int fp8,
                           const int32_t *recv_count, const void *payload,
                           const float *scales, const float *out_w,
                           const int32_t *out_idx, float *y)
{
    int Er = E / W;
    int nb = fp8 ? H / 128 : 0;
    for (int r = 0; r < W; ++r) {
        int n = recv_count[r] < cap ? recv_count[r] : cap;
        for (int p = 0; p < n; ++p) {
            int64_t rp = (int64_t)r * cap + p;
            float alpha = 0.0f;
            for (int j = 0; j < k; ++j)
                if (out_idx[rp * k + j] / Er == r)
                    alpha = alpha + out_w[rp * k + j];
            for (int h = 0; h < H; ++h) {
                float v;
                if (fp8)
                    v = or_e4m3_value(((const uint8_t *)payload)[rp * H + h]) *
                        scales[rp * nb + h / 128];
                else
                    v = or_bf16_to_f32(((const uint16_t *)payload)[rp * H + h]);
                y[rp * H + h] = v * alpha;
            }
        }
    }
    return OR_OK;
}

/* Combine of fp32 expert rows: out[s][t][h] = bf16_rne(+0.0f + y_r0[p0][h]
 * + y_r1[p1][h] + ...) over r in D(s,t) ascending (slots < cap), each '+'
 * an fp32 add; out_w as in or_combine.  y float [W][cap][H]. */
int or_combine_f32(int W, int k, int T, int H, int cap, const int32_t *num_tokens,
                   const int32_t *pos, const float *y, const float *w_in,
                   uint16_t *out, float *out_w)
{
    for (int s = 0; s < W; ++s)
        for (int t = 0; t < num_tokens[s]; ++t) {
            int64_t tok = (int64_t)s * T + t;
            for (int h = 0; h < H; ++h) {
                float acc = 0.0f;
                for (int r = 0; r < W; ++r) {
                    int32_t p = pos[tok * W + r];
                    if (p < 0 || p >= cap) continue;
                    acc = acc + y[((int64_t)r * cap + p) * H + h];
                }
                out[tok * H + h] = or_bf16_rne(acc);
            }
            if (w_in && out_w)
                for (int j = 0; j < k; ++j) {
                    float acc = 0.0f;
                    for (int r = 0; r < W; ++r) {
                        int32_t p = pos[tok * W + r];
                        if (p < 0 || p >= cap) continue;
                        acc = acc + w_in[((int64_t)r * cap + p) * k + j];
                    }
                    out_w[tok * k + j] = acc;
                }
        }
    return OR_OK;
}

/* ------------------------------------------- standard-MoE conversion */

/* Standard-MoE grouping of one rank's received rows (the EPv2 feature list
 * of "Choosing an EP API and backend" names a "standard-MoE conversion";
 * reading: per-local-expert contiguous groups).  On rank r, with
 * n_r = min(recv_count[r], cap) received rows, the entries are the pairs
 * (p, j), p < n_r, j < k, whose expert out_idx[r][p][j] lives on r, in
 * (p, j) ascending order; e = out_idx - r*Er is the entry's local expert.
 *   count[r][e]  = number of entries of expert e
 *   offset[r][e] = sum_{e' < e} count[r][e']
 *   slot(p, j)   = offset[r][e] + #{entries of e before (p, j)}
 * entry_slot[r][p][j] = slot(p, j), or -1 for a non-local j or p >= n_r.
 * count, offset int32 [W][Er]; entry_slot int32 [W][cap][k]. */
int or_expert_layout(int W, int E, int k, int cap, const int32_t *recv_count,
                     const int32_t *out_idx, int32_t *count, int32_t *offset,
                     int32_t *entry_slot)
{
    int Er = E / W;
    for (int r = 0; r < W; ++r) {
        int n = recv_count[r] < cap ? recv_count[r] : cap;
        for (int e = 0; e < Er; ++e) count[r * Er + e] = 0;
        for (int p = 0; p < n; ++p)
            for (int j = 0; j < k; ++j) {
                int32_t g = out_idx[((int64_t)r * cap + p) * k + j];
                if (g / Er == r) count[r * Er + (g - r * Er)] += 1;
            }
        int32_t run = 0;
        for (int e = 0; e < Er; ++e) { offset[r * Er + e] = run; run += count[r * Er + e]; }
        for (int64_t o = (int64_t)r * cap * k; o < (int64_t)(r + 1) * cap * k; ++o)
            entry_slot[o] = -1;
        for (int e = 0; e < Er; ++e) {
            int32_t before = 0;   /* entries of e seen so far, in (p, j) order */
            for (int p = 0; p < n; ++p)
                for (int j = 0; j < k; ++j) {
                    int64_t o = ((int64_t)r * cap + p) * k + j;
                    int32_t g = out_idx[o];
                    if (g / Er == r && g - r * Er == e) {
                        entry_slot[o] = offset[r * Er + e] + before;
                        before += 1;
                    }
                }
        }
    }
    return OR_OK;
}

/* Grouped copy: for every entry (p, j) of rank r with q = entry_slot < gcap,
 *   xg[r][q] = out[r][p] (payload row, elem_bytes per element),
 *   xg_scales[r][q] = out_scales[r][p] (FP8 only, nb floats),
 *   g_src[r][q] = p*k + j,  g_w[r][q] = out_w[r][p][j].
 * Payload rows are H*elem_bytes bytes. */
int or_group_rows(int W, int k, int H, int elem_bytes, int nb, int cap, int gcap,
                  const int32_t *recv_count, const void *out, const float *out_scales,
                  const float *out_w, const int32_t *entry_slot, void *xg,
                  float *xg_scales, int32_t *g_src, float *g_w)
{
    int64_t rb = (int64_t)H * elem_bytes;
    for (int r = 0; r < W; ++r) {
        int n = recv_count[r] < cap ? recv_count[r] : cap;
        for (int p = 0; p < n; ++p)
            for (int j = 0; j < k; ++j) {
                int64_t o = ((int64_t)r * cap + p) * k + j;
                int32_t q = entry_slot[o];
                if (q < 0 || q >= gcap) continue;
                int64_t rq = (int64_t)r * gcap + q;
                memcpy((char *)xg + rq * rb, (const char *)out + ((int64_t)r * cap + p) * rb, rb);
                for (int b = 0; b < nb; ++b)
                    xg_scales[rq * nb + b] = out_scales[((int64_t)r * cap + p) * nb + b];
                g_src[rq] = p * k + j;
                g_w[rq] = out_w[o];
            }
    }
    return OR_OK;
}

/* Un-grouping (the standard MoE's weighted sum of a token's expert outputs
 * on one rank): for each received row p < min(recv_count[r], cap),
 *   acc = +0.0f; for j ascending with q = entry_slot[r][p][j] in [0, gcap):
 *     acc = fl32(acc + fl32(out_w[r][p][j] * fp32(yg[r][q][h])))
 *   y[r][p][h] = bf16_rne(acc).
 * yg uint16 [W][gcap][H]; y uint16 [W][cap][H]. */
int or_ungroup(int W, int k, int H, int cap, int gcap, const int32_t *recv_count,
               const float *out_w, const int32_t *entry_slot, const uint16_t *yg,
               uint16_t *y)
{
    for (int r = 0; r < W; ++r) {
        int n = recv_count[r] < cap ? recv_count[r] : cap;
        for (int p = 0; p < n; ++p)
            for (int h = 0; h < H; ++h) {
                float acc = 0.0f;
                for (int j = 0; j < k; ++j) {
                    int64_t o = ((int64_t)r * cap + p) * k + j;
                    int32_t q = entry_slot[o];
                    if (q < 0 || q >= gcap) continue;
                    float prod = out_w[o] * or_bf16_to_f32(yg[((int64_t)r * gcap + q) * H + h]);
                    acc = acc + prod;
                }
                y[((int64_t)r * cap + p) * H + h] = or_bf16_rne(acc);
            }
    }
    return OR_OK;
}

/* ---------------------------------------------- FP8 combine payload */

/* One FP8 block of n fp32 values, the dispatch formula applied to fp32
 * input: a = max |v_i|, scale = fl32(a / 448), q_i = E4M3(fl32(v_i / scale));
 * a == 0 gives scale 0 and codes 0x00. */
void or_quant_block_f32(const float *v, int n, uint8_t *q, float *scale)
{
    float a = 0.0f;
    for (int i = 0; i < n; ++i) {
        float m = fabsf(v[i]);
        if (m > a) a = m;
    }
    if (a == 0.0f) {
        *scale = 0.0f;
        for (int i = 0; i < n; ++i) q[i] = 0x00;
        return;
    }
    float s = a / 448.0f;
    *scale = s;
    for (int i = 0; i < n; ++i) q[i] = or_e4m3_encode(v[i] / s);
}

/* Identity expert writing an FP8 combine payload: the fp32 product
 * fl32(v_h * alpha) of or_identity_expert_f32, quantised per 128-element
 * block with or_quant_block_f32.  yq uint8 [W][cap][H], ysc [W][cap][H/128].
 * Rows past min(recv_count, cap) are left as they are. */
int or_identity_expert_fp8(int W, int E, int k, int H, int cap, int fp8,
                           const int32_t *recv_count, const void *payload,
                           const float *scales, const float *out_w,
                           const int32_t *out_idx, float *tmp_row,
                           uint8_t *yq, float *ysc)
{
    int Er = E / W;
    int nb_in = fp8 ? H / 128 : 0;
    int nb = H / 128;
    for (int r = 0; r < W; ++r) {
        int n = recv_count[r] < cap ? recv_count[r] : cap;
        for (int p = 0; p < n; ++p) {
            int64_t rp = (int64_t)r * cap + p;
            float alpha = 0.0f;
            for (int j = 0; j < k; ++j)
                if (out_idx[rp * k + j] / Er == r)
                    alpha = alpha + out_w[rp * k + j];
            for (int h = 0; h < H; ++h) {
                float v;
                if (fp8)
                    v = or_e4m3_value(((const uint8_t *)payload)[rp * H + h]) *
                        scales[rp * nb_in + h / 128];
                else
                    v = or_bf16_to_f32(((const uint16_t *)payload)[rp * H + h]);
                tmp_row[h] = v * alpha;
            }
            for (int b = 0; b < nb; ++b)
                or_quant_block_f32(tmp_row + b * 128, 128, yq + rp * H + b * 128,
                                   ysc + rp * nb + b);
        }
    }
    return OR_OK;
}

/* Combine of an FP8 expert payload: out[s][t][h] = bf16_rne(+0.0f +
 * sum over r in D(s,t) ascending of fl32(value(yq[r][p][h]) * ysc[r][p][h/128])),
 * each product and '+' an fp32 operation; out_w as in or_combine. */
int or_combine_fp8(int W, int k, int T, int H, int cap, const int32_t *num_tokens,
                   const int32_t *pos, const uint8_t *yq, const float *ysc,
                   const float *w_in, uint16_t *out, float *out_w)
{
    int nb = H / 128;
    for (int s = 0; s < W; ++s)
        for (int t = 0; t < num_tokens[s]; ++t) {
            int64_t tok = (int64_t)s * T + t;
            for (int h = 0; h < H; ++h) {
                float acc = 0.0f;
                for (int r = 0; r < W; ++r) {
                    int32_t p = pos[tok * W + r];
                    if (p < 0 || p >= cap) continue;
                    int64_t rp = (int64_t)r * cap + p;
                    float v = or_e4m3_value(yq[rp * H + h]) * ysc[rp * nb + h / 128];
                    acc = acc + v;
                }
                out[tok * H + h] = or_bf16_rne(acc);
            }
            if (w_in && out_w)
                for (int j = 0; j < k; ++j) {
                    float acc = 0.0f;
                    for (int r = 0; r < W; ++r) {
                        int32_t p = pos[tok * W + r];
                        if (p < 0 || p >= cap) continue;
                        acc = acc + w_in[((int64_t)r * cap + p) * k + j];
                    }
                    out_w[tok * k + j] = acc;
                }
        }
    return OR_OK;
}
