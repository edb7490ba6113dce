/*
 * CPU oracle for the routed multi-tenant LoRA delta.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It is the plain,
 * slow, obviously correct statement of what the GPU path computes, and it
 * shares no code, header or helper with that path.
 *
 * Each function states the page and section it follows:
 *   [punica]    "vllm/lora/punica_wrapper/punica_base.py" (Punica wrapper base)
 *   [sharded]   "vllm.lora.fully_sharded_layers" (S-LoRA fully sharded layers)
 *   [metrale]   "Module lora_delta" (metrale_model_layers::layers::ops)
 *   [flashinfer]"flashinfer.fused_moe.bgmv_moe_gemm1_lora_delta"
 *
 * Precision (the readings that the pages leave open):
 *   - bf16 values travel as their 16-bit patterns (uint16_t).
 *   - acc64 == 0: products and sums in fp32, k ascending then r ascending,
 *     the intermediate h kept in fp32 (the [sharded] shrink buffer is a
 *     float32 tensor); the fold v = scale * d in fp32; the output is
 *     RN_bf16(f32(out) + v), i.e. one fp32 add then one round-to-nearest-even.
 *   - acc64 == 1: the same steps with every intermediate in fp64 and a single
 *     rounding of (out + v) from fp64 to bf16.  Used to bound the fp32
 *     variant from above in the tests.
 * Compiled with -ffp-contract=off so that no multiply-add is fused.
 *
 * Device-style error word: bit 1 = a routing slot >= max_loras (row skipped),
 * bit 2 = an MoE expert id outside [0, E) (pair written as zeros), bit 4 =
 * an MoE adapter id >= num_loras (pair written as zeros).  Host-style return
 * value: 0 on success, 1 on a bad argument.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_ERR_SLOT 1u
#define ORACLE_ERR_EXPERT 2u
#define ORACLE_ERR_LORA 4u

/* ------------------------------------------------------------------ */
/* bf16 <-> float, from the IEEE-754 binary16-brain layout: the upper   */
/* 16 bits of an IEEE binary32.                                         */
/* ------------------------------------------------------------------ */

float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest, ties to even, of a binary32 to its upper 16 bits. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN, sign kept */
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u; /* carries into the exponent when the mantissa overflows */
    return (uint16_t)upper;
}

/* Round-to-nearest-even of a binary64 straight to bf16 (one rounding). */
uint16_t oracle_f64_to_bf16(double v)
{
    if (isnan(v))
        return 0x7fc0u;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7f80u);
    /* bf16 has 8 significant bits; its smallest normal is 2^-126 and its
     * subnormal quantum is 2^-133. */
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    double q;
    int qexp;
    if (e - 1 < -126) {
        q = nearbyint(ldexp(a, 133)); /* subnormal: fixed quantum 2^-133 */
        qexp = -133;
    } else {
        q = nearbyint(ldexp(m, 8)); /* 8 significant bits, ties to even */
        qexp = e - 8;
    }
    double r = ldexp(q, qexp);
    if (r > 0x1.fep127)
        return (uint16_t)(sign | 0x7f80u); /* rounded past the largest bf16 */
    float rf = (float)r;                 /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* ------------------------------------------------------------------ */
/* Scale rule.  [metrale] LoraPair: scale = lora_alpha / r, or          */
/* lora_alpha / sqrt(r) with use_rslora; applied in the fold, never     */
/* folded into B.                                                       */
/* ------------------------------------------------------------------ */
float oracle_lora_scale(float alpha, int r, int use_rslora)
{
    if (r <= 0)
        return 0.0f;
    return use_rslora ? (float)((double)alpha / sqrt((double)r))
                      : (float)((double)alpha / (double)r);
}

/* ------------------------------------------------------------------ */
/* Pool packing.  [metrale] module invariants + LoraPair: the pool is    */
/* zeroed before packing; a: [max_rank, k_in] row-major with the PEFT    */
/* lora_A [r, k_in] in its first r rows and zero rows after; b:          */
/* [n_out, max_rank] row-major with the PEFT lora_B [n_out, r] in the    */
/* first r columns of each row and zero columns after.                   */
/* ------------------------------------------------------------------ */
int oracle_pool_pack(uint16_t *a_slot, uint16_t *b_slot, const uint16_t *a_r,
                     const uint16_t *b_r, int r, int R, int k_in, int w)
{
    if (r < 0 || r > R || k_in < 0 || w < 0)
        return 1;
    for (int q = 0; q < R; ++q)
        for (int k = 0; k < k_in; ++k)
            a_slot[(size_t)q * k_in + k] = (q < r) ? a_r[(size_t)q * k_in + k] : 0;
    for (int c = 0; c < w; ++c)
        for (int q = 0; q < R; ++q)
            b_slot[(size_t)c * R + q] = (q < r) ? b_r[(size_t)c * r + q] : 0;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Routing metadata.  [punica] prefill_metadata: the batch clustered by  */
/* identical lora index, with per-cluster start and length; an index of  */
/* -1 applies no LoRA.  Reading: clusters in ascending slot order, rows  */
/* of a cluster in ascending original index (a stable sort by slot);     */
/* rows with slot < 0 or slot >= max_loras belong to no cluster.         */
/* perm[0 .. seg_start[max_loras]) lists the clustered rows;             */
/* cluster s is perm[seg_start[s] .. seg_start[s+1]).                    */
/* ------------------------------------------------------------------ */
int oracle_segments(const int32_t *seq_slot, int n, int max_loras, int32_t *perm,
                    int32_t *seg_start, uint32_t *err)
{
    if (n < 0 || max_loras <= 0)
        return 1;
    int pos = 0;
    for (int s = 0; s < max_loras; ++s) {
        seg_start[s] = pos;
        for (int i = 0; i < n; ++i)
            if (seq_slot[i] == s)
                perm[pos++] = i;
    }
    seg_start[max_loras] = pos;
    for (int i = 0; i < n; ++i)
        if (seq_slot[i] >= max_loras && err)
            *err |= ORACLE_ERR_SLOT;
    return 0;
}

/* Slot of row i, or -1 when the row gets no delta (flagging bad slots). */
static int row_slot(const int32_t *seq_slot, int i, int max_loras, uint32_t *err)
{
    int s = seq_slot[i];
    if (s < 0)
        return -1;
    if (s >= max_loras) {
        if (err) {
#pragma omp atomic
            *err |= ORACLE_ERR_SLOT;
        }
        return -1;
    }
    return s;
}

/* ------------------------------------------------------------------ */
/* Shrink.  [punica] add_shrink "Semantics": for every slice i,          */
/* y[i] += (x @ lora_a_stacked[i]) * scale, routed per row.  With the    */
/* [metrale] LoraPair layout a = [max_rank, k_in] this is               */
/* h[j][i][q] += scale_s * sum_k x[i,k] * A_j,s[q,k] over the padded     */
/* rank q < R.  a_table[j*max_loras + s] is the slot's A (NULL = the     */
/* slot does not adapt slice j, [metrale] LoraRoute).  scale_table NULL  */
/* means scale 1 (the [sharded] layers pass 1.0 here).  Rows with no    */
/* slot and slices with no adapter are left untouched.                  */
/* ------------------------------------------------------------------ */
int oracle_shrink(float *h, const uint16_t *x, int n, int k_in, const int32_t *seq_slot,
                  const uint16_t *const *a_table, const float *scale_table, int S, int R,
                  int max_loras, int acc64, uint32_t *err)
{
    if (n < 0 || k_in < 0 || S < 0 || R < 0 || max_loras <= 0)
        return 1;
#pragma omp parallel for schedule(dynamic, 4)
    for (int i = 0; i < n; ++i) {
        int s = row_slot(seq_slot, i, max_loras, err);
        if (s < 0)
            continue;
        float scale = scale_table ? scale_table[s] : 1.0f;
        for (int j = 0; j < S; ++j) {
            const uint16_t *A = a_table[(size_t)j * max_loras + s];
            if (!A)
                continue;
            float *hrow = h + ((size_t)j * n + i) * R;
            for (int q = 0; q < R; ++q) {
                const uint16_t *arow = A + (size_t)q * k_in;
                const uint16_t *xrow = x + (size_t)i * k_in;
                if (acc64) {
                    double acc = 0.0;
                    for (int k = 0; k < k_in; ++k)
                        acc += (double)oracle_bf16_to_f32(xrow[k]) *
                               (double)oracle_bf16_to_f32(arow[k]);
                    hrow[q] = (float)((double)hrow[q] + acc * (double)scale);
                } else {
                    float acc = 0.0f;
                    for (int k = 0; k < k_in; ++k)
                        acc += oracle_bf16_to_f32(xrow[k]) * oracle_bf16_to_f32(arow[k]);
                    hrow[q] = hrow[q] + acc * scale;
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Expand.  [punica] add_expand "Semantics": offset = offset_start; for  */
/* each slice i: y[:, offset:offset+slice] += x[i] @ lora_b_stacked[i];  */
/* offset += slice.  With b = [n_out, max_rank] ([metrale] LoraPair):    */
/* d = sum_q h[j][i][q] * B_j,s[c,q]; v = scale_s * d ("applied in the  */
/* fold", scale_table NULL means 1); out = RN_bf16(out + v), or RN_bf16(v)*/
/* when add_inputs is 0.  Rows with no slot and slices whose b_table     */
/* entry is NULL are left untouched bit for bit.                        */
/* ------------------------------------------------------------------ */
int oracle_expand(uint16_t *out, int64_t ld_out, const float *h, const int32_t *seq_slot,
                  const uint16_t *const *b_table, const float *scale_table,
                  const int *widths, int S, int R, int n, int max_loras, int offset_start,
                  int add_inputs, uint32_t *err)
{
    if (n < 0 || S < 0 || R < 0 || max_loras <= 0 || offset_start < 0)
        return 1;
#pragma omp parallel for schedule(dynamic, 4)
    for (int i = 0; i < n; ++i) {
        int s = row_slot(seq_slot, i, max_loras, err);
        if (s < 0)
            continue;
        float scale = scale_table ? scale_table[s] : 1.0f;
        int64_t off = offset_start;
        for (int j = 0; j < S; ++j) {
            const uint16_t *B = b_table[(size_t)j * max_loras + s];
            if (B) {
                const float *hrow = h + ((size_t)j * n + i) * R;
                for (int c = 0; c < widths[j]; ++c) {
                    float d = 0.0f;
                    for (int q = 0; q < R; ++q)
                        d += hrow[q] * oracle_bf16_to_f32(B[(size_t)c * R + q]);
                    float v = scale * d;
                    uint16_t *o = out + (size_t)i * ld_out + off + c;
                    *o = oracle_f32_to_bf16(add_inputs ? oracle_bf16_to_f32(*o) + v : v);
                }
            }
            off += widths[j];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* The routed delta in one call.  [punica] add_lora_linear "Semantics"  */
/* (y[i] += x[i] @ A[indices[i]] @ B[indices[i]] * scale, per slice)    */
/* and [metrale] apply_lora_bgmv (out[i,:] += scale_s * (x[i,:] @ A_s^T) */
/* @ B_s^T with s = seq_slot[i]; a negative slot gets no delta).  Both   */
/* stages contract at the padded rank R ([metrale] invariants).  A slice */
/* applies only when both its A and B table entries are set.            */
/* ------------------------------------------------------------------ */
int oracle_delta(uint16_t *out, int64_t ld_out, const uint16_t *x, int n, int k_in,
                 const int32_t *seq_slot, const uint16_t *const *a_table,
                 const uint16_t *const *b_table, const float *scale_table, const int *widths,
                 int S, int R, int max_loras, int offset_start, int add_inputs, int acc64,
                 uint32_t *err)
{
    if (n < 0 || k_in < 0 || S < 0 || R < 0 || R > 512 || max_loras <= 0 || offset_start < 0)
        return 1;
#pragma omp parallel for schedule(dynamic, 2)
    for (int i = 0; i < n; ++i) {
        int s = row_slot(seq_slot, i, max_loras, err);
        if (s < 0)
            continue;
        float scale = scale_table ? scale_table[s] : 1.0f;
        const uint16_t *xrow = x + (size_t)i * k_in;
        int64_t off = offset_start;
        for (int j = 0; j < S; ++j) {
            const uint16_t *A = a_table[(size_t)j * max_loras + s];
            const uint16_t *B = b_table[(size_t)j * max_loras + s];
            if (A && B) {
                float hf[512];
                double hd[512];
                for (int q = 0; q < R; ++q) {
                    const uint16_t *arow = A + (size_t)q * k_in;
                    if (acc64) {
                        double acc = 0.0;
                        for (int k = 0; k < k_in; ++k)
                            acc += (double)oracle_bf16_to_f32(xrow[k]) *
                                   (double)oracle_bf16_to_f32(arow[k]);
                        hd[q] = acc;
                    } else {
                        float acc = 0.0f;
                        for (int k = 0; k < k_in; ++k)
                            acc += oracle_bf16_to_f32(xrow[k]) * oracle_bf16_to_f32(arow[k]);
                        hf[q] = acc;
                    }
                }
                for (int c = 0; c < widths[j]; ++c) {
                    uint16_t *o = out + (size_t)i * ld_out + off + c;
                    const uint16_t *brow = B + (size_t)c * R;
                    if (acc64) {
                        double d = 0.0;
                        for (int q = 0; q < R; ++q)
                            d += hd[q] * (double)oracle_bf16_to_f32(brow[q]);
                        double v = (double)scale * d;
                        *o = oracle_f64_to_bf16(add_inputs ? (double)oracle_bf16_to_f32(*o) + v
                                                           : v);
                    } else {
                        float d = 0.0f;
                        for (int q = 0; q < R; ++q)
                            d += hf[q] * oracle_bf16_to_f32(brow[q]);
                        float v = scale * d;
                        *o = oracle_f32_to_bf16(add_inputs ? oracle_bf16_to_f32(*o) + v : v);
                    }
                }
            }
            off += widths[j];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Routed-MoE FC1 delta.  [flashinfer] bgmv_moe_gemm1_lora_delta: for   */
/* each (token t, slot j), e = topk_ids[t, j], l = lora_ids[t] (skipped  */
/* when l < 0):                                                          */
/*   delta[t, j] = scale * concat(B_gate[l,e] @ (A_gate[l,e] @ x[t]),    */
/*                                B_up[l,e]   @ (A_up[l,e]   @ x[t]))    */
/* unweighted, per (token, slot).  Regular mode: w_ptr_a/w_ptr_b are     */
/* [2, E] tables of [A_gate, A_up] / [B_gate, B_up] bank bases; shared   */
/* mode (shared_a != 0): [E] tables, one shared A and B fused as         */
/* [2I, rank] (gate rows 0:I, up rows I:2I), delta = scale * B_fused @   */
/* (A_shared @ x[t]).  Adapter l of a bank starts l * stride elements    */
/* after the bank base.  Readings: A[l,e] is [rank, H] row-major, B is    */
/* [I, rank] (or [2I, rank]) row-major; the output [T, top_k, 2I] is     */
/* freshly written, so a skipped pair (l < 0, l >= num_loras, or e       */
/* outside [0, E)) is written as +0.                                     */
/* ------------------------------------------------------------------ */
int oracle_moe_fc1(uint16_t *out, const uint16_t *x, const uint16_t *const *w_ptr_a,
                   int64_t stride_a, const uint16_t *const *w_ptr_b, int64_t stride_b,
                   int shared_a, const int32_t *topk_ids, const int32_t *lora_ids, int T,
                   int top_k, int E, int H, int I, int rank, int num_loras, float scale,
                   int acc64, uint32_t *err)
{
    if (T < 0 || top_k < 0 || E <= 0 || H < 0 || I < 0 || rank < 0 || rank > 512)
        return 1;
    const int n_slices = shared_a ? 1 : 2;
    const int width = shared_a ? 2 * I : I;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t p = 0; p < (int64_t)T * top_k; ++p) {
        int t = (int)(p / top_k);
        int e = topk_ids[p];
        int l = lora_ids[t];
        uint16_t *orow = out + (size_t)p * 2 * I;
        int skip = 0;
        if (l < 0) {
            skip = 1;
        } else if (l >= num_loras) {
            skip = 1;
            if (err) {
#pragma omp atomic
                *err |= ORACLE_ERR_LORA;
            }
        } else if (e < 0 || e >= E) {
            skip = 1;
            if (err) {
#pragma omp atomic
                *err |= ORACLE_ERR_EXPERT;
            }
        }
        if (skip) {
            for (int c = 0; c < 2 * I; ++c)
                orow[c] = 0;
            continue;
        }
        const uint16_t *xrow = x + (size_t)t * H;
        for (int j = 0; j < n_slices; ++j) {
            const uint16_t *A = w_ptr_a[(size_t)j * E + e] + (size_t)l * stride_a;
            const uint16_t *B = w_ptr_b[(size_t)j * E + e] + (size_t)l * stride_b;
            float hf[512];
            double hd[512];
            for (int q = 0; q < rank; ++q) {
                const uint16_t *arow = A + (size_t)q * H;
                if (acc64) {
                    double acc = 0.0;
                    for (int k = 0; k < H; ++k)
                        acc += (double)oracle_bf16_to_f32(xrow[k]) *
                               (double)oracle_bf16_to_f32(arow[k]);
                    hd[q] = acc;
                } else {
                    float acc = 0.0f;
                    for (int k = 0; k < H; ++k)
                        acc += oracle_bf16_to_f32(xrow[k]) * oracle_bf16_to_f32(arow[k]);
                    hf[q] = acc;
                }
            }
            for (int c = 0; c < width; ++c) {
                const uint16_t *brow = B + (size_t)c * rank;
                uint16_t *o = orow + (size_t)j * I + c;
                if (acc64) {
                    double d = 0.0;
                    for (int q = 0; q < rank; ++q)
                        d += hd[q] * (double)oracle_bf16_to_f32(brow[q]);
                    *o = oracle_f64_to_bf16((double)scale * d);
                } else {
                    float d = 0.0f;
                    for (int q = 0; q < rank; ++q)
                        d += hf[q] * oracle_bf16_to_f32(brow[q]);
                    *o = oracle_f32_to_bf16(scale * d);
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* In-place MoE LoRA around the two expert GEMMs.  [punica] add_lora_w13 */
/* adds the gate/up delta to y = intermediate_cache1 [T, top_k, 2I] in   */
/* place, before the activation; add_lora_w2 adds the down delta to      */
/* y = intermediate_cache3 [T, top_k, H] in place, before moe_sum, from  */
/* x = intermediate_cache2 [T * top_k, I], one input row per (token,     */
/* slot).  Per pair the delta is the [flashinfer] one:                   */
/*   w13: scale * concat(B_gate @ (A_gate @ x[t]), B_up @ (A_up @ x[t])) */
/*        or scale * B_fused @ (A_shared @ x[t]);                        */
/*   w2:  scale * B_down @ (A_down @ x[t * top_k + j]), A_down [rank, I], */
/*        B_down [H, rank].                                              */
/* Readings (the page gives signatures and docstrings only):             */
/*   - the pair's adapter is lora_ids[t] (the token-to-adapter mapping); */
/*     l < 0, or adapter_enabled[l] == 0 when that table is given, means */
/*     no delta; l >= num_loras is an error (no delta, bit 4);           */
/*   - expert_map, when given, maps a global expert id in [0, n_global)  */
/*     to this rank's local id, -1 = not on this rank (no delta); a      */
/*     global id outside the map or a local id outside [0, E) is an      */
/*     error (no delta, bit 2);                                          */
/*   - y is the caller's buffer: a pair with no delta is left untouched; */
/*   - add_inputs: y = RN(f32(y) + v), else y = RN(v), on pairs with a   */
/*     delta;                                                            */
/*   - w2 with topk_weights: v = w[t, j] * (scale * d), the routing       */
/*     weight that the down GEMM applied before moe_sum; without them    */
/*     v = scale * d.                                                    */
/* ------------------------------------------------------------------ */

/* The (adapter, local expert) of pair p; 0 when the pair gets no delta. */
static int moe_pair_key(int64_t p, int top_k, const int32_t *topk_ids, const int32_t *lora_ids,
                        const int32_t *expert_map, int n_global, const int32_t *adapter_enabled,
                        int E, int num_loras, int *l_out, int *e_out, uint32_t *err)
{
    int l = lora_ids[p / top_k];
    int e = topk_ids[p];
    uint32_t bit = 0;
    if (l < 0)
        return 0;
    if (l >= num_loras) {
        bit = ORACLE_ERR_LORA;
    } else if (adapter_enabled && adapter_enabled[l] == 0) {
        return 0;
    } else if (expert_map) {
        if (e < 0 || e >= n_global)
            bit = ORACLE_ERR_EXPERT;
        else if (expert_map[e] < 0)
            return 0;
        else if (expert_map[e] >= E)
            bit = ORACLE_ERR_EXPERT;
        else
            e = expert_map[e];
    } else if (e < 0 || e >= E) {
        bit = ORACLE_ERR_EXPERT;
    }
    if (bit) {
        if (err) {
#pragma omp atomic
            *err |= bit;
        }
        return 0;
    }
    *l_out = l;
    *e_out = e;
    return 1;
}

/* y[c] (c < width) gets the delta scale * B @ (A @ x) of one pair, with
 * A [rank, k_in] and B [width, rank] row-major; `w` multiplies the folded
 * value when has_w. */
static void moe_pair_fold(uint16_t *y, const uint16_t *xrow, int k_in, const uint16_t *A,
                          const uint16_t *B, int width, int rank, float scale, int has_w,
                          float w, int add_inputs, int acc64)
{
    float hf[512];
    double hd[512];
    for (int q = 0; q < rank; ++q) {
        const uint16_t *arow = A + (size_t)q * k_in;
        if (acc64) {
            double acc = 0.0;
            for (int k = 0; k < k_in; ++k)
                acc += (double)oracle_bf16_to_f32(xrow[k]) * (double)oracle_bf16_to_f32(arow[k]);
            hd[q] = acc;
        } else {
            float acc = 0.0f;
            for (int k = 0; k < k_in; ++k)
                acc += oracle_bf16_to_f32(xrow[k]) * oracle_bf16_to_f32(arow[k]);
            hf[q] = acc;
        }
    }
    for (int c = 0; c < width; ++c) {
        const uint16_t *brow = B + (size_t)c * rank;
        if (acc64) {
            double d = 0.0;
            for (int q = 0; q < rank; ++q)
                d += hd[q] * (double)oracle_bf16_to_f32(brow[q]);
            double v = (double)scale * d;
            if (has_w)
                v = (double)w * v;
            y[c] = oracle_f64_to_bf16(add_inputs ? (double)oracle_bf16_to_f32(y[c]) + v : v);
        } else {
            float d = 0.0f;
            for (int q = 0; q < rank; ++q)
                d += hf[q] * oracle_bf16_to_f32(brow[q]);
            float v = scale * d;
            if (has_w)
                v = w * v;
            y[c] = oracle_f32_to_bf16(add_inputs ? oracle_bf16_to_f32(y[c]) + v : v);
        }
    }
}

int oracle_moe_w13(uint16_t *y, const uint16_t *x, const uint16_t *const *w_ptr_a,
                   int64_t stride_a, const uint16_t *const *w_ptr_b, int64_t stride_b,
                   int shared_a, const int32_t *topk_ids, const int32_t *lora_ids,
                   const int32_t *expert_map, int n_global, const int32_t *adapter_enabled,
                   int T, int top_k, int E, int H, int I, int rank, int num_loras, float scale,
                   int add_inputs, int acc64, uint32_t *err)
{
    if (T < 0 || top_k < 0 || E <= 0 || H < 0 || I < 0 || rank < 0 || rank > 512 ||
        (expert_map && n_global <= 0))
        return 1;
    const int n_slices = shared_a ? 1 : 2;
    const int width = shared_a ? 2 * I : I;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t p = 0; p < (int64_t)T * top_k; ++p) {
        int l, e;
        if (!moe_pair_key(p, top_k, topk_ids, lora_ids, expert_map, n_global, adapter_enabled, E,
                          num_loras, &l, &e, err))
            continue;
        const uint16_t *xrow = x + (size_t)(p / top_k) * H;
        for (int j = 0; j < n_slices; ++j)
            moe_pair_fold(y + (size_t)p * 2 * I + (size_t)j * I, xrow, H,
                          w_ptr_a[(size_t)j * E + e] + (size_t)l * stride_a,
                          w_ptr_b[(size_t)j * E + e] + (size_t)l * stride_b, width, rank, scale,
                          0, 1.0f, add_inputs, acc64);
    }
    return 0;
}

int oracle_moe_w2(uint16_t *y, const uint16_t *x, const uint16_t *const *w_ptr_a,
                  int64_t stride_a, const uint16_t *const *w_ptr_b, int64_t stride_b,
                  const int32_t *topk_ids, const int32_t *lora_ids, const int32_t *expert_map,
                  int n_global, const int32_t *adapter_enabled, const float *topk_weights,
                  int T, int top_k, int E, int H, int I, int rank, int num_loras, float scale,
                  int add_inputs, int acc64, uint32_t *err)
{
    if (T < 0 || top_k < 0 || E <= 0 || H < 0 || I < 0 || rank < 0 || rank > 512 ||
        (expert_map && n_global <= 0))
        return 1;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t p = 0; p < (int64_t)T * top_k; ++p) {
        int l, e;
        if (!moe_pair_key(p, top_k, topk_ids, lora_ids, expert_map, n_global, adapter_enabled, E,
                          num_loras, &l, &e, err))
            continue;
        moe_pair_fold(y + (size_t)p * H, x + (size_t)p * I, I,
                      w_ptr_a[e] + (size_t)l * stride_a, w_ptr_b[e] + (size_t)l * stride_b, H,
                      rank, scale, topk_weights != NULL,
                      topk_weights ? topk_weights[p] : 1.0f, add_inputs, acc64);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Tensor-parallel sharded LoRA [sharded].  Between the per-rank shrink */
/* (scale 1, fp32 buffer) and the per-rank expand sits one collective:  */
/*  - column parallel (_mcp_apply, ColumnParallelLinearWithShardedLoRA: */
/*    A sliced along the rank): rank p's shard of h, [S, n, Rs] from    */
/*    its Rs rows of A, is all-gathered along the last dimension,       */
/*    h[j][i][p*Rs + q] = shard_p[j][i][q]; a pure copy, so every rank  */
/*    holds the unsharded h exactly;                                    */
/*  - row parallel (RowParallelLinearWithShardedLoRA apply: A sliced    */
/*    along the input, like x): rank p's partial h, [S, n, R] over its  */
/*    k columns, is all-reduced, h = ((part_0 + part_1) + ...) +        */
/*    part_{tp-1} in fp32, rank order (reading: the page leaves the     */
/*    order to the collective).                                         */
/* ------------------------------------------------------------------ */
int oracle_gather_rank_blocks(float *h, const float *shards, int tp, int S, int n, int Rs)
{
    if (tp <= 0 || S < 0 || n < 0 || Rs < 0)
        return 1;
    const int R = tp * Rs;
    for (int p = 0; p < tp; ++p)
        for (int j = 0; j < S; ++j)
            for (int i = 0; i < n; ++i)
                for (int q = 0; q < Rs; ++q)
                    h[((size_t)j * n + i) * R + (size_t)p * Rs + q] =
                        shards[(((size_t)p * S + j) * n + i) * Rs + q];
    return 0;
}

int oracle_rank_sum(float *h, const float *parts, int tp, int64_t len)
{
    if (tp <= 0 || len < 0)
        return 1;
    for (int64_t e = 0; e < len; ++e) {
        float s = parts[e];
        for (int p = 1; p < tp; ++p)
            s = s + parts[(size_t)p * len + e];
        h[e] = s;
    }
    return 0;
}
