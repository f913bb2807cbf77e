/*
 * ep_oracle.c -- plain CPU oracle of rank-major MoE expert-parallel
 * dispatch/combine.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
 * baseline leg load this file. The CUDA library never includes, links or
 * calls it, and this file includes nothing of the CUDA library.
 *
 * What it follows (FlashInfer moe_ep API pages):
 *  - "flashinfer.moe_ep.MoEEpCommunication", dispatch(): a token is delivered
 *    to every rank owning one of its top-k experts; combine(): per token, the
 *    ranks' expert outputs are added up; the combine input has one row per
 *    (source rank, slot), ep_size*tokens_per_rank rows of `hidden`;
 *    runtime_max_tokens_per_rank fixes tokens_per_rank, the capacity
 *    standing in when it is not given.
 *  - "flashinfer.moe_ep.NVLinkOneSidedAlltoAll", class description: one
 *    dispatch carries the hidden row, its scales, the ids and the weights;
 *    a receiving rank keeps token t of source rank s in row
 *    s*tokens_per_rank + t; slots past a source's token count, and tokens
 *    the rank does not receive, are marked with invalid_expert_id.
 *    dispatch(): a rank left out of active_rank_mask receives nothing.
 *  - "flashinfer.moe_ep.CakeAlltoAll", class description: padding slots are
 *    marked the same way.
 *
 * Readings where the pages say nothing (each also fixed by a test):
 *  - invalid_expert_id is -1; ids are int32; weights and scales are fp32.
 *  - experts are split contiguously: rank d owns ids [d*E/ep, (d+1)*E/ep).
 *  - ids outside [0, E) route nowhere; duplicate ids reach a rank once.
 *  - a valid receive row carries the token's full top-k id row unchanged.
 *  - the rank mask filters destinations only.
 *  - combine sums only the ranks a token was routed to, in ascending rank
 *    order, in fp32 starting from +0.0, and rounds once to bf16 (round to
 *    nearest, ties to even); no flush of subnormals.
 *
 * Compile with -O2 -ffp-contract=off and without -ffast-math so every fp32
 * operation is one IEEE binary32 operation in round-to-nearest-even.
 */
#include <stdint.h>
#include <string.h>

#define ORACLE_INVALID_EXPERT_ID (-1)
#define ORACLE_MAX_EP 64

/* ---- number formats, from their definitions ---------------------------- */

/* bfloat16 is the top 16 bits of an IEEE binary32: widening is a shift. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even. The dropped low 16
 * bits decide: above half an ulp rounds up, below rounds down, exactly half
 * rounds to the even neighbour. A carry out of the significand steps the
 * exponent (and reaches infinity from the largest finite value), which is
 * the correct rounded result in this encoding. NaN keeps its sign and
 * becomes the quiet NaN with the top mantissa bit set. */
uint16_t oracle_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t exp = (u >> 23) & 0xFFu;
    uint32_t man = u & 0x7FFFFFu;
    if (exp == 0xFFu && man != 0)
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
    uint32_t hi = u >> 16;
    uint32_t lo = u & 0xFFFFu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u)))
        hi += 1u;
    return (uint16_t)hi;
}

/* OCP 8-bit float E4M3 ("fn" variant): 1 sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits; no infinities; S.1111.111 is NaN. Exponent field 0 is
 * subnormal: m/8 * 2^-6. Otherwise (1 + m/8) * 2^(e-7). */
float oracle_e4m3_to_f32(uint8_t v)
{
    int sign = (v >> 7) & 1;
    int e = (v >> 3) & 0xF;
    int m = v & 0x7;
    float mag;
    if (e == 0xF && m == 0x7) {
        uint32_t qnan = 0x7FC00000u;
        memcpy(&mag, &qnan, sizeof mag);
    } else if (e == 0) {
        mag = (float)m / 8.0f;
        for (int i = 0; i < 6; ++i) mag = mag / 2.0f;
    } else {
        mag = 1.0f + (float)m / 8.0f;
        for (int i = 7; i < e; ++i) mag = mag * 2.0f;
        for (int i = e; i < 7; ++i) mag = mag / 2.0f;
    }
    return sign ? -mag : mag;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits with bias 15, 10 mantissa
 * bits. Exponent field 0 is subnormal (m * 2^-24), 31 is infinity (m = 0)
 * or NaN. Widening to binary32 is exact. */
float oracle_f16_to_f32(uint16_t v)
{
    int sign = (v >> 15) & 1;
    int e = (v >> 10) & 0x1F;
    int m = v & 0x3FF;
    float mag;
    if (e == 0x1F) {
        uint32_t bits = m ? 0x7FC00000u : 0x7F800000u;
        memcpy(&mag, &bits, sizeof mag);
    } else if (e == 0) {
        mag = (float)m;
        for (int i = 0; i < 24; ++i) mag = mag / 2.0f;
    } else {
        mag = 1.0f + (float)m / 1024.0f;
        for (int i = 15; i < e; ++i) mag = mag * 2.0f;
        for (int i = e; i < 15; ++i) mag = mag / 2.0f;
    }
    return sign ? -mag : mag;
}

/* binary32 -> binary16, round to nearest, ties to even. The binary32 value
 * is (2^23 + mantissa) * 2^(e-23) for a normal input; it is cut to the
 * binary16 grid (2^(e-10) for normal results, 2^-24 for subnormal ones) and
 * the dropped bits decide the rounding. Results past the largest finite
 * binary16 (65504) become infinity; binary32 subnormals are far below half
 * the smallest binary16 subnormal and become signed zero. NaN becomes the
 * quiet NaN with the sign kept. */
uint16_t oracle_f32_to_f16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    int exp = (int)((u >> 23) & 0xFFu);
    uint32_t man = u & 0x7FFFFFu;
    if (exp == 0xFF)
        return (uint16_t)(sign | (man ? 0x7E00u : 0x7C00u));
    if (exp == 0)
        return sign;
    int e = exp - 127;
    uint32_t full = (1u << 23) | man;  /* 24 significant bits */
    if (e > 15)
        return (uint16_t)(sign | 0x7C00u);
    int shift;     /* dropped low bits of `full` */
    int base_exp;  /* biased exponent field before any carry */
    if (e >= -14) {
        shift = 13;
        base_exp = e + 15;
    } else {
        shift = 13 + (-14 - e);  /* subnormal: grid of 2^-24 */
        base_exp = 0;
        if (shift > 24 + 1)
            return sign; /* below half of the smallest subnormal */
    }
    uint32_t keep = full >> shift;
    uint32_t rem = full & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (keep & 1u)))
        keep += 1u;
    if (base_exp == 0)
        return (uint16_t)(sign | keep); /* keep == 0x400 is the smallest normal */
    /* normal: keep holds the implicit bit at 0x400; a carry to 0x800 steps the exponent */
    uint32_t field = ((uint32_t)base_exp << 10) + (keep - 0x400u);
    if (field >= 0x7C00u)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | field);
}

/* ---- routing ------------------------------------------------------------ */

/* Does the token with top-k id row `ids` go to rank d? Yes when rank d is
 * active and owns at least one of its valid expert ids. */
int oracle_routed_to(const int32_t *ids, int top_k, int num_experts, int ep_size, int d,
                     int mask_enabled, uint64_t active_rank_mask)
{
    int experts_per_rank = num_experts / ep_size;
    if (mask_enabled && !((active_rank_mask >> d) & 1u))
        return 0;
    for (int k = 0; k < top_k; ++k) {
        int32_t e = ids[k];
        if (e < 0 || e >= num_experts)
            continue;
        if (e / experts_per_rank == d)
            return 1;
    }
    return 0;
}

static int check_geometry(int ep_size, int num_experts, int top_k, int tokens_per_rank,
                          const int32_t *num_tokens)
{
    if (ep_size < 1 || ep_size > ORACLE_MAX_EP || num_experts < ep_size || num_experts % ep_size)
        return -1;
    if (top_k < 1 || tokens_per_rank < 0)
        return -1;
    for (int s = 0; s < ep_size; ++s)
        if (num_tokens[s] < 0 || num_tokens[s] > tokens_per_rank)
            return -1;
    return 0;
}

/* ---- dispatch ----------------------------------------------------------- */

/* Fills every destination rank's receive rows. Destination d's arrays hold
 * ep_size*tokens_per_rank rows; row s*tokens_per_rank + t belongs to token t
 * of source rank s.
 *  - routed token: hidden row (row_bytes raw bytes), scale row (scale_cols
 *    floats), id row and weight row copied unchanged;
 *  - padding slot (t >= num_tokens[s]) or token not routed to d: id row set
 *    to top_k x invalid_expert_id; the other payload rows are not touched.
 * Any output array pointer (or the array of them) may be NULL to skip that
 * payload; recv_ids may not. Returns 0, or -1 on inconsistent sizes. */
int oracle_dispatch(int ep_size, int num_experts, int top_k, int row_bytes, int scale_cols,
                    int tokens_per_rank, int mask_enabled, uint64_t active_rank_mask,
                    const int32_t *num_tokens,
                    const uint8_t *const *hidden, const float *const *scale,
                    const int32_t *const *topk_ids, const float *const *topk_weights,
                    uint8_t *const *recv_hidden, float *const *recv_scale,
                    int32_t *const *recv_ids, float *const *recv_weights)
{
    if (check_geometry(ep_size, num_experts, top_k, tokens_per_rank, num_tokens))
        return -1;
    const int T = tokens_per_rank;
    for (int d = 0; d < ep_size; ++d) {
        for (int s = 0; s < ep_size; ++s) {
            for (int t = 0; t < T; ++t) {
                long r = (long)s * T + t;
                int32_t *id_row = recv_ids[d] + r * top_k;
                int routed = 0;
                if (t < num_tokens[s])
                    routed = oracle_routed_to(topk_ids[s] + (long)t * top_k, top_k, num_experts,
                                              ep_size, d, mask_enabled, active_rank_mask);
                if (!routed) {
                    for (int k = 0; k < top_k; ++k)
                        id_row[k] = ORACLE_INVALID_EXPERT_ID;
                    continue;
                }
                for (int k = 0; k < top_k; ++k)
                    id_row[k] = topk_ids[s][(long)t * top_k + k];
                if (recv_hidden && recv_hidden[d])
                    for (int b = 0; b < row_bytes; ++b)
                        recv_hidden[d][r * row_bytes + b] = hidden[s][(long)t * row_bytes + b];
                if (scale_cols > 0 && scale && recv_scale && recv_scale[d])
                    for (int j = 0; j < scale_cols; ++j)
                        recv_scale[d][r * scale_cols + j] = scale[s][(long)t * scale_cols + j];
                if (topk_weights && recv_weights && recv_weights[d])
                    for (int k = 0; k < top_k; ++k)
                        recv_weights[d][r * top_k + k] = topk_weights[s][(long)t * top_k + k];
            }
        }
    }
    return 0;
}

/* ---- combine ------------------------------------------------------------ */

/* out[s][t][h] = bf16( sum over d = 0..ep_size-1 ascending, for the ranks d
 * that token t of rank s was routed to, of float(expert_output[d][s*T+t][h]) ),
 * accumulated in fp32 from +0.0 and rounded once. expert_output[d] holds
 * ep_size*tokens_per_rank bf16 rows of `hidden` columns; out[s] holds
 * num_tokens[s] rows. Returns 0, or -1 on inconsistent sizes. */
int oracle_combine(int ep_size, int num_experts, int top_k, int hidden, int tokens_per_rank,
                   int mask_enabled, uint64_t active_rank_mask, const int32_t *num_tokens,
                   const int32_t *const *topk_ids, const uint16_t *const *expert_output,
                   uint16_t *const *out)
{
    if (check_geometry(ep_size, num_experts, top_k, tokens_per_rank, num_tokens))
        return -1;
    const int T = tokens_per_rank;
    for (int s = 0; s < ep_size; ++s) {
        for (int t = 0; t < num_tokens[s]; ++t) {
            long r = (long)s * T + t;
            const int32_t *ids = topk_ids[s] + (long)t * top_k;
            for (int h = 0; h < hidden; ++h) {
                float acc = 0.0f;
                for (int d = 0; d < ep_size; ++d) {
                    if (!oracle_routed_to(ids, top_k, num_experts, ep_size, d, mask_enabled,
                                          active_rank_mask))
                        continue;
                    acc = acc + oracle_bf16_to_f32(expert_output[d][r * hidden + h]);
                }
                out[s][(long)t * hidden + h] = oracle_f32_to_bf16_rne(acc);
            }
        }
    }
    return 0;
}

/* The same combine for expert outputs stored as bf16 (dtype 0), binary16
 * (dtype 2) or binary32 (dtype 3): each element is widened to fp32, the
 * routed ranks are added in ascending order from +0.0 in fp32, and the sum
 * is rounded once to the same storage type (not rounded for binary32). */
int oracle_combine_typed(int ep_size, int num_experts, int top_k, int hidden, int tokens_per_rank,
                         int mask_enabled, uint64_t active_rank_mask, const int32_t *num_tokens,
                         const int32_t *const *topk_ids, int dtype, const void *const *expert_output,
                         void *const *out)
{
    if (check_geometry(ep_size, num_experts, top_k, tokens_per_rank, num_tokens))
        return -1;
    if (dtype != 0 && dtype != 2 && dtype != 3)
        return -1;
    const int T = tokens_per_rank;
    for (int s = 0; s < ep_size; ++s) {
        for (int t = 0; t < num_tokens[s]; ++t) {
            long r = (long)s * T + t;
            const int32_t *ids = topk_ids[s] + (long)t * top_k;
            for (int h = 0; h < hidden; ++h) {
                float acc = 0.0f;
                for (int d = 0; d < ep_size; ++d) {
                    if (!oracle_routed_to(ids, top_k, num_experts, ep_size, d, mask_enabled,
                                          active_rank_mask))
                        continue;
                    long i = r * hidden + h;
                    float x;
                    if (dtype == 0)
                        x = oracle_bf16_to_f32(((const uint16_t *)expert_output[d])[i]);
                    else if (dtype == 2)
                        x = oracle_f16_to_f32(((const uint16_t *)expert_output[d])[i]);
                    else
                        x = ((const float *)expert_output[d])[i];
                    acc = acc + x;
                }
                long o = (long)t * hidden + h;
                if (dtype == 0)
                    ((uint16_t *)out[s])[o] = oracle_f32_to_bf16_rne(acc);
                else if (dtype == 2)
                    ((uint16_t *)out[s])[o] = oracle_f32_to_f16_rne(acc);
                else
                    ((float *)out[s])[o] = acc;
            }
        }
    }
    return 0;
}

/* ---- eplb statistics all-gather ----------------------------------------- */

/* Every rank's expert-load statistics gathered alongside the dispatch
 * ("flashinfer.moe_ep.MoEEpCommunication", dispatch(), parameter
 * eplb_local_stats): row r of `global` is rank r's `bytes` bytes. */
int oracle_eplb_gather(int ep_size, int bytes, const uint8_t *const *local, uint8_t *global)
{
    if (ep_size < 1 || ep_size > ORACLE_MAX_EP || bytes < 0)
        return -1;
    for (int r = 0; r < ep_size; ++r)
        for (int b = 0; b < bytes; ++b)
            global[(long)r * bytes + b] = local[r][b];
    return 0;
}

/* ---- identity expert (outside the method; used by invariant tests) ------ */

/* What a rank whose experts are all the identity would hand to combine:
 * for every receive row of rank d that dispatch routed, each column becomes
 * bf16( x * w ), where x is the received value in fp32 (bf16 widened, or
 * e4m3 decoded times its group's scale when scale_cols > 0) and w is the
 * fp32 sum, in ascending k, of the weights of the token's ids that rank d
 * owns (1.0 per such id when recv_weights is NULL). A row that holds no id
 * owned by d (padding, unrouted or masked off) is not written. elem is 2 (bf16) or 1 (e4m3). */
int oracle_identity_expert(int ep_size, int num_experts, int top_k, int hidden, int elem,
                           int scale_cols, int tokens_per_rank,
                           const uint8_t *const *recv_hidden, const float *const *recv_scale,
                           const int32_t *const *recv_ids, const float *const *recv_weights,
                           uint16_t *const *expert_output)
{
    if (ep_size < 1 || ep_size > ORACLE_MAX_EP || num_experts % ep_size)
        return -1;
    if (elem == 1 && (scale_cols <= 0 || hidden % scale_cols))
        return -1;
    const int experts_per_rank = num_experts / ep_size;
    const long rows = (long)ep_size * tokens_per_rank;
    for (int d = 0; d < ep_size; ++d) {
        for (long r = 0; r < rows; ++r) {
            const int32_t *ids = recv_ids[d] + r * top_k;
            float w = 0.0f;
            int owned = 0;
            for (int k = 0; k < top_k; ++k) {
                int32_t e = ids[k];
                if (e < 0 || e >= num_experts || e / experts_per_rank != d)
                    continue;
                owned += 1;
                w = w + (recv_weights ? recv_weights[d][r * top_k + k] : 1.0f);
            }
            if (!owned) /* padding, unrouted or masked row: nothing to compute */
                continue;
            for (int h = 0; h < hidden; ++h) {
                float x;
                if (elem == 2) {
                    const uint8_t *p = recv_hidden[d] + (r * hidden + h) * 2;
                    x = oracle_bf16_to_f32((uint16_t)(p[0] | (p[1] << 8)));
                } else {
                    int group = h / (hidden / scale_cols);
                    x = oracle_e4m3_to_f32(recv_hidden[d][r * hidden + h]) *
                        recv_scale[d][r * scale_cols + group];
                }
                expert_output[d][r * hidden + h] = oracle_f32_to_bf16_rne(x * w);
            }
        }
    }
    return 0;
}
