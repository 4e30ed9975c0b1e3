/*
 * moe_oracle.c -- CPU oracle for routed Mixture-of-Experts expert execution.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link or
 * call this file: only tests/, __graft_entry__.smoke() and the CPU-baseline
 * leg of bench.py use it. It shares no code, header, table or helper with the
 * CUDA library under moe_routed_expert_routing_gb300/csrc.
 *
 * What it computes (plain definitions, written out loop by loop, in fp32):
 *
 *  1. Local dispatch -- TileOps PR #1738 "Separate dispatched expert compute",
 *     Summary ("Compose routed expert execution from local dispatch, expert
 *     compute, and combine") and Scope ("BF16 tight/no-pad expert compute";
 *     consumers read the valid-row count from expert_offsets[-1:]).
 *     A routed slot is s = t*k + j. Count the slots of each expert, take the
 *     exclusive prefix sum as expert_offsets[E+1], then walk s = 0..R-1 in
 *     ascending order and give each slot the next free row of its expert.
 *     That walk is the definition of a stable scatter: inside one expert the
 *     rows keep slot order. perm[row] = s, inv[s] = row.
 *     Reading: an id of -1 marks a dropped slot (no row, contributes nothing);
 *     any other id outside [0, E) is also dropped and counted as an error.
 *
 *  2. Expert MLP for one routed row (the dispatched-expert MLP of the same
 *     page, Summary, with its fused-gated epilogue, Review follow-up):
 *       g_n = sum_h x_h * W13[e, n, h]        n in [0, I)   (gate: rows 0..I-1)
 *       u_n = sum_h x_h * W13[e, I + n, h]                  (up:   rows I..2I-1)
 *       a_n = bf16( (g_n / (1 + exp(-g_n))) * u_n )         SiLU(gate) * up
 *       y_m = sum_n a_n * W2[e, m, n]         m in [0, H)
 *     All sums in fp32, index ascending. The activation is rounded to bf16
 *     (round to nearest, ties to even); y stays fp32.
 *
 *  3. Combine -- same page, Summary ("Keep routing weights ... outside expert
 *     compute"): out_acc[t, m] = sum_{j ascending} w[t, j] * y_{t,j}[m] in
 *     fp32, then out[t, m] = bf16(out_acc[t, m]). Weights are used as given.
 *
 *  4. MXFP8 weights -- the pages' MXFP8 path (FlashInfer moe_ep page, PR
 *     #3980: MXFP8 mega MoE with prequantized weight packs; its quantized
 *     combine wire spells the format out as 'mxfp8' = 32 e4m3 x e8m0). The
 *     format is the OCP Microscaling (MX) v1.0 one: each block of 32
 *     consecutive elements along K shares one E8M0 scale X = 2^e, each
 *     element is an FP8 E4M3 value P, and the block stands for X * P. One
 *     block is quantized the way the MX spec describes:
 *       e = floor(log2(max |V|)) - 8      (8 = exponent of E4M3's largest
 *                                          normal, 448 = 1.75 * 2^8),
 *           clamped to E8M0's [-127, 127], stored as e + 127;
 *       P = E4M3(V / X), round to nearest, ties to even; a magnitude above
 *           448 becomes 448 (V / X of the block maximum lies in [256, 512)).
 *     A block of zeros gets e = -127 and zero elements. E4M3 (OCP FP8):
 *     sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
 *     holds the subnormals m * 2^-9; no infinities; S.1111.111 is NaN.
 *     Dequantization X * P is exact in bf16 (3 mantissa bits fit in 7), so
 *     the MXFP8 forward is the bf16 forward above on dequantized weights.
 *
 * Parity pins (tests/test_oracle_pins.py): dispatch invariants and a brute
 * force restatement; bf16 rounding against an independent library cast; the
 * one-expert k=1 special case against a dense MLP built from library matmuls;
 * dispatch+combine with an identity expert against the closed form
 * sum_j w[t,j] * x[t]; a naive fp64 restatement on tiny shapes.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (oracle/build.py).
 * -ffp-contract=off keeps every multiply and add separately rounded, so the
 * x86 container and the aarch64 GPU host give identical bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- bf16 <-> fp32 (bf16 is the top 16 bits of an IEEE-754 binary32) ---- */

static float bf16_bits_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round to nearest, ties to even: add half of the dropped range, plus one
 * when the kept part is odd, then truncate. NaN stays a quiet NaN. */
static uint16_t f32_to_bf16_bits_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

void oracle_round_bf16(int64_t n, const float *in, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_bits_rne(in[i]);
}

/* ---- 1. dispatch ---------------------------------------------------------- */

/* ids[R] -> counts[E], offsets[E+1], perm[R] (rows >= offsets[E] set to -1),
 * inv[R] (-1 for a dropped slot). Returns the number of ids that were neither
 * -1 nor inside [0, E). */
int32_t oracle_dispatch(int32_t R, int32_t E, const int32_t *ids,
                        int32_t *counts, int32_t *offsets, int32_t *perm,
                        int32_t *inv)
{
    int32_t bad = 0;
    for (int32_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int32_t s = 0; s < R; ++s) {
        int32_t e = ids[s];
        if (e >= 0 && e < E)
            counts[e] += 1;
        else if (e != -1)
            bad += 1;
    }
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];

    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int32_t e = 0; e < E; ++e)
        cursor[e] = offsets[e];
    for (int32_t r = 0; r < R; ++r)
        perm[r] = -1;
    for (int32_t s = 0; s < R; ++s) {
        int32_t e = ids[s];
        if (e >= 0 && e < E) {
            int32_t row = cursor[e];
            cursor[e] += 1;
            perm[row] = s;
            inv[s] = row;
        } else {
            inv[s] = -1;
        }
    }
    free(cursor);
    return bad;
}

/* ---- 2. expert MLP --------------------------------------------------------- */

/* Gate/up sums for output n of one row, then the rounded activation. */
static uint16_t gate_up_one(int32_t H, int32_t I, const uint16_t *x, const uint16_t *W13e, int32_t n)
{
    const uint16_t *wg = W13e + (size_t)n * (size_t)H;
    const uint16_t *wu = W13e + (size_t)(I + n) * (size_t)H;
    float g = 0.0f, u = 0.0f;
    for (int32_t h = 0; h < H; ++h) {
        float xh = bf16_bits_to_f32(x[h]);
        g += xh * bf16_bits_to_f32(wg[h]);
        u += xh * bf16_bits_to_f32(wu[h]);
    }
    float silu = g / (1.0f + expf(-g));
    return f32_to_bf16_bits_rne(silu * u);
}

/* Down-projection sum for output m of one row, from the activation a[I]. */
static float down_one(int32_t I, const float *a, const uint16_t *W2e, int32_t m)
{
    const uint16_t *w2 = W2e + (size_t)m * (size_t)I;
    float y = 0.0f;
    for (int32_t n = 0; n < I; ++n)
        y += a[n] * bf16_bits_to_f32(w2[n]);
    return y;
}

/* One routed row through one expert. x[H], W13e[2I, H], W2e[H, I] are bf16
 * bit patterns; y_out[H] fp32; a_scratch[I] holds the activation. */
static void expert_mlp_row(int32_t H, int32_t I, const uint16_t *x, const uint16_t *W13e,
                           const uint16_t *W2e, float *y_out, float *a_scratch)
{
    for (int32_t n = 0; n < I; ++n)
        a_scratch[n] = bf16_bits_to_f32(gate_up_one(H, I, x, W13e, n));
    for (int32_t m = 0; m < H; ++m)
        y_out[m] = down_one(I, a_scratch, W2e, m);
}

/* Several rows through one expert: x_rows[n_rows, H] -> a_rows[n_rows, I]
 * (bf16 bits, required), y_rows[n_rows, H]. Every output element is independent and
 * computed exactly as in expert_mlp_row, so the work is spread over
 * (row, output) pairs; the bits do not depend on the thread count. */
void oracle_expert_rows(int32_t H, int32_t I, const uint16_t *W13e,
                        const uint16_t *W2e, int32_t n_rows,
                        const uint16_t *x_rows, uint16_t *a_rows, float *y_rows)
{
    float *a = (float *)malloc(sizeof(float) * (size_t)I * (size_t)(n_rows > 0 ? n_rows : 1));
    int64_t n_ru = (int64_t)n_rows * I;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < n_ru; ++i) {
        int32_t r = (int32_t)(i / I), n = (int32_t)(i % I);
        uint16_t ab = gate_up_one(H, I, x_rows + (size_t)r * H, W13e, n);
        a_rows[i] = ab;
        a[i] = bf16_bits_to_f32(ab);
    }
    int64_t n_rm = (int64_t)n_rows * H;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < n_rm; ++i) {
        int32_t r = (int32_t)(i / H), m = (int32_t)(i % H);
        y_rows[i] = down_one(I, a + (size_t)r * I, W2e, m);
    }
    free(a);
}

/* ---- 3. combine ------------------------------------------------------------ */

/* y_slot[n_tok, k, H] holds each routed slot's expert output (fp32); valid[n_tok,
 * k] is 0 for a dropped slot. out_acc[n_tok, H] fp32, out[n_tok, H] bf16. */
void oracle_combine_slots(int32_t n_tok, int32_t k, int32_t H,
                          const float *y_slot, const float *w,
                          const int32_t *valid, float *out_acc, uint16_t *out)
{
    for (int32_t t = 0; t < n_tok; ++t) {
        for (int32_t m = 0; m < H; ++m) {
            float acc = 0.0f;
            for (int32_t j = 0; j < k; ++j) {
                size_t s = (size_t)t * k + j;
                if (valid[s])
                    acc += w[s] * y_slot[s * (size_t)H + m];
            }
            out_acc[(size_t)t * H + m] = acc;
            out[(size_t)t * H + m] = f32_to_bf16_bits_rne(acc);
        }
    }
}

/* Combine from the expert-major (sorted) batch: y_sorted[rows, H] fp32,
 * inv[T*k] maps slot -> row (-1 = dropped). This is the form the dispatched
 * batch takes between expert compute and combine. */
void oracle_combine_sorted(int32_t T, int32_t k, int32_t H,
                           const float *y_sorted, const int32_t *inv,
                           const float *w, float *out_acc, uint16_t *out)
{
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t m = 0; m < H; ++m) {
            float acc = 0.0f;
            for (int32_t j = 0; j < k; ++j) {
                size_t s = (size_t)t * k + j;
                int32_t row = inv[s];
                if (row >= 0)
                    acc += w[s] * y_sorted[(size_t)row * H + m];
            }
            out_acc[(size_t)t * H + m] = acc;
            out[(size_t)t * H + m] = f32_to_bf16_bits_rne(acc);
        }
    }
}

/* ---- whole forward over a token subset ------------------------------------ */

/* Loops over the listed tokens and their k experts: steps 2 and 3 above.
 * x[T, H], ids[T, k], w[T, k], W13[E, 2I, H], W2[E, H, I]. tok[n_tok] lists
 * the tokens to evaluate; out_acc / out are [n_tok, H]. Returns the number of
 * ids that were neither -1 nor inside [0, E). */
int32_t oracle_moe_tokens(int32_t T, int32_t E, int32_t k, int32_t H, int32_t I,
                          const uint16_t *x, const int32_t *ids, const float *w,
                          const uint16_t *W13, const uint16_t *W2, int32_t n_tok,
                          const int32_t *tok, float *out_acc, uint16_t *out)
{
    (void)T;
    int32_t bad = 0;
    size_t per13 = (size_t)2 * I * H, per2 = (size_t)H * I;
#pragma omp parallel reduction(+ : bad)
    {
        float *scratch = (float *)malloc(sizeof(float) * (size_t)I);
        float *y = (float *)malloc(sizeof(float) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
        for (int32_t q = 0; q < n_tok; ++q) {
            int32_t t = tok[q];
            float *acc = out_acc + (size_t)q * H;
            for (int32_t m = 0; m < H; ++m)
                acc[m] = 0.0f;
            for (int32_t j = 0; j < k; ++j) {
                int32_t e = ids[(size_t)t * k + j];
                if (e < 0 || e >= E) {
                    if (e != -1)
                        bad += 1;
                    continue;
                }
                expert_mlp_row(H, I, x + (size_t)t * H, W13 + (size_t)e * per13,
                               W2 + (size_t)e * per2, y, scratch);
                float wj = w[(size_t)t * k + j];
                for (int32_t m = 0; m < H; ++m)
                    acc[m] += wj * y[m];
            }
            for (int32_t m = 0; m < H; ++m)
                out[(size_t)q * H + m] = f32_to_bf16_bits_rne(acc[m]);
        }
        free(y);
        free(scratch);
    }
    return bad;
}

/* ---- 4. MXFP8 weights (OCP MX v1.0: E4M3 elements, one E8M0 scale per 32) ---- */

/* Value of an E4M3 code, from the format's fields. */
static float e4m3_value(uint8_t c)
{
    int sign = (c >> 7) & 1, ex = (c >> 3) & 15, man = c & 7;
    float mag;
    if (ex == 15 && man == 7)
        mag = NAN;
    else if (ex == 0)
        mag = ldexpf((float)man, -9);                   /* subnormal: m * 2^-9 */
    else
        mag = ldexpf(1.0f + (float)man / 8.0f, ex - 7);
    return sign ? -mag : mag;
}

void oracle_e4m3_values(float *out)
{
    for (int c = 0; c < 256; ++c)
        out[c] = e4m3_value((uint8_t)c);
}

/* Nearest E4M3 code to a finite v, ties to the even mantissa, magnitudes
 * above 448 saturated to 448. The spacing of the codes around |v| is
 * 2^(floor(log2|v|) - 3) among the normals and 2^-9 among the subnormals;
 * |v| divided by that spacing is rounded to an integer (rintf rounds to
 * nearest even), and a carry into the next binade is renormalised. */
static uint8_t e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    float a = fabsf(v);
    if (a >= 448.0f)
        return sign | 0x7E;
    if (a < ldexpf(1.0f, -6)) {
        int q = (int)rintf(ldexpf(a, 9));              /* 0..8; 8 is the smallest normal, code 0x08 */
        return sign | (uint8_t)q;
    }
    int ex2;
    frexpf(a, &ex2);                                    /* a = f * 2^ex2, f in [0.5, 1) */
    int e = ex2 - 1;                                    /* a in [2^e, 2^(e+1)) */
    int q = (int)rintf(ldexpf(a, 3 - e));               /* 8..16 */
    if (q == 16) {
        q = 8;
        e += 1;
    }
    int field = e + 7, man = q - 8;
    if (field > 15 || (field == 15 && man == 7))
        return sign | 0x7E;
    return sign | (uint8_t)((field << 3) | man);
}

/* rows x K bf16 weights (K a multiple of 32) -> q[rows, K] E4M3 codes and
 * s[rows, K/32] E8M0 scale codes, both row-major. */
void oracle_mx_quantize(int64_t rows, int32_t K, const uint16_t *w, uint8_t *q, uint8_t *s)
{
    int32_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int32_t b = 0; b < nb; ++b) {
            const uint16_t *v = w + r * K + (int64_t)b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(bf16_bits_to_f32(v[i]));
                if (a > amax)
                    amax = a;
            }
            int e = -127;
            if (amax > 0.0f) {
                int ex2;
                frexpf(amax, &ex2);
                e = (ex2 - 1) - 8;
                if (e < -127)
                    e = -127;
                if (e > 127)
                    e = 127;
            }
            s[r * nb + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i)
                q[r * K + (int64_t)b * 32 + i] = e4m3_encode(ldexpf(bf16_bits_to_f32(v[i]), -e));
        }
    }
}

/* q[rows, K], s[rows, K/32] -> bf16 bits of X * P. */
void oracle_mx_dequantize(int64_t rows, int32_t K, const uint8_t *q, const uint8_t *s, uint16_t *out)
{
    int32_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int32_t k = 0; k < K; ++k) {
            int e = (int)s[r * nb + k / 32] - 127;
            out[r * K + k] = f32_to_bf16_bits_rne(ldexpf(e4m3_value(q[r * K + k]), e));
        }
}
