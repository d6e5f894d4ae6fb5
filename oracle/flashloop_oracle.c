/*
 * flashloop_oracle.c -- plain CPU oracle of the FlashLoop lazy loop step.
 *
 * TEST INFRASTRUCTURE, not product code. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load this file. It shares no
 * source, header, table or helper with the CUDA library, and it includes
 * nothing from it.
 *
 * Method source: the rit.work page "FlashLoop: Fast and Memory-Efficient
 * Looped Transformers via Lazy Updates" (a summary of the Yang & Liu
 * preprint), in particular
 *   [P2-late]  section "Later loops change only part of the state"
 *              (each loop has its own KV cache; few tokens keep changing and
 *              the active group narrows and nests; a small stable key group
 *              drives the loop-to-loop change of attention; neighbouring KV
 *              sets differ less than whole states, so base + small deltas);
 *   [P2-three] section "FlashLoop combines three kinds of saving"
 *              (dense early loops; rank tokens by how much their hidden
 *              state changed and recompute only the active ones, the rest
 *              reuse state and KV entries; choose keys from the previous
 *              loop's statistics and keep the selected group's total
 *              probability mass; KV cache = compressed base + a sequence of
 *              compressed deltas, a low-bit delta for active tokens and no
 *              entry for inactive ones, 4-bit deltas).
 * Where the page leaves a step open, the plain readings used here are:
 *   R1  previous-loop probability of row i, key j:
 *       p_ij = exp(qhat_i . krec_j / sqrt(d) - Z_i) with the row's last
 *       query qhat_i and log-normaliser Z_i (state that persists).
 *   R2  one key set S per (sequence, head), ranked by column mass c_j.
 *   R3  causal: S_i = {j in S : j <= i}; a row with S_i empty (or whose
 *       old mass m_i is below FLT_MIN) keeps its O, Z and qhat.
 *   R4  attention reads the reconstructed cache: base + dequantised deltas
 *       in ascending loop order, fp32, rounded RNE to bf16.
 *   R6  quantiser: symmetric int4 codes in [-7, 7], one fp16 scale per 32
 *       contiguous elements, scale = fp16_rne(amax / 7) (fp32 divide),
 *       code = rint_even(delta / scale) clamped to +-7, zero scale -> zero
 *       codes; element 2t in the low nibble of byte t.
 *   R6' narrower deltas (variants beyond the page's 4-bit setting; it says quality drops
 *       noticeably below 4 bits): the same quantiser with codes of `bits`
 *       bits, 2 <= bits <= 4: qmax = 2^(bits-1) - 1, scale =
 *       fp16_rne(amax / qmax), codes clamped to [-qmax, qmax]; element x of
 *       an (entry, head) row occupies bits [bits x, bits x + bits) of the row
 *       read as a little-endian bit string, two's complement (for bits = 4
 *       this is R6's nibble order).
 *   R8  compressed base (the page: "a compressed base plus a sequence of
 *       compressed deltas"): int8 codes with one fp16 scale per 32 elements,
 *       scale = fp16_rne(amax / 127), code = rint_even(x / scale) clamped to
 *       [-127, 127], zero scale -> zero codes; the base value is scale * code.
 *   R7  R = ceil(r N), K = ceil(k N), clamped to [1, N]; ties in every
 *       ranking go to the lower index; index lists ascending.
 *   R9  synthetic looped block around the step (an extension of the step; the
 *       page says a later loop recomputes only its active tokens but gives
 *       no block): with x = H_{l-1}[i], q, k, v = bf16(x W_q), bf16(x W_k),
 *       bf16(x W_v); O from the loop's attention; y = bf16(x + bf16(O) W_o);
 *       u = bf16(relu(y W_1)); H_l[i] = bf16(y + u W_2). Every output is the
 *       exact value (products summed in double) rounded ONCE to bf16, nearest
 *       even (orc_round_bf16 below); tokens a lazy loop leaves inactive keep
 *       H_l[i] = H_{l-1}[i]. No normalisation layers.
 * Build with gcc -O2 -ffp-contract=off so every fp32 expression rounds
 * exactly as written. Attention and norms accumulate in double.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <omp.h>

/* ------------------------------------------------------------------ */
/* number formats (IEEE 754 binary16 and bfloat16, round to nearest even) */

float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

float orc_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
    float f;
    if (e == 0) {               /* zero or subnormal: m * 2^-24 */
        f = (float)m * 5.9604644775390625e-8f;
        return sign ? -f : f;
    }
    uint32_t u;
    if (e == 31) u = sign | 0x7F800000u | (m << 13);
    else u = sign | ((e - 15u + 127u) << 23) | (m << 13);
    memcpy(&f, &u, 4);
    return f;
}

uint16_t orc_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax > 0x7F800000u) return sign | 0x7E00u;          /* NaN */
    if (ax >= 0x477FF000u) return sign | 0x7C00u;         /* >= 65520 rounds to inf */
    if (ax < 0x38800000u) {                               /* below 2^-14: subnormal */
        float v;
        memcpy(&v, &ax, 4);
        double q = nearbyint((double)v * 16777216.0);     /* units of 2^-24, ties to even */
        return (uint16_t)(sign | (uint16_t)q);
    }
    uint32_t e = (ax >> 23) - 127u + 15u;
    uint32_t m = ax & 0x7FFFFFu;
    uint32_t h = (e << 10) | (m >> 13);
    uint32_t rem = m & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
    return (uint16_t)(sign | h);
}

/* ------------------------------------------------------------------ */
/* [P2-three] "rank tokens by how much their hidden states changed":
 * score_i = || h_cur_i - h_prev_i ||_2^2 over the D hidden features.
 * Ranking by the square is ranking by the norm. Exact up to double rounding. */
void orc_token_scores(const uint16_t *h_prev, const uint16_t *h_cur,
                      int64_t B, int64_t N, int64_t D, double *score) {
#pragma omp parallel for schedule(static)
    for (int64_t row = 0; row < B * N; ++row) {
        const uint16_t *a = h_prev + row * D, *b = h_cur + row * D;
        double s = 0.0;
        for (int64_t x = 0; x < D; ++x) {
            double dx = (double)orc_bf16_to_f32(b[x]) - (double)orc_bf16_to_f32(a[x]);
            s += dx * dx;
        }
        score[row] = s;
    }
}

/* ------------------------------------------------------------------ */
/* [P2-three] keep the top-k of a ranking (tokens by change, keys by the
 * previous loop's column statistics). R7: ties go to the lower index; the
 * kept indices are returned in ascending order. Plain sort, row by row. */
typedef struct { double s; int32_t i; } orc_item;

static int orc_by_score_desc(const void *pa, const void *pb) {
    const orc_item *a = (const orc_item *)pa, *b = (const orc_item *)pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

static int orc_by_i32(const void *pa, const void *pb) {
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

void orc_topk_rows(const double *score, int64_t rows, int64_t n, int64_t k, int32_t *out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        orc_item *it = (orc_item *)malloc(sizeof(orc_item) * (size_t)n);
        for (int64_t j = 0; j < n; ++j) { it[j].s = score[r * n + j]; it[j].i = (int32_t)j; }
        qsort(it, (size_t)n, sizeof(orc_item), orc_by_score_desc);
        int32_t *o = out + r * k;
        for (int64_t t = 0; t < k; ++t) o[t] = it[t].i;
        qsort(o, (size_t)k, sizeof(int32_t), orc_by_i32);
        free(it);
    }
}

/* ------------------------------------------------------------------ */
/* KV cache as [P2-three] describes it: a base plus a sequence of deltas.
 * A delta layer holds, per sequence b, `cnt` entries with ascending token
 * indices idx[b][e], codes [b][e][h][d * bits / 8] (R6') and fp16 scales
 * [b][e][h][d/32]. The base is bf16 [b][j][h][d], or (R8) int8 codes
 * [b][j][h][d] with fp16 scales [b][j][h][d/32]. */
typedef struct {
    const uint16_t *bf16;        /* bf16 base, or NULL */
    const int8_t *codes;         /* R8 base codes (when bf16 is NULL) */
    const uint16_t *scales;
} orc_base;
typedef struct {
    const int32_t *idx;
    const uint8_t *codes;
    const uint16_t *scales;
    int64_t cnt;
} orc_layer;

static int64_t orc_find(const int32_t *idx, int64_t cnt, int64_t j) {
    int64_t lo = 0, hi = cnt - 1;
    while (lo <= hi) {
        int64_t mid = (lo + hi) / 2;
        if (idx[mid] == j) return mid;
        if (idx[mid] < j) lo = mid + 1; else hi = mid - 1;
    }
    return -1;
}

/* R6': code of element x of a row of `bits`-bit codes (little-endian bit string). */
static int orc_code(const uint8_t *row, int64_t x, int bits) {
    int v = 0;
    for (int k = 0; k < bits; ++k) {
        int64_t bit = x * bits + k;
        v |= ((row[bit / 8] >> (bit % 8)) & 1) << k;
    }
    return v >= (1 << (bits - 1)) ? v - (1 << bits) : v;
}

static void orc_put_code(uint8_t *row, int64_t x, int bits, int v) {
    for (int k = 0; k < bits; ++k) {
        int64_t bit = x * bits + k;
        uint8_t m = (uint8_t)(1u << (bit % 8));
        if ((v >> k) & 1) row[bit / 8] |= m; else row[bit / 8] &= (uint8_t)~m;
    }
}

/* R4: fp32 reconstruction of token j, head h: base (R8: scale * code), then
 * each delta layer in ascending order that holds an entry for j adds
 * scale * code. */
static void orc_recon(const orc_base *base, int64_t Nk, int64_t H, int64_t d, int bits,
                      const orc_layer *L, int nl, int64_t b, int64_t j, int64_t h, float *out) {
    const int64_t row = ((b * Nk + j) * H + h);
    if (base->bf16) {
        for (int64_t x = 0; x < d; ++x) out[x] = orc_bf16_to_f32(base->bf16[row * d + x]);
    } else {
        for (int64_t x = 0; x < d; ++x)
            out[x] = orc_f16_to_f32(base->scales[row * (d / 32) + x / 32]) * (float)base->codes[row * d + x];
    }
    for (int m = 0; m < nl; ++m) {
        int64_t e = orc_find(L[m].idx + b * L[m].cnt, L[m].cnt, j);
        if (e < 0) continue;
        const uint8_t *cd = L[m].codes + ((b * L[m].cnt + e) * H + h) * (d * bits / 8);
        const uint16_t *sc = L[m].scales + ((b * L[m].cnt + e) * H + h) * (d / 32);
        for (int64_t x = 0; x < d; ++x) {
            float s = orc_f16_to_f32(sc[x / 32]);
            float t = s * (float)orc_code(cd, x, bits);
            out[x] = out[x] + t;
        }
    }
}

static void orc_pack_layers(orc_layer *L, int nl, const int32_t *const *idx,
                            const uint8_t *const *codes, const uint16_t *const *scales,
                            const int64_t *cnt) {
    for (int m = 0; m < nl; ++m) {
        L[m].idx = idx[m]; L[m].codes = codes[m]; L[m].scales = scales[m]; L[m].cnt = cnt[m];
    }
}

/* R6 / R6' / R8 applied to one group of 32 fp32 values with codes in
 * [-qmax, qmax]: qmax = 7 for int4 deltas, 3 for int3, 1 for int2, 127 for the
 * int8 base. */
static void orc_quant_group(const float *delta, int qmax, uint16_t *scale_out, int *q) {
    float amax = 0.0f;
    for (int e = 0; e < 32; ++e) {
        float a = fabsf(delta[e]);
        if (a > amax) amax = a;
    }
    float sf = amax / (float)qmax;
    uint16_t sh = orc_f32_to_f16(sf);
    float s = orc_f16_to_f32(sh);
    *scale_out = sh;
    for (int e = 0; e < 32; ++e) {
        int v = 0;
        if (s > 0.0f) {
            float t = delta[e] / s;
            v = (int)nearbyintf(t);
            if (v > qmax) v = qmax;
            if (v < -qmax) v = -qmax;
        }
        q[e] = v;
    }
}

/* R8: the compressed base of a bf16 layer x [B,Nk,H,d]: int8 codes [B,Nk,H,d]
 * and fp16 scales [B,Nk,H,d/32]. */
void orc_quantize_base(const uint16_t *x, int64_t B, int64_t Nk, int64_t H, int64_t d,
                       int8_t *codes, uint16_t *scales) {
#pragma omp parallel for schedule(static)
    for (int64_t row = 0; row < B * Nk * H; ++row) {
        float v[512];
        int q[32];
        for (int64_t t = 0; t < d; ++t) v[t] = orc_bf16_to_f32(x[row * d + t]);
        for (int64_t g = 0; g < d / 32; ++g) {
            orc_quant_group(v + g * 32, 127, &scales[row * (d / 32) + g], q);
            for (int e = 0; e < 32; ++e) codes[row * d + g * 32 + e] = (int8_t)q[e];
        }
    }
}

/* [P2-three] "for tokens that stay active, write the low-bit difference
 * from the previous state; inactive tokens get no new entry"; 4-bit deltas.
 * For every active token i of sequence b and every head, the delta of the
 * loop-l tensor x_l against the previous loop's reconstruction is quantised
 * per 32-element group (R6). Writes the new layer's entries in the order of
 * `active` (ascending). `x_l` and `base` are [B,Nk,H,d] bf16. */
void orc_kv_delta_append(const uint16_t *x_l, const uint16_t *base_bf16, const int8_t *base_codes,
                         const uint16_t *base_scales, int bits,
                         int nl, const int32_t *const *idx, const uint8_t *const *codes,
                         const uint16_t *const *scales, const int64_t *cnt,
                         int64_t B, int64_t Nk, int64_t H, int64_t d,
                         const int32_t *active, int64_t R,
                         int32_t *out_idx, uint8_t *out_codes, uint16_t *out_scales) {
    orc_layer L[64];
    orc_pack_layers(L, nl, idx, codes, scales, cnt);
    const orc_base base = {base_bf16, base_codes, base_scales};
    const int qmax = (1 << (bits - 1)) - 1;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t e = 0; e < R; ++e) {
            int64_t i = active[b * R + e];
            out_idx[b * R + e] = (int32_t)i;
            float rec[512], delta[512];
            int q[32];
            for (int64_t h = 0; h < H; ++h) {
                orc_recon(&base, Nk, H, d, bits, L, nl, b, i, h, rec);
                const uint16_t *src = x_l + ((b * Nk + i) * H + h) * d;
                for (int64_t x = 0; x < d; ++x) delta[x] = orc_bf16_to_f32(src[x]) - rec[x];
                uint8_t *cd = out_codes + ((b * R + e) * H + h) * (d * bits / 8);
                uint16_t *sc = out_scales + ((b * R + e) * H + h) * (d / 32);
                for (int64_t g = 0; g < d / 32; ++g) {
                    orc_quant_group(delta + g * 32, qmax, &sc[g], q);
                    for (int t = 0; t < 32; ++t) orc_put_code(cd, g * 32 + t, bits, q[t]);
                }
            }
        }
    }
}

/* R4: reconstruct every token of the cache (base + `nl` delta layers) as
 * fp32 (out_f32, may be NULL) and rounded RNE to bf16 (out_bf16, may be NULL). */
void orc_reconstruct(const uint16_t *base_bf16, const int8_t *base_codes, const uint16_t *base_scales, int bits,
                     int nl, const int32_t *const *idx,
                     const uint8_t *const *codes, const uint16_t *const *scales, const int64_t *cnt,
                     int64_t B, int64_t Nk, int64_t H, int64_t d,
                     float *out_f32, uint16_t *out_bf16) {
    orc_layer L[64];
    orc_pack_layers(L, nl, idx, codes, scales, cnt);
    const orc_base base = {base_bf16, base_codes, base_scales};
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t j = 0; j < Nk; ++j) {
            float rec[512];
            for (int64_t h = 0; h < H; ++h) {
                orc_recon(&base, Nk, H, d, bits, L, nl, b, j, h, rec);
                int64_t off = ((b * Nk + j) * H + h) * d;
                for (int64_t x = 0; x < d; ++x) {
                    if (out_f32) out_f32[off + x] = rec[x];
                    if (out_bf16) out_bf16[off + x] = orc_f32_to_bf16(rec[x]);
                }
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* [P2-three] lazy attention with preserved probability mass, in double.
 *
 * For each sequence b, head h, and row r (key position pos_i, state slot s):
 *   S_i   = {j in S[b,h] : j <= pos_i}                       (R3)
 *   p_j   = exp(qhat_s . kold_j / sqrt(d) - Z_s)             (R1)
 *   m     = sum_{S_i} p_j,   u = sum_{S_i} p_j vold_j
 *   tau_j = q_s . knew_j / sqrt(d),  lam = logsumexp_{S_i} tau
 *   w     = sum_{S_i} exp(tau_j - lam) vnew_j
 *   O_s  <- O_s - u + m w,  Z_s <- lam - ln m,  qhat_s <- q_s
 *   c_j  += m exp(tau_j - lam) - p_j                         (column mass)
 * so the selected keys keep the old total mass m instead of being
 * renormalised to one. `first` is the first dense loop: no previous state,
 * m := 1, u := 0, p := 0, and c is overwritten rather than updated.
 * Rows are independent; the column-mass changes of all rows are summed in
 * double and added to c once per (b, h). `bh_mask` (may be NULL) restricts
 * the work to a subset of (b, h) pairs.
 * Shapes: q, qhat [B,Ns,H,d] bf16; o [B,Ns,H,d] f32; z [B,H,Ns] f32;
 * c [B,H,Nk] f32; S [B,H,K] i32; k/v old/new [B,Nk,H,d] bf16;
 * pos, slot [B,R] i32; m_out [B,H,R] double (may be NULL; NaN when skipped). */
typedef struct {
    int first;
    int64_t B, H, d, Nk, Ns, R, K;
    const int32_t *pos, *slot;
    const uint16_t *q;
    uint16_t *qhat;
    float *o, *z;
    const int32_t *S;
    const uint16_t *k_old, *v_old, *k_new, *v_new;
    double *m_out;
} orc_attn_args;

/* One row: updates its own state row and adds its column-mass changes to
 * dc[0..K) (indexed like S). Scratch p, tau hold K doubles, u, w hold d. */
static void orc_attention_row(const orc_attn_args *a, int64_t b, int64_t h, int64_t r, double *dc,
                              double *p, double *tau, double *u, double *w) {
    const int64_t d = a->d, H = a->H, Nk = a->Nk, Ns = a->Ns, K = a->K;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    const int32_t *Sb = a->S + (b * H + h) * K;
    int64_t i = a->pos[b * a->R + r], s = a->slot[b * a->R + r];
    if (a->m_out) a->m_out[(b * H + h) * a->R + r] = NAN;
    int64_t ns = 0;                     /* |S_i|: S is ascending */
    while (ns < K && Sb[ns] <= i) ++ns;
    if (ns == 0) return;
    const uint16_t *qs = a->q + ((b * Ns + s) * H + h) * d;
    uint16_t *qh = a->qhat + ((b * Ns + s) * H + h) * d;
    float *os = a->o + ((b * Ns + s) * H + h) * d;
    float *zs = a->z + (b * H + h) * Ns + s;
    double m = 0.0;
    for (int64_t x = 0; x < d; ++x) u[x] = 0.0;
    if (a->first) {
        m = 1.0;
        for (int64_t t = 0; t < ns; ++t) p[t] = 0.0;
    } else {
        for (int64_t t = 0; t < ns; ++t) {
            int64_t j = Sb[t];
            const uint16_t *kj = a->k_old + ((b * Nk + j) * H + h) * d;
            const uint16_t *vj = a->v_old + ((b * Nk + j) * H + h) * d;
            double dot = 0.0;
            for (int64_t x = 0; x < d; ++x)
                dot += (double)orc_bf16_to_f32(qh[x]) * (double)orc_bf16_to_f32(kj[x]);
            p[t] = exp(dot * inv_sqrt_d - (double)*zs);
            m += p[t];
            for (int64_t x = 0; x < d; ++x) u[x] += p[t] * (double)orc_bf16_to_f32(vj[x]);
        }
        if (!(m >= (double)FLT_MIN)) return;     /* R3: old mass underflowed */
    }
    double mx = -INFINITY;
    for (int64_t t = 0; t < ns; ++t) {
        int64_t j = Sb[t];
        const uint16_t *kj = a->k_new + ((b * Nk + j) * H + h) * d;
        double dot = 0.0;
        for (int64_t x = 0; x < d; ++x)
            dot += (double)orc_bf16_to_f32(qs[x]) * (double)orc_bf16_to_f32(kj[x]);
        tau[t] = dot * inv_sqrt_d;
        if (tau[t] > mx) mx = tau[t];
    }
    double sum = 0.0;
    for (int64_t t = 0; t < ns; ++t) sum += exp(tau[t] - mx);
    double lam = mx + log(sum);
    for (int64_t x = 0; x < d; ++x) w[x] = 0.0;
    for (int64_t t = 0; t < ns; ++t) {
        int64_t j = Sb[t];
        const uint16_t *vj = a->v_new + ((b * Nk + j) * H + h) * d;
        double e = exp(tau[t] - lam);
        for (int64_t x = 0; x < d; ++x) w[x] += e * (double)orc_bf16_to_f32(vj[x]);
        dc[t] += m * e - p[t];
    }
    for (int64_t x = 0; x < d; ++x) {
        double prev = a->first ? 0.0 : (double)os[x];
        os[x] = (float)(prev - u[x] + m * w[x]);
    }
    *zs = (float)(lam - log(m));
    for (int64_t x = 0; x < d; ++x) qh[x] = qs[x];
    if (a->m_out) a->m_out[(b * H + h) * a->R + r] = m;
}

static void orc_apply_dc(const orc_attn_args *a, int64_t b, int64_t h, float *c, const double *dc) {
    const int32_t *Sb = a->S + (b * a->H + h) * a->K;
    float *cb = c + (b * a->H + h) * a->Nk;
    if (a->first) for (int64_t j = 0; j < a->Nk; ++j) cb[j] = 0.0f;
    for (int64_t t = 0; t < a->K; ++t) cb[Sb[t]] = (float)((double)cb[Sb[t]] + dc[t]);
}

void orc_attention(int first, int64_t B, int64_t H, int64_t d, int64_t Nk, int64_t Ns,
                   int64_t R, const int32_t *pos, const int32_t *slot,
                   const uint16_t *q, uint16_t *qhat, float *o, float *z, float *c,
                   int64_t K, const int32_t *S,
                   const uint16_t *k_old, const uint16_t *v_old,
                   const uint16_t *k_new, const uint16_t *v_new,
                   const uint8_t *bh_mask, double *m_out) {
    orc_attn_args a = {first, B, H, d, Nk, Ns, R, K, pos, slot, q, qhat, o, z, S,
                       k_old, v_old, k_new, v_new, m_out};
    int nthreads = omp_get_max_threads();
    int64_t n_bh = 0;
    for (int64_t bh = 0; bh < B * H; ++bh) n_bh += (!bh_mask || bh_mask[bh]);
    if (n_bh >= nthreads) {
        /* enough (b, h) pairs to keep every thread busy: one pair per task */
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < B * H; ++bh) {
            if (bh_mask && !bh_mask[bh]) continue;
            double *dc = (double *)calloc((size_t)K, sizeof(double));
            double *p = (double *)malloc(sizeof(double) * (size_t)(K + 1));
            double *tau = (double *)malloc(sizeof(double) * (size_t)(K + 1));
            double *u = (double *)malloc(sizeof(double) * (size_t)d);
            double *w = (double *)malloc(sizeof(double) * (size_t)d);
            for (int64_t r = 0; r < R; ++r) orc_attention_row(&a, bh / H, bh % H, r, dc, p, tau, u, w);
            orc_apply_dc(&a, bh / H, bh % H, c, dc);
            free(dc); free(p); free(tau); free(u); free(w);
        }
        return;
    }
    /* few (b, h) pairs: split the rows of each pair across threads; each
     * thread sums its rows' column-mass changes, and the per-thread sums are
     * added in thread order */
    double *dc_all = (double *)calloc((size_t)nthreads * (size_t)K, sizeof(double));
    for (int64_t bh = 0; bh < B * H; ++bh) {
        if (bh_mask && !bh_mask[bh]) continue;
        memset(dc_all, 0, sizeof(double) * (size_t)nthreads * (size_t)K);
#pragma omp parallel num_threads(nthreads)
        {
            int t = omp_get_thread_num();
            double *dc = dc_all + (size_t)t * (size_t)K;
            double *p = (double *)malloc(sizeof(double) * (size_t)(K + 1));
            double *tau = (double *)malloc(sizeof(double) * (size_t)(K + 1));
            double *u = (double *)malloc(sizeof(double) * (size_t)d);
            double *w = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static, 16)
            for (int64_t r = 0; r < R; ++r) orc_attention_row(&a, bh / H, bh % H, r, dc, p, tau, u, w);
            free(p); free(tau); free(u); free(w);
        }
        for (int t = 1; t < nthreads; ++t)
            for (int64_t k = 0; k < K; ++k) dc_all[k] += dc_all[(size_t)t * (size_t)K + k];
        orc_apply_dc(&a, bh / H, bh % H, c, dc_all);
    }
    free(dc_all);
}

/* Textbook causal softmax attention in double (used to pin the lazy
 * attention above in its full-set special case). q,k,v [B,N,H,d] bf16;
 * o [B,N,H,d] double; lse [B,H,N] double. */
void orc_softmax_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           int64_t B, int64_t N, int64_t H, int64_t d, double *o, double *lse) {
    const double sc = 1.0 / sqrt((double)d);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            double *lg = (double *)malloc(sizeof(double) * (size_t)N);
            for (int64_t i = 0; i < N; ++i) {
                const uint16_t *qi = q + ((b * N + i) * H + h) * d;
                double mx = -INFINITY;
                for (int64_t j = 0; j <= i; ++j) {
                    const uint16_t *kj = k + ((b * N + j) * H + h) * d;
                    double dot = 0.0;
                    for (int64_t x = 0; x < d; ++x)
                        dot += (double)orc_bf16_to_f32(qi[x]) * (double)orc_bf16_to_f32(kj[x]);
                    lg[j] = dot * sc;
                    if (lg[j] > mx) mx = lg[j];
                }
                double den = 0.0;
                for (int64_t j = 0; j <= i; ++j) den += exp(lg[j] - mx);
                double *oi = o + ((b * N + i) * H + h) * d;
                for (int64_t x = 0; x < d; ++x) oi[x] = 0.0;
                for (int64_t j = 0; j <= i; ++j) {
                    const uint16_t *vj = v + ((b * N + j) * H + h) * d;
                    double pj = exp(lg[j] - mx) / den;
                    for (int64_t x = 0; x < d; ++x) oi[x] += pj * (double)orc_bf16_to_f32(vj[x]);
                }
                lse[(b * H + h) * N + i] = mx + log(den);
            }
            free(lg);
        }
    }
}

/* Round doubles to bfloat16 (8 significant bits, exponent range of binary32),
 * to nearest, ties to even, in ONE step (no intermediate binary32 rounding,
 * which could round a value just above a bf16 tie down to the tie and then to
 * even). Overflow gives infinity; NaN gives the canonical quiet NaN. */
void orc_round_bf16(const double *x, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) {
        const double v = x[i];
        double r;
        if (isnan(v)) {
            out[i] = 0x7FC0u;
            continue;
        }
        if (v == 0.0 || isinf(v)) {
            r = v;
        } else if (fabs(v) < ldexp(1.0, -126)) {   /* subnormal range: spacing 2^-133 */
            r = ldexp(rint(ldexp(v, 133)), -133);
        } else {
            int e;
            const double m = frexp(v, &e);        /* v = m 2^e, 0.5 <= |m| < 1 */
            r = ldexp(rint(ldexp(m, 8)), e - 8);  /* 8 significant bits */
            if (fabs(r) >= ldexp(1.0, 128)) r = v > 0 ? INFINITY : -INFINITY;
        }
        const float f = (float)r;                 /* exact: every bf16 value is a binary32 value */
        uint32_t u;
        memcpy(&u, &f, 4);
        out[i] = (uint16_t)(u >> 16);
    }
}

/* OpenMP threads of the parallel regions above, for timing the oracle on one
 * core or on all of them. Results do not depend on it except through the
 * order in which per-thread column-mass sums are added (in double). */
void orc_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
int orc_get_threads(void) { return omp_get_max_threads(); }
