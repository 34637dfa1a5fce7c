/*
 * oscar_oracle.c -- plain, slow, float64 CPU oracle for the OSCAR 2-bit
 * KV-cache hot path (eviction into INT2 history; decode attention over the
 * three-segment pool).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; it re-derives every step from the method description and
 * from the pool format stated below (which the library documents
 * independently in its public header).
 *
 * Sources (page title, then section):
 *   [NEWS]  "卓绝TurboQuant：Together AI把2-bit KV Cache推向实在行状"
 *           (www.sanyangsrq.com news article on OSCAR; the text is a
 *           synonym-spun copy of a Chinese write-up).
 *           sec. A = "不是更会'压缩向量'，而是运转保护 attention"
 *           sec. B = "OSCAR 把旋转瞄准 attention" (rotation formula)
 *           sec. C = figure "从离线校准到在线推理的 pipeline" and the
 *                    serving-path text under it
 *   [HOME]  "Zhongzhu (Charlie) Zhou" home page, Featured Projects,
 *           "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
 *           Cache Quantization".
 *
 * Readings taken where the pages are silent (each listed in the design
 * notes): row-vector convention (y = x.R); Sylvester-ordered orthonormal
 * Hadamard; groups of g consecutive *stored* (post bit-reversal) positions;
 * symmetric clip to +-c*max|y| per group; asymmetric fp16 scale/zero with
 * zero = clipped minimum and scale = (max-min)/3; codes from the stored
 * fp16 scale/zero with round-half-even; all-zero codes when the fp16 scale
 * is 0; four codes per byte, byte j holding stored positions j, j + d/4,
 * j + 2d/4, j + 3d/4 in bits 0-1, 2-3, 4-5, 6-7 (the pages fix only that
 * four codes share a byte; with d = 128 and g = 32 a byte then holds in-group index
 * j of each of the four groups); attention with the softmax scale given by
 * the caller.
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Status codes (same meaning as the library's; values restated here). */
#define ORC_OK 0
#define ORC_ERR_INVALID_ARG 1
#define ORC_ERR_UNSUPPORTED 2
#define ORC_ERR_OUT_OF_PAGES 3

typedef struct {
    int32_t head_dim;     /* d */
    int32_t quant_group;  /* g: elements per scale/zero group */
    int32_t sink;         /* BF16 sink tokens (64) */
    int32_t recent;       /* BF16 recent-window tokens (256) */
    int32_t page_size;    /* tokens per history page (64) */
    int32_t num_q_heads;  /* Hq */
    int32_t num_kv_heads; /* Hk */
} oracle_shape;

static int ilog2_exact(int v) {
    int b = 0;
    if (v <= 0) return -1;
    while ((1 << b) < v) ++b;
    return ((1 << b) == v) ? b : -1;
}

static int shape_ok(const oracle_shape* s) {
    if (!s) return 0;
    if (ilog2_exact(s->head_dim) < 2 || s->head_dim > 1024) return 0;
    if (s->quant_group <= 0 || s->head_dim % s->quant_group) return 0;
    if (s->quant_group % 4) return 0;
    if (s->page_size <= 0 || s->sink < 0 || s->recent < 0) return 0;
    if (s->num_kv_heads <= 0 || s->num_q_heads <= 0) return 0;
    if (s->num_q_heads % s->num_kv_heads) return 0;
    return 1;
}

/* ------------------------------------------------------------------ */
/* Rotation R = U . Hadamard . bit-reversal  ([NEWS] sec. B)          */
/* ------------------------------------------------------------------ */

/* Reverse the low nbits bits of j. */
int oracle_bitrev(int j, int nbits) {
    int r = 0;
    for (int b = 0; b < nbits; ++b)
        if (j & (1 << b)) r |= 1 << (nbits - 1 - b);
    return r;
}

static int popcount_u(unsigned v) {
    int c = 0;
    while (v) { c += (int)(v & 1u); v >>= 1; }
    return c;
}

/* Orthonormal Hadamard matrix in Sylvester (natural) order:
 * H[i][j] = (-1)^popcount(i & j) / sqrt(d).  Row-major d x d. */
void oracle_hadamard(int d, double* H) {
    double c = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            H[(size_t)i * d + j] = (popcount_u((unsigned)(i & j)) & 1) ? -c : c;
}

/* R = U . H . P with P the bit-reversal permutation matrix:
 * P[l][j] = 1 iff l = bitrev(j), so (v.P)[j] = v[bitrev(j)].
 * U, R row-major d x d; a row vector x is rotated as y = x . R. */
void oracle_build_R(int d, const double* U, double* R) {
    int nb = ilog2_exact(d);
    double* H = (double*)malloc(sizeof(double) * d * d);
    double* UH = (double*)malloc(sizeof(double) * d * d);
    oracle_hadamard(d, H);
    for (int i = 0; i < d; ++i)
        for (int l = 0; l < d; ++l) {
            double acc = 0.0;
            for (int k = 0; k < d; ++k) acc += U[(size_t)i * d + k] * H[(size_t)k * d + l];
            UH[(size_t)i * d + l] = acc;
        }
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            R[(size_t)i * d + j] = UH[(size_t)i * d + oracle_bitrev(j, nb)];
    free(H);
    free(UH);
}

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* IEEE binary16 from float64, round to nearest, ties to even, overflow to
 * infinity, subnormals kept.  Written from the binary16 definition. */
uint16_t oracle_f16_from_f64(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = m * 2^-24, m in [0, 1024] */
        double m = nearbyint(ldexp(a, 24)); /* default mode: ties to even */
        return (uint16_t)(sign | (uint16_t)m); /* m == 1024 is the smallest normal */
    }
    int e2;
    (void)frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;      /* a in [2^E, 2^(E+1)) */
    double m = nearbyint((ldexp(a, -E) - 1.0) * 1024.0);
    if (m >= 1024.0) { m = 0.0; E += 1; }
    if (E > 15) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)m);
}

double oracle_f64_from_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int E = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (E == 0) v = ldexp((double)m, -24);
    else if (E == 31) v = m ? NAN : INFINITY;
    else v = ldexp(1.0 + m / 1024.0, E - 15);
    return sign ? -v : v;
}

/* bfloat16 bits -> float64 (exact): the bf16 pattern is the top half of a
 * binary32 pattern. */
double oracle_f64_from_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Four 2-bit codes share one byte ([NEWS] sec. C, the storage note under
 * the pipeline figure); code i in bits 2i..2i+1. */
uint8_t oracle_pack4(const uint8_t* c) {
    return (uint8_t)((c[0] & 3u) | ((c[1] & 3u) << 2) | ((c[2] & 3u) << 4) | ((c[3] & 3u) << 6));
}

void oracle_unpack4(uint8_t byte, uint8_t* c) {
    for (int i = 0; i < 4; ++i) c[i] = (uint8_t)((byte >> (2 * i)) & 3u);
}

/* ------------------------------------------------------------------ */
/* Clip + INT2 asymmetric group quantisation ([NEWS] sec. A: 4 discrete */
/* levels; sec. C: rotate, clip, quantize, pack; scale/zero-point)      */
/* ------------------------------------------------------------------ */

/* y: d values in stored order (already rotated and bit-reversed).
 * For each group k of g consecutive stored positions:
 *   t = clip * max|y|;  yc = min(max(y, -t), t)
 *   s16 = fp16(( max yc - min yc ) / 3),  z16 = fp16(min yc)
 *   code = 0 if s == 0, else clamp(round_half_even((yc - z) / s), 0, 3)
 * Outputs: codes[d] (0..3), s16[d/g], z16[d/g]; optional u[d] (the
 * pre-rounding (yc-z)/s, 0 where s == 0), s_pre[d/g], z_pre[d/g] (the
 * float64 values before fp16 rounding). */
void oracle_quantize_vec(int d, int g, const double* y, double clip, uint8_t* codes,
                         uint16_t* s16, uint16_t* z16, double* u, double* s_pre, double* z_pre) {
    int ng = d / g;
    for (int k = 0; k < ng; ++k) {
        const double* yg = y + (size_t)k * g;
        double amax = 0.0;
        for (int j = 0; j < g; ++j) amax = fmax(amax, fabs(yg[j]));
        double t = clip * amax;
        double lo = INFINITY, hi = -INFINITY;
        for (int j = 0; j < g; ++j) {
            double yc = fmin(fmax(yg[j], -t), t);
            lo = fmin(lo, yc);
            hi = fmax(hi, yc);
        }
        double sp = (hi - lo) / 3.0, zp = lo;
        uint16_t sh = oracle_f16_from_f64(sp), zh = oracle_f16_from_f64(zp);
        double s = oracle_f64_from_f16(sh), z = oracle_f64_from_f16(zh);
        s16[k] = sh;
        z16[k] = zh;
        if (s_pre) s_pre[k] = sp;
        if (z_pre) z_pre[k] = zp;
        for (int j = 0; j < g; ++j) {
            double yc = fmin(fmax(yg[j], -t), t);
            double uj = 0.0;
            int c = 0;
            if (s != 0.0) {
                uj = (yc - z) / s;
                double r = nearbyint(uj);
                if (r < 0.0) r = 0.0;
                if (r > 3.0) r = 3.0;
                c = (int)r;
            }
            codes[(size_t)k * g + j] = (uint8_t)c;
            if (u) u[(size_t)k * g + j] = uj;
        }
    }
}

/* yhat[j] = s * code[j] + z, stored order. */
void oracle_dequantize_vec(int d, int g, const uint8_t* codes, const uint16_t* s16,
                           const uint16_t* z16, double* yhat) {
    for (int j = 0; j < d; ++j) {
        int k = j / g;
        yhat[j] = oracle_f64_from_f16(s16[k]) * (double)codes[j] + oracle_f64_from_f16(z16[k]);
    }
}

/* ------------------------------------------------------------------ */
/* Pool format (paged INT2 history, [NEWS] sec. C + paged-KV remark)   */
/*                                                                     */
/* One block per (page, kv head), at byte offset                       */
/*   (page * Hk + kv) * block_bytes,                                   */
/* block_bytes = 2*P*d/4 + 2*P*(d/g)*4  (P = page_size):               */
/*   [0, P*d/4)            K codes, token-major: byte t*(d/4)+j        */
/*   [P*d/4, 2*P*d/4)      V codes, byte-plane-major: byte j*P+t       */
/*   next P*(d/g)*4 bytes  K (s,z): at (t*(d/g)+k)*4, fp16 s then z,   */
/*                         little-endian                               */
/*   next P*(d/g)*4 bytes  V (s,z), same arrangement                   */
/* where t = token slot in the page, j = code byte (stored positions   */
/* j + i*d/4 in bits 2i..2i+1, i = 0..3), k = group.  History position */
/* pos of sequence b lives in page page_table[b*max_pages + pos/P],    */
/* slot pos%P.                                                         */
/* ------------------------------------------------------------------ */

size_t oracle_block_bytes(int d, int g, int P) {
    return (size_t)2 * P * (d / 4) + (size_t)2 * P * (d / g) * 4;
}

static void store_u16le(uint8_t* p, uint16_t v) {
    p[0] = (uint8_t)(v & 0xFF);
    p[1] = (uint8_t)(v >> 8);
}

static uint16_t load_u16le(const uint8_t* p) {
    return (uint16_t)(p[0] | (p[1] << 8));
}

/* Write one quantised token-vector into its block. which: 0 = K, 1 = V. */
static void pool_write(uint8_t* block, int d, int g, int P, int slot, int which,
                       const uint8_t* codes, const uint16_t* s16, const uint16_t* z16) {
    int nbytes = d / 4, ng = d / g;
    size_t codes_bytes = (size_t)P * nbytes;
    size_t sz_bytes = (size_t)P * ng * 4;
    for (int j = 0; j < nbytes; ++j) {
        uint8_t four[4];
        for (int i = 0; i < 4; ++i) four[i] = codes[j + i * nbytes];
        uint8_t byte = oracle_pack4(four);
        if (which == 0) block[(size_t)slot * nbytes + j] = byte;
        else block[codes_bytes + (size_t)j * P + slot] = byte;
    }
    uint8_t* sz = block + 2 * codes_bytes + (size_t)which * sz_bytes;
    for (int k = 0; k < ng; ++k) {
        store_u16le(sz + ((size_t)slot * ng + k) * 4, s16[k]);
        store_u16le(sz + ((size_t)slot * ng + k) * 4 + 2, z16[k]);
    }
}

/* Read back the dequantised stored-order vector of one token-vector. */
static void pool_read(const uint8_t* block, int d, int g, int P, int slot, int which, double* yhat) {
    int nbytes = d / 4, ng = d / g;
    size_t codes_bytes = (size_t)P * nbytes;
    size_t sz_bytes = (size_t)P * ng * 4;
    uint8_t codes[1024];
    uint16_t s16[256], z16[256];
    for (int j = 0; j < nbytes; ++j) {
        uint8_t byte = (which == 0) ? block[(size_t)slot * nbytes + j]
                                    : block[codes_bytes + (size_t)j * P + slot];
        uint8_t four[4];
        oracle_unpack4(byte, four);
        for (int i = 0; i < 4; ++i) codes[j + i * nbytes] = four[i];
    }
    const uint8_t* sz = block + 2 * codes_bytes + (size_t)which * sz_bytes;
    for (int k = 0; k < ng; ++k) {
        s16[k] = load_u16le(sz + ((size_t)slot * ng + k) * 4);
        z16[k] = load_u16le(sz + ((size_t)slot * ng + k) * 4 + 2);
    }
    oracle_dequantize_vec(d, g, codes, s16, z16, yhat);
}

/* ------------------------------------------------------------------ */
/* Eviction ([NEWS] sec. C: the oldest recent token is rotated,        */
/* clipped, quantised and packed, then moved into the INT2 history)    */
/* ------------------------------------------------------------------ */

/* src_kv: bf16 bits, rows of [Hk][2][d] (K then V); token i reads row
 *   src_row ? src_row[i] : i.
 * U: float64 [Hk][2][d][d] (U_K, U_V per KV head); clip: [Hk][2].
 * dst_seq, dst_pos: history position each token is written to.
 * u_out (nullable): [n_tok][Hk][2][d] pre-rounding code values;
 * s_pre/z_pre (nullable): [n_tok][Hk][2][d/g] pre-fp16 scale and zero. */
int oracle_evict(const oracle_shape* sh, int n_tok, const uint16_t* src_kv, const int32_t* src_row,
                 const int32_t* dst_seq, const int32_t* dst_pos, const double* U, const double* clip,
                 uint8_t* pool, const int32_t* page_table, int max_pages, double* u_out,
                 double* s_pre, double* z_pre) {
    if (!shape_ok(sh) || n_tok < 0 || !src_kv || !dst_seq || !dst_pos || !U || !clip || !pool ||
        !page_table || max_pages <= 0)
        return ORC_ERR_INVALID_ARG;
    int d = sh->head_dim, g = sh->quant_group, P = sh->page_size, Hk = sh->num_kv_heads;
    int ng = d / g;
    size_t bb = oracle_block_bytes(d, g, P);
    for (int i = 0; i < n_tok; ++i)
        if (dst_pos[i] < 0 || dst_pos[i] / P >= max_pages || dst_seq[i] < 0) return ORC_ERR_INVALID_ARG;

    double* R = (double*)malloc(sizeof(double) * (size_t)Hk * 2 * d * d);
    for (int h = 0; h < Hk * 2; ++h) oracle_build_R(d, U + (size_t)h * d * d, R + (size_t)h * d * d);

    int n_units = n_tok * Hk * 2;
#pragma omp parallel for schedule(dynamic, 4)
    for (int unit = 0; unit < n_units; ++unit) {
        int i = unit / (Hk * 2), kv = (unit / 2) % Hk, which = unit % 2;
        long row = src_row ? src_row[i] : i;
        const uint16_t* x = src_kv + ((size_t)row * Hk * 2 + (size_t)kv * 2 + which) * d;
        const double* Rm = R + ((size_t)kv * 2 + which) * d * d;
        double xd[1024], y[1024];
        uint8_t codes[1024];
        uint16_t s16[256], z16[256];
        for (int a = 0; a < d; ++a) xd[a] = oracle_f64_from_bf16(x[a]);
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int a = 0; a < d; ++a) acc += xd[a] * Rm[(size_t)a * d + j];
            y[j] = acc;
        }
        size_t off = ((size_t)i * Hk + kv) * 2 + which;
        oracle_quantize_vec(d, g, y, (double)clip[kv * 2 + which], codes, s16, z16,
                            u_out ? u_out + off * d : NULL, s_pre ? s_pre + off * ng : NULL,
                            z_pre ? z_pre + off * ng : NULL);
        int page = page_table[(size_t)dst_seq[i] * max_pages + dst_pos[i] / P];
        uint8_t* block = pool + ((size_t)page * Hk + kv) * bb;
        pool_write(block, d, g, P, dst_pos[i] % P, which, codes, s16, z16);
    }
    free(R);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Decode attention: plain definition                                  */
/* out[b,h] = softmax_t(sm_scale * q[b,h] . k_t) . V over the          */
/* concatenation of the BF16 tokens (sink + recent window) and the     */
/* dequantised INT2 history mapped back by R^T ([NEWS] sec. C).        */
/* ------------------------------------------------------------------ */

static int decode_args_ok(const oracle_shape* sh, int batch, const uint16_t* q,
                          const uint16_t* bf16_kv, const int32_t* bf16_len, const uint8_t* pool,
                          const int32_t* page_table, int max_pages, const int32_t* hist_len,
                          const double* U, const double* out) {
    if (!shape_ok(sh) || batch < 0 || !q || !bf16_kv || !bf16_len || !hist_len || !U || !out)
        return 0;
    int nslot = sh->sink + sh->recent;
    for (int b = 0; b < batch; ++b) {
        if (bf16_len[b] < 0 || bf16_len[b] > nslot || hist_len[b] < 0) return 0;
        if (hist_len[b] > 0 &&
            (!pool || !page_table || max_pages <= 0 || (hist_len[b] - 1) / sh->page_size >= max_pages))
            return 0;
    }
    return 1;
}

/* q: bf16 [B][Hq][d]; bf16_kv: bf16 [B][sink+recent][Hk][2][d], slots
 * [0, bf16_len[b]) valid; pool/page_table as above; hist_len[b] history
 * tokens at positions [0, hist_len[b]); U float64 [Hk][2][d][d].
 * out: float64 [B][Hq][d] (zeros for an empty context).
 * unit_mask (nullable): [B][Hk]; units with mask 0 are skipped (their
 * outputs are left untouched), so a test can check a sample of a large
 * batch. */
int oracle_decode(const oracle_shape* sh, int batch, const uint16_t* q, const uint16_t* bf16_kv,
                  const int32_t* bf16_len, const uint8_t* pool, const int32_t* page_table,
                  int max_pages, const int32_t* hist_len, const double* U, double sm_scale,
                  const uint8_t* unit_mask, double* out) {
    if (!decode_args_ok(sh, batch, q, bf16_kv, bf16_len, pool, page_table, max_pages, hist_len, U, out))
        return ORC_ERR_INVALID_ARG;
    int d = sh->head_dim, g = sh->quant_group, P = sh->page_size, Hk = sh->num_kv_heads;
    int Hq = sh->num_q_heads, G = Hq / Hk, nslot = sh->sink + sh->recent;
    size_t bb = oracle_block_bytes(d, g, P);
    double* R = (double*)malloc(sizeof(double) * (size_t)Hk * 2 * d * d);
    for (int h = 0; h < Hk * 2; ++h) oracle_build_R(d, U + (size_t)h * d * d, R + (size_t)h * d * d);

#pragma omp parallel for schedule(dynamic, 1)
    for (int unit = 0; unit < batch * Hk; ++unit) {
        if (unit_mask && !unit_mask[unit]) continue;
        int b = unit / Hk, kv = unit % Hk;
        int nb = bf16_len[b], nh = hist_len[b], n = nb + nh;
        const double* RK = R + ((size_t)kv * 2 + 0) * d * d;
        const double* RV = R + ((size_t)kv * 2 + 1) * d * d;
        double* K = (double*)malloc(sizeof(double) * ((size_t)n + 1) * d);
        double* V = (double*)malloc(sizeof(double) * ((size_t)n + 1) * d);
        double* logit = (double*)malloc(sizeof(double) * ((size_t)n + 1));
        double yh[1024];
        /* BF16 tokens, unrotated */
        for (int t = 0; t < nb; ++t) {
            const uint16_t* base = bf16_kv + (((size_t)b * nslot + t) * Hk + kv) * 2 * d;
            for (int a = 0; a < d; ++a) {
                K[(size_t)t * d + a] = oracle_f64_from_bf16(base[a]);
                V[(size_t)t * d + a] = oracle_f64_from_bf16(base[d + a]);
            }
        }
        /* INT2 history: dequantise (rotated domain), then map back by R^T:
         * x_a = sum_j yhat_j R[a][j]. */
        for (int pos = 0; pos < nh; ++pos) {
            int page = page_table[(size_t)b * max_pages + pos / P];
            const uint8_t* block = pool + ((size_t)page * Hk + kv) * bb;
            double* kr = K + (size_t)(nb + pos) * d;
            double* vr = V + (size_t)(nb + pos) * d;
            pool_read(block, d, g, P, pos % P, 0, yh);
            for (int a = 0; a < d; ++a) {
                double acc = 0.0;
                for (int j = 0; j < d; ++j) acc += yh[j] * RK[(size_t)a * d + j];
                kr[a] = acc;
            }
            pool_read(block, d, g, P, pos % P, 1, yh);
            for (int a = 0; a < d; ++a) {
                double acc = 0.0;
                for (int j = 0; j < d; ++j) acc += yh[j] * RV[(size_t)a * d + j];
                vr[a] = acc;
            }
        }
        for (int hh = 0; hh < G; ++hh) {
            int h = kv * G + hh;
            const uint16_t* qb = q + ((size_t)b * Hq + h) * d;
            double qd[1024];
            for (int a = 0; a < d; ++a) qd[a] = oracle_f64_from_bf16(qb[a]);
            double* o = out + ((size_t)b * Hq + h) * d;
            for (int a = 0; a < d; ++a) o[a] = 0.0;
            if (n == 0) continue;
            double m = -INFINITY;
            for (int t = 0; t < n; ++t) {
                double acc = 0.0;
                for (int a = 0; a < d; ++a) acc += qd[a] * K[(size_t)t * d + a];
                logit[t] = sm_scale * acc;
                m = fmax(m, logit[t]);
            }
            double l = 0.0;
            for (int t = 0; t < n; ++t) {
                double p = exp(logit[t] - m);
                l += p;
                for (int a = 0; a < d; ++a) o[a] += p * V[(size_t)t * d + a];
            }
            for (int a = 0; a < d; ++a) o[a] /= l;
        }
        free(K);
        free(V);
        free(logit);
    }
    free(R);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Decode attention in the pages' segmented form ([NEWS] sec. C):     */
/* the INT2 segment attends in the rotated domain (q' = q.R_K, values */
/* kept rotated, output mapped back by R_V^T), the BF16 segment       */
/* attends unrotated, and the two partial softmaxes are merged by      */
/* their log-sum-exp.  Equal to oracle_decode up to rounding.          */
/* ------------------------------------------------------------------ */
int oracle_decode_segmented(const oracle_shape* sh, int batch, const uint16_t* q,
                            const uint16_t* bf16_kv, const int32_t* bf16_len, const uint8_t* pool,
                            const int32_t* page_table, int max_pages, const int32_t* hist_len,
                            const double* U, double sm_scale, double* out) {
    if (!decode_args_ok(sh, batch, q, bf16_kv, bf16_len, pool, page_table, max_pages, hist_len, U, out))
        return ORC_ERR_INVALID_ARG;
    int d = sh->head_dim, g = sh->quant_group, P = sh->page_size, Hk = sh->num_kv_heads;
    int Hq = sh->num_q_heads, G = Hq / Hk, nslot = sh->sink + sh->recent;
    size_t bb = oracle_block_bytes(d, g, P);
    double* R = (double*)malloc(sizeof(double) * (size_t)Hk * 2 * d * d);
    for (int h = 0; h < Hk * 2; ++h) oracle_build_R(d, U + (size_t)h * d * d, R + (size_t)h * d * d);

#pragma omp parallel for schedule(dynamic, 1)
    for (int unit = 0; unit < batch * Hq; ++unit) {
        int b = unit / Hq, h = unit % Hq, kv = h / G;
        const double* RK = R + ((size_t)kv * 2 + 0) * d * d;
        const double* RV = R + ((size_t)kv * 2 + 1) * d * d;
        double qd[1024], qr[1024], yk[1024], yv[1024], o_bf[1024], o_i2r[1024], o_i2[1024];
        const uint16_t* qb = q + ((size_t)b * Hq + h) * d;
        for (int a = 0; a < d; ++a) qd[a] = oracle_f64_from_bf16(qb[a]);
        /* q' = q . R_K */
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int a = 0; a < d; ++a) acc += qd[a] * RK[(size_t)a * d + j];
            qr[j] = acc;
        }
        /* BF16 segment */
        int nb = bf16_len[b];
        double m_bf = -INFINITY, l_bf = 0.0;
        for (int a = 0; a < d; ++a) o_bf[a] = 0.0;
        double* lg = (double*)malloc(sizeof(double) * ((size_t)nb + (size_t)hist_len[b] + 1));
        for (int t = 0; t < nb; ++t) {
            const uint16_t* base = bf16_kv + (((size_t)b * nslot + t) * Hk + kv) * 2 * d;
            double acc = 0.0;
            for (int a = 0; a < d; ++a) acc += qd[a] * oracle_f64_from_bf16(base[a]);
            lg[t] = sm_scale * acc;
            m_bf = fmax(m_bf, lg[t]);
        }
        for (int t = 0; t < nb; ++t) {
            const uint16_t* base = bf16_kv + (((size_t)b * nslot + t) * Hk + kv) * 2 * d;
            double p = exp(lg[t] - m_bf);
            l_bf += p;
            for (int a = 0; a < d; ++a) o_bf[a] += p * oracle_f64_from_bf16(base[d + a]);
        }
        /* INT2 segment, rotated domain */
        int nh = hist_len[b];
        double m_i2 = -INFINITY, l_i2 = 0.0;
        for (int a = 0; a < d; ++a) o_i2r[a] = 0.0;
        for (int pos = 0; pos < nh; ++pos) {
            int page = page_table[(size_t)b * max_pages + pos / P];
            const uint8_t* block = pool + ((size_t)page * Hk + kv) * bb;
            pool_read(block, d, g, P, pos % P, 0, yk);
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += qr[j] * yk[j];
            lg[pos] = sm_scale * acc;
            m_i2 = fmax(m_i2, lg[pos]);
        }
        for (int pos = 0; pos < nh; ++pos) {
            int page = page_table[(size_t)b * max_pages + pos / P];
            const uint8_t* block = pool + ((size_t)page * Hk + kv) * bb;
            pool_read(block, d, g, P, pos % P, 1, yv);
            double p = exp(lg[pos] - m_i2);
            l_i2 += p;
            for (int j = 0; j < d; ++j) o_i2r[j] += p * yv[j];
        }
        /* map the INT2 output back: o = o' . R_V^T, o_a = sum_j o'_j R[a][j] */
        for (int a = 0; a < d; ++a) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += o_i2r[j] * RV[(size_t)a * d + j];
            o_i2[a] = acc;
        }
        /* online-softmax (log-sum-exp) merge of the two partials */
        double* o = out + ((size_t)b * Hq + h) * d;
        double M = fmax(m_bf, m_i2);
        double w_bf = (l_bf > 0.0) ? exp(m_bf - M) : 0.0;
        double w_i2 = (l_i2 > 0.0) ? exp(m_i2 - M) : 0.0;
        double L = w_bf * l_bf + w_i2 * l_i2;
        for (int a = 0; a < d; ++a) o[a] = (L > 0.0) ? (w_bf * o_bf[a] + w_i2 * o_i2[a]) / L : 0.0;
        free(lg);
    }
    free(R);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Page-table layout (paged KV with shared prefix pages: [NEWS] sec. C,*/
/* compatibility with paged KV and the radix prefix cache)             */
/* ------------------------------------------------------------------ */

/* SplitMix64 (Steele, Lea, Flood 2014; constants as published by Vigna). */
static uint64_t splitmix64_next(uint64_t* state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* First n outputs of SplitMix64 started from state = seed (for pinning the
 * generator against its published test vector). */
void oracle_splitmix64(uint64_t seed, int n, uint64_t* out) {
    uint64_t st = seed;
    for (int i = 0; i < n; ++i) out[i] = splitmix64_next(&st);
}

/* Logical allocation order: for each prefix group in order of first
 * appearance, its shared pages; then, sequence by sequence, each
 * sequence's private pages.  With perm_seed != 0 the logical page L maps
 * to the physical page pi[L], pi = Fisher-Yates shuffle of the identity
 * driven by SplitMix64 seeded with perm_seed (for i = N-1 down to 1:
 * j = r mod (i+1), swap pi[i], pi[j]).  Unused table entries are -1. */
int oracle_pool_layout(const oracle_shape* sh, int batch, const int32_t* hist_capacity,
                       const int32_t* prefix_group, int shared_hist_tokens, uint64_t perm_seed,
                       int max_pages, int32_t* page_table, int32_t* num_pages_out,
                       uint64_t* pool_bytes_out) {
    if (!shape_ok(sh) || batch < 0 || !hist_capacity || !page_table || max_pages <= 0)
        return ORC_ERR_INVALID_ARG;
    int P = sh->page_size;
    if (shared_hist_tokens < 0 || shared_hist_tokens % P) return ORC_ERR_INVALID_ARG;
    int nshared = shared_hist_tokens / P;
    for (int b = 0; b < batch; ++b) {
        if (hist_capacity[b] < 0) return ORC_ERR_INVALID_ARG;
        if ((hist_capacity[b] + P - 1) / P > max_pages) return ORC_ERR_OUT_OF_PAGES;
        if (prefix_group && prefix_group[b] >= 0 && hist_capacity[b] < shared_hist_tokens)
            return ORC_ERR_INVALID_ARG;
    }
    for (size_t i = 0; i < (size_t)batch * max_pages; ++i) page_table[i] = -1;
    long next = 0;
    /* shared pages of each prefix group, in order of first appearance */
    for (int b = 0; b < batch; ++b) {
        if (!prefix_group || prefix_group[b] < 0) continue;
        int first = b;
        for (int c = 0; c < b; ++c)
            if (prefix_group[c] == prefix_group[b]) { first = c; break; }
        if (first == b) {
            for (int p = 0; p < nshared; ++p) page_table[(size_t)b * max_pages + p] = (int32_t)(next++);
        } else {
            for (int p = 0; p < nshared; ++p)
                page_table[(size_t)b * max_pages + p] = page_table[(size_t)first * max_pages + p];
        }
    }
    /* private pages */
    for (int b = 0; b < batch; ++b) {
        int need = (hist_capacity[b] + P - 1) / P;
        int start = (prefix_group && prefix_group[b] >= 0) ? nshared : 0;
        for (int p = start; p < need; ++p) page_table[(size_t)b * max_pages + p] = (int32_t)(next++);
    }
    if (perm_seed != 0 && next > 1) {
        int32_t* pi = (int32_t*)malloc(sizeof(int32_t) * (size_t)next);
        for (long i = 0; i < next; ++i) pi[i] = (int32_t)i;
        uint64_t st = perm_seed;
        for (long i = next - 1; i >= 1; --i) {
            uint64_t r = splitmix64_next(&st);
            long j = (long)(r % (uint64_t)(i + 1));
            int32_t tmp = pi[i];
            pi[i] = pi[j];
            pi[j] = tmp;
        }
        for (size_t i = 0; i < (size_t)batch * max_pages; ++i)
            if (page_table[i] >= 0) page_table[i] = pi[page_table[i]];
        free(pi);
    }
    if (num_pages_out) *num_pages_out = (int32_t)next;
    if (pool_bytes_out)
        *pool_bytes_out = (uint64_t)next * sh->num_kv_heads *
                          oracle_block_bytes(sh->head_dim, sh->quant_group, P);
    return ORC_OK;
}

/* Number of OpenMP threads the oracle will use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
