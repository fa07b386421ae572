/*
 * Engram memory read -- CPU oracle.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline /
 * reference legs may load this file's library.  It shares no code, header,
 * table or constant generator with the CUDA library; it is a plain,
 * single-threaded restatement of what the memory read computes, in double
 * precision, written for a reader to check against the sources by eye.
 *
 * Sources (DeepSeek-V4.1-Flash pages):
 *  - vramglass.com "deepseek-v4-1-flash-local-deployment", section "What
 *    makes up the 511 GB of weights?": hashed 2/3/4-gram tables, two modules
 *    with 8 hash heads each, 48 rows and about 12 KB read per token, row
 *    addresses that depend only on the input tokens.
 *  - rohitghumare.com "guides/deepseek-v4-1-flash", section "Engram: the
 *    table that is never multiplied": suffix n-grams of order 2, 3, 4, 8
 *    independent heads each, one row per (order, head), 24 rows per layer,
 *    48 per token, FP8 rows, a learned gate into the residual stream; section
 *    "The architecture": rows are added into the residual stream.
 *  The workload definition fixes the rest: the 64-bit mix chain, idx = h mod
 *  R, pad id V before a sequence start, 256 e4m3 values per row with one
 *  fp32 scale, per-module sums, the [T,512] bf16 concatenation, the 512 x d
 *  projection and the rmsnorm-sigmoid gate.
 *
 * Readings where the sources are silent (each also listed in the design
 * notes): ids enter the chain oldest first, zero-extended to 64 bits; the
 * shift in the mix is logical; table j = (module*3 + order-2)*8 + head; the
 * rmsnorm has no weight and eps is a parameter; y is not rounded before the
 * residual add; every sum here is taken in double.
 *
 * Exactness: a scale (fp32 in [0.5,2)) times an e4m3 value is a multiple of
 * 2^-33 below 2^10 in magnitude, so the 24-term module sums below are exact
 * in double; mem is the true value of the definition, not an fp32 rounding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_TABLES 48
#define ORC_TABLES_PER_MODULE 24
#define ORC_ROW 256
#define ORC_MEM 512

/* status codes returned by the oracle entry points */
#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ERANGE 3

/* Table j -> (module, order, head). */
static int table_module(int j) { return j / 24; }
static int table_order(int j) { return 2 + (j % 24) / 8; }

/* The 64-bit mix chain over the ids of one n-gram, oldest id first:
 * h <- (h xor id) * 0x9E3779B97F4A7C15 mod 2^64, then h <- h xor (h >> 29). */
uint64_t orc_mix_chain(uint64_t seed, const uint64_t *ids, int n) {
    uint64_t h = seed;
    for (int i = 0; i < n; ++i) {
        h = (h ^ ids[i]) * 0x9E3779B97F4A7C15ULL;
        h ^= h >> 29;
    }
    return h;
}

/* Sequence holding global position p (offs is ascending, n_seqs+1 long). */
static int64_t find_seq(const int64_t *offs, int64_t n_seqs, int64_t p) {
    for (int64_t s = 0; s < n_seqs; ++s)
        if (p >= offs[s] && p < offs[s + 1]) return s;
    return -1;
}

/* The 48 row indices of the token at global position p. */
static int hash_position(const int32_t *tokens, const int64_t *offs, int64_t n_seqs, int32_t V,
                         int64_t R, const uint64_t *seeds, int64_t p, int64_t *idx48) {
    int64_t s = find_seq(offs, n_seqs, p);
    if (s < 0) return ORC_ERANGE;
    int64_t start = offs[s];
    for (int j = 0; j < ORC_TABLES; ++j) {
        int n = table_order(j);
        uint64_t ids[4];
        for (int i = 0; i < n; ++i) {
            int64_t q = p - (n - 1) + i; /* oldest first */
            int32_t id = V;                  /* pad before the sequence start */
            if (q >= start) {
                id = tokens[q];
                if (id < 0 || id >= V) return ORC_ERANGE;
            }
            ids[i] = (uint64_t)(uint32_t)id; /* zero-extend */
        }
        uint64_t h = orc_mix_chain(seeds[j], ids, n);
        idx48[j] = (int64_t)(h % (uint64_t)R);
    }
    return ORC_OK;
}

/* idx for explicit global positions: idx[i][j] for positions[i]. */
int orc_hash_positions(const int32_t *tokens, const int64_t *offs, int64_t n_seqs, int32_t V,
                       int64_t R, const uint64_t *seeds, const int64_t *positions, int64_t n_pos,
                       int64_t *idx) {
    if (R < 1 || V < 0) return ORC_EINVAL;
    for (int64_t i = 0; i < n_pos; ++i) {
        int st = hash_position(tokens, offs, n_seqs, V, R, seeds, positions[i], idx + i * ORC_TABLES);
        if (st != ORC_OK) return st;
    }
    return ORC_OK;
}

/* idx for every query token: all positions (last_n == 0) or the last last_n
 * positions of each sequence, sequence by sequence. */
int orc_hash(const int32_t *tokens, const int64_t *offs, int64_t n_seqs, int32_t last_n, int32_t V,
             int64_t R, const uint64_t *seeds, int64_t *idx) {
    if (R < 1 || V < 0 || last_n < 0) return ORC_EINVAL;
    int64_t q = 0;
    for (int64_t s = 0; s < n_seqs; ++s) {
        int64_t lo = offs[s], hi = offs[s + 1];
        int64_t first = lo;
        if (last_n > 0) {
            if (hi - lo < last_n) return ORC_ERANGE;
            first = hi - last_n;
        }
        for (int64_t p = first; p < hi; ++p, ++q) {
            int st = hash_position(tokens, offs, n_seqs, V, R, seeds, p, idx + q * ORC_TABLES);
            if (st != ORC_OK) return st;
        }
    }
    return ORC_OK;
}

/* OCP 8-bit E4M3FN: sign, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities. */
double orc_e4m3_value(uint8_t code) {
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* One token: mem[256*m + c] = sum over the module's 24 tables, in ascending
 * j, of scale_j * value(row_j[c]).  rows[j] points at table j's row. */
static void reduce_token(const uint8_t *const *rows, const float *scale48, double *mem512) {
    for (int k = 0; k < ORC_MEM; ++k) mem512[k] = 0.0;
    for (int j = 0; j < ORC_TABLES; ++j) {
        int m = table_module(j);
        double sc = (double)scale48[j];
        for (int c = 0; c < ORC_ROW; ++c) mem512[ORC_ROW * m + c] += sc * orc_e4m3_value(rows[j][c]);
    }
}

/* OCP MX E8M0 scale byte: 2^(E - 127); E = 255 is NaN. */
double orc_e8m0_value(uint8_t e) {
    if (e == 255) return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* MXFP8-style rows (256 bytes of FP8 plus 8 bytes of scales per row,
 * "Engram: the table that is never multiplied"): code c of table j's row is
 * scaled by the E8M0 scale of its 32-code block, escale[j][c / 32].
 * mem[256*m + c] = sum over the module's 24 tables, ascending j. */
static void reduce_token_mx(const uint8_t *const *rows, const uint8_t *const *esc, double *mem512) {
    for (int k = 0; k < ORC_MEM; ++k) mem512[k] = 0.0;
    for (int j = 0; j < ORC_TABLES; ++j) {
        int m = table_module(j);
        for (int c = 0; c < ORC_ROW; ++c)
            mem512[ORC_ROW * m + c] += orc_e8m0_value(esc[j][c / 32]) * orc_e4m3_value(rows[j][c]);
    }
}

/* MX rows given explicitly: rows [T][48][256] codes, escales [T][48][8]. */
void orc_gather_reduce_mx_rows(const uint8_t *rows, const uint8_t *escales, int64_t T, double *mem) {
    for (int64_t t = 0; t < T; ++t) {
        const uint8_t *ptr[ORC_TABLES], *esc[ORC_TABLES];
        for (int j = 0; j < ORC_TABLES; ++j) {
            ptr[j] = rows + (t * ORC_TABLES + j) * ORC_ROW;
            esc[j] = escales + (t * ORC_TABLES + j) * 8;
        }
        reduce_token_mx(ptr, esc, mem + t * ORC_MEM);
    }
}

/* Gather from explicit rows: rows [T][48][256] bytes, scales [T][48]. */
void orc_gather_reduce_rows(const uint8_t *rows, const float *scales, int64_t T, double *mem) {
    for (int64_t t = 0; t < T; ++t) {
        const uint8_t *ptr[ORC_TABLES];
        for (int j = 0; j < ORC_TABLES; ++j) ptr[j] = rows + (t * ORC_TABLES + j) * ORC_ROW;
        reduce_token(ptr, scales + t * ORC_TABLES, mem + t * ORC_MEM);
    }
}

/* Gather from whole tables: tables [48][R][256], scales [48][R], idx [T][48]. */
int orc_gather_reduce(const uint8_t *tables, const float *scales, int64_t R, const int64_t *idx,
                      int64_t T, double *mem) {
    for (int64_t t = 0; t < T; ++t) {
        const uint8_t *ptr[ORC_TABLES];
        float sc[ORC_TABLES];
        for (int j = 0; j < ORC_TABLES; ++j) {
            int64_t r = idx[t * ORC_TABLES + j];
            if (r < 0 || r >= R) return ORC_ERANGE;
            ptr[j] = tables + ((int64_t)j * R + r) * ORC_ROW;
            sc[j] = scales[(int64_t)j * R + r];
        }
        reduce_token(ptr, sc, mem + t * ORC_MEM);
    }
    return ORC_OK;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double orc_bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to the nearest bfloat16, ties to even (one rounding).
 * Normal bf16 values in [2^e, 2^(e+1)) are spaced 2^(e-7); below 2^-126 the
 * spacing is the subnormal quantum 2^-133; results past the largest finite
 * value become infinity. */
uint16_t orc_bf16_rne(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e); /* a in [2^(e-1), 2^e) */
    int qexp = (e - 1 >= -126) ? (e - 1 - 7) : -133;
    double r = ldexp(nearbyint(ldexp(a, -qexp)), qexp); /* default mode: ties to even */
    const double bf16_max = ldexp(255.0, 127 - 7);      /* (2 - 2^-7) * 2^127 */
    if (r > bf16_max) return sign | 0x7F80;
    if (r < ldexp(1.0, -126)) return sign | (uint16_t)ldexp(r, 133); /* subnormal (or 0x80) */
    int e2;
    frexp(r, &e2); /* r in [2^(e2-1), 2^e2): field e2-1+127, significand r*2^(8-e2) in [128,256) */
    uint32_t sig = (uint32_t)ldexp(r, 8 - e2);
    return sign | (uint16_t)(((uint32_t)(e2 - 1 + 127) << 7) | (sig - 128));
}

/* The gated projection into the residual stream, in place on h.
 *   X      = bf16(mem)                                   [T,512]
 *   gate_t = sigmoid( <h_t / rms(h_t), g> / sqrt(d) ),  rms = sqrt(mean h^2 + eps)
 *   y      = X @ W_out                                   (double accumulation)
 *   h_t    = bf16(h_t + gate_t * y_t)
 * W [512][d], g [d], h [T][d] are bf16 bit patterns. gate_out may be NULL. */
int orc_fuse(const double *mem, const uint16_t *W, const uint16_t *g, uint16_t *h, int64_t T, int32_t d,
             double eps, double *gate_out) {
    if (d <= 0) return ORC_EINVAL;
    double X[ORC_MEM];
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    if (!y) return ORC_EINVAL;
    for (int64_t t = 0; t < T; ++t) {
        for (int k = 0; k < ORC_MEM; ++k) X[k] = orc_bf16_value(orc_bf16_rne(mem[t * ORC_MEM + k]));
        uint16_t *ht = h + t * (int64_t)d;
        double ss = 0.0, dot = 0.0;
        for (int c = 0; c < d; ++c) {
            double v = orc_bf16_value(ht[c]);
            ss += v * v;
            dot += v * orc_bf16_value(g[c]);
        }
        double rr = 1.0 / sqrt(ss / (double)d + eps);
        double gate = 1.0 / (1.0 + exp(-(rr * dot) / sqrt((double)d)));
        if (gate_out) gate_out[t] = gate;
        /* y_c = sum over k = 0..511 (ascending) of X_k * W[k][c] */
        for (int c = 0; c < d; ++c) y[c] = 0.0;
        for (int k = 0; k < ORC_MEM; ++k)
            for (int c = 0; c < d; ++c) y[c] += X[k] * orc_bf16_value(W[(int64_t)k * d + c]);
        for (int c = 0; c < d; ++c) ht[c] = orc_bf16_rne(orc_bf16_value(ht[c]) + gate * y[c]);
    }
    free(y);
    return ORC_OK;
}

/*
 * One Engram layer with a per-row, content-aware gate (rohitghumare.com
 * "guides/deepseek-v4-1-flash": section "The architecture", two layers, 1 and
 * 14, each adding looked-up rows into the residual stream through a learned
 * gate; section "Engram: the table that is never multiplied", 24 rows per
 * Engram layer and a gate that compares each retrieved row with the hidden
 * state and suppresses it when it contradicts the context).
 *
 * The pages give no gate formula; this is the plainest one that matches the
 * description (a reading, listed in the design notes): for each of the
 * layer's 24 rows r_j (dequantized, scale times e4m3 value),
 *   q   = rmsnorm(h) W_q            (W_q: d x 256)
 *   k_j = rmsnorm(r_j) W_k          (W_k: 256 x 256)
 *   g_j = sigmoid(<q, k_j> / sqrt(256))
 *   e   = sum_j g_j r_j             (in table order j)
 *   X   = bf16(e);  y = X W_m       (W_m: 256 x d)
 *   h   = bf16(h + y)
 * rmsnorm(v) = v / sqrt(mean(v^2) + eps), without a weight.  All sums in
 * double; weights and h are bf16 bit patterns.
 *
 * codes: e4m3 [T][24][256]; scales: fp32 [T][24]; h: bf16 [T][d], updated in
 * place; gates (optional): [T][24] out; e_out (optional): [T][256] out.
 * With MXFP8-style rows (orc_layer_gated_mx) r_j's code c is scaled by the
 * E8M0 scale of its 32-code block instead, escales [T][24][8].
 */
static int layer_gated(const uint8_t *codes, const float *scales, const uint8_t *escales, const uint16_t *Wq,
                       const uint16_t *Wk, const uint16_t *Wm, uint16_t *h, int64_t T, int32_t d, double eps,
                       double *gates, double *e_out);

int orc_layer_gated(const uint8_t *codes, const float *scales, const uint16_t *Wq, const uint16_t *Wk,
                    const uint16_t *Wm, uint16_t *h, int64_t T, int32_t d, double eps, double *gates,
                    double *e_out) {
    return layer_gated(codes, scales, NULL, Wq, Wk, Wm, h, T, d, eps, gates, e_out);
}

int orc_layer_gated_mx(const uint8_t *codes, const uint8_t *escales, const uint16_t *Wq, const uint16_t *Wk,
                       const uint16_t *Wm, uint16_t *h, int64_t T, int32_t d, double eps, double *gates,
                       double *e_out) {
    return layer_gated(codes, NULL, escales, Wq, Wk, Wm, h, T, d, eps, gates, e_out);
}

static int layer_gated(const uint8_t *codes, const float *scales, const uint8_t *escales, const uint16_t *Wq,
                       const uint16_t *Wk, const uint16_t *Wm, uint16_t *h, int64_t T, int32_t d, double eps,
                       double *gates, double *e_out) {
    enum { R = 256, J = 24 };
    if (d <= 0) return ORC_EINVAL;
    double *q = (double *)malloc(sizeof(double) * R);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    double *hv = (double *)malloc(sizeof(double) * (size_t)d);
    if (!q || !y || !hv) {
        free(q);
        free(y);
        free(hv);
        return ORC_EINVAL;
    }
    double v[R], k[R], e[R], X[R];
    for (int64_t t = 0; t < T; ++t) {
        uint16_t *ht = h + t * (int64_t)d;
        double ss = 0.0;
        for (int i = 0; i < d; ++i) {
            hv[i] = orc_bf16_value(ht[i]);
            ss += hv[i] * hv[i];
        }
        const double rh = 1.0 / sqrt(ss / (double)d + eps);
        for (int c = 0; c < R; ++c) q[c] = 0.0;
        for (int i = 0; i < d; ++i)
            for (int c = 0; c < R; ++c) q[c] += (hv[i] * rh) * orc_bf16_value(Wq[(int64_t)i * R + c]);
        for (int c = 0; c < R; ++c) e[c] = 0.0;
        for (int j = 0; j < J; ++j) {
            const uint8_t *row = codes + (t * J + j) * R;
            double vs = 0.0;
            for (int c = 0; c < R; ++c) {
                const double s = escales ? orc_e8m0_value(escales[(t * J + j) * 8 + c / 32]) : (double)scales[t * J + j];
                v[c] = s * orc_e4m3_value(row[c]);
                vs += v[c] * v[c];
            }
            const double rr = 1.0 / sqrt(vs / (double)R + eps);
            for (int c = 0; c < R; ++c) k[c] = 0.0;
            for (int i = 0; i < R; ++i)
                for (int c = 0; c < R; ++c) k[c] += (v[i] * rr) * orc_bf16_value(Wk[i * R + c]);
            double score = 0.0;
            for (int c = 0; c < R; ++c) score += q[c] * k[c];
            const double g = 1.0 / (1.0 + exp(-score / sqrt((double)R)));
            if (gates) gates[t * J + j] = g;
            for (int c = 0; c < R; ++c) e[c] += g * v[c];
        }
        for (int c = 0; c < R; ++c) {
            if (e_out) e_out[t * R + c] = e[c];
            X[c] = orc_bf16_value(orc_bf16_rne(e[c]));
        }
        for (int n = 0; n < d; ++n) y[n] = 0.0;
        for (int c = 0; c < R; ++c)
            for (int n = 0; n < d; ++n) y[n] += X[c] * orc_bf16_value(Wm[(int64_t)c * d + n]);
        for (int n = 0; n < d; ++n) ht[n] = orc_bf16_rne(hv[n] + y[n]);
    }
    free(q);
    free(y);
    free(hv);
    return ORC_OK;
}
