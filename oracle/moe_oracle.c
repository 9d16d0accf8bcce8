/*
 * CPU oracle for the routed-expert MoE FFN layer — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 restatement of what the layer computes.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may load this file's
 * library; the product path never does.  It shares no code, header or table
 * with the CUDA library.
 *
 * What it follows:
 *  - Gating: logits = x . W_r + b, a softmax, then the k largest scores
 *    (page 1, "MoE 模型卸载" blog, section 3.1, the CPU gating snippet).  The
 *    softmax is taken over the selected k logits only, which equals a softmax
 *    over all E followed by renormalising over the k selected.  Ties in the
 *    selection go to the lower expert id.
 *  - Expert FFN: SwiGLU, h = silu(W_gate x) * (W_up x), y = W_down h, with
 *    silu(z) = z / (1 + e^-z); one FFN per routed expert (page 3, tiered MoE
 *    scheduling note, shared/routed expert split; page 2, ffn_{gate,up,down}_exps).
 *  - Weights stay in their quantised blocks and are dequantised exactly:
 *    q8_0 w = d*q, 4-bit scale+min w = d*q + m (page 5, section 1.2: quantised
 *    blocks used as-is by the GPU GEMV; block layouts as stated in synth.py).
 *  - Output: y = sum_j w_j * y_{e_j} (+ shared experts with weight 1), summed in
 *    the caller (the layer composition in oracle/__init__.py) in fp64.
 *
 * Everything is double precision.  fp16 / bf16 inputs are decoded exactly from
 * their bit patterns.  OpenMP (if enabled) only splits independent output rows;
 * each dot product is one sequential fp64 loop.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- scalars */

/* IEEE 754 binary16 -> double, exact (sign, 5-bit exponent, 10-bit fraction). */
double oracle_fp16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);               /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 -> double, exact: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

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

/* ------------------------------------------------------------ dequantise */

/* q8_0: 34-byte block = fp16 d (little-endian) + 32 int8 q; w[i] = d * q[i]. */
void oracle_dequant_q8_0(const uint8_t *blocks, int64_t n_blocks, double *out) {
    for (int64_t b = 0; b < n_blocks; ++b) {
        const uint8_t *blk = blocks + 34 * b;
        double d = oracle_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
        for (int i = 0; i < 32; ++i) {
            int q = (int)(int8_t)blk[2 + i];
            out[32 * b + i] = d * (double)q;
        }
    }
}

/* 4-bit scale+min: 20-byte block = fp16 d, fp16 m, 16 bytes of codes; byte i holds
 * q[2i] (low nibble) and q[2i+1] (high nibble); w[j] = d * q[j] + m. */
void oracle_dequant_q4(const uint8_t *blocks, int64_t n_blocks, double *out) {
    for (int64_t b = 0; b < n_blocks; ++b) {
        const uint8_t *blk = blocks + 20 * b;
        double d = oracle_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
        double m = oracle_fp16_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
        for (int i = 0; i < 16; ++i) {
            int lo = blk[4 + i] & 0x0F;
            int hi = blk[4 + i] >> 4;
            out[32 * b + 2 * i] = d * (double)lo + m;
            out[32 * b + 2 * i + 1] = d * (double)hi + m;
        }
    }
}

/* One row (cols weights) of a canonical quantised matrix, dequantised. */
static void dequant_row(int qtype, const uint8_t *mat, int64_t row, int cols, double *out) {
    int64_t nb = cols / 32;
    if (qtype == 0)
        oracle_dequant_q8_0(mat + row * nb * 34, nb, out);
    else
        oracle_dequant_q4(mat + row * nb * 20, nb, out);
}

/* y[r] = sum_c W[r][c] * x[c] for a canonical quantised matrix W [rows][cols]. */
void oracle_qmatvec(int qtype, const uint8_t *mat, int rows, int cols, const double *x,
                    double *y) {
#pragma omp parallel
    {
        double wrow[32768];
#pragma omp for schedule(static)
        for (int r = 0; r < rows; ++r) {
            dequant_row(qtype, mat, r, cols, wrow);
            double acc = 0.0;
            for (int c = 0; c < cols; ++c) acc += wrow[c] * x[c];
            y[r] = acc;
        }
    }
}

/* ----------------------------------------------------------------- router */

/* logits[t][e] = sum_h x[t][h] * W_r[h][e] + bias[e]; W_r fp16 bits, row-major [H][E]. */
void oracle_router_logits(const double *x, int T, int H, const uint16_t *w_router,
                          const double *bias, int E, double *logits) {
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += x[(int64_t)t * H + h] * oracle_fp16_to_double(w_router[(int64_t)h * E + e]);
            logits[(int64_t)t * E + e] = acc + (bias ? bias[e] : 0.0);
        }
    }
}

/* Top-k by (logit descending, id ascending), then softmax over the k selected.
 * ids/weights are [T][k] in selection order; gap[t] = l_(k) - l_(k+1) (the margin
 * between the last selected and the first rejected logit; +inf when k == E). */
void oracle_topk_softmax(const double *logits, int T, int E, int k, int32_t *ids,
                         double *weights, double *gap) {
    for (int t = 0; t < T; ++t) {
        const double *l = logits + (int64_t)t * E;
        unsigned char taken[4096];
        memset(taken, 0, sizeof taken);
        for (int j = 0; j <= k && j < E; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* strict: equal keeps lower id */
            }
            if (j < k) {
                taken[best] = 1;
                ids[(int64_t)t * k + j] = best;
            } else {
                gap[t] = l[ids[(int64_t)t * k + k - 1]] - l[best];
            }
        }
        if (k >= E) gap[t] = INFINITY;
        double lmax = l[ids[(int64_t)t * k]];
        double denom = 0.0;
        for (int j = 0; j < k; ++j) denom += exp(l[ids[(int64_t)t * k + j]] - lmax);
        for (int j = 0; j < k; ++j)
            weights[(int64_t)t * k + j] = exp(l[ids[(int64_t)t * k + j]] - lmax) / denom;
    }
}

/* ------------------------------------------------------------------- FFN */

double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* One expert's SwiGLU FFN on one token: g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h.
 * gate/up are canonical [F][H] block matrices, down is [H][F]. scratch >= 3*F doubles. */
void oracle_expert_ffn(int qtype, int H, int F, const uint8_t *gate, const uint8_t *up,
                       const uint8_t *down, const double *x, double *y, double *scratch) {
    double *g = scratch, *u = scratch + F, *h = scratch + 2 * F;
    oracle_qmatvec(qtype, gate, F, H, x, g);
    oracle_qmatvec(qtype, up, F, H, x, u);
    for (int f = 0; f < F; ++f) h[f] = oracle_silu(g[f]) * u[f];
    oracle_qmatvec(qtype, down, H, F, h, y);
}
