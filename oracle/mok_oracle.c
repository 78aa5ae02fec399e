/*
 * mok_oracle.c - plain CPU oracle of the routed MoE layer.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library. The CUDA library never calls
 * it and shares no code, header, table or helper with it.
 *
 * Sources (news pages about Cursor's "Mixture-of-Kittens", MoK):
 *   [K-ja]  KuCoin (ja) "Cursor's MoK achieves 2.37x performance boost on
 *           NVIDIA GB300 NVL72", sections 01 (MoE "communication tax"),
 *           02 (push -> pull, megakernel, minibatch, ring buffer), 03 (results).
 *   [K-fil] The same article in Filipino, same sections.
 *   [RW]    RuntimeWire "Cursor open-sources MoK MoE training kernel",
 *           sections "Cursor's benchmark claims" and "Rebuilding the MoE layer
 *           around communication".
 * The pages describe the layer in prose only: the router picks several
 * experts per token [K-ja 01], per-expert counts and an expert-contiguous
 * placement feed a grouped GEMM [K-ja 01], each expert runs a SwiGLU FFN
 * [K-ja 02, last paragraphs], results return to their tokens and the layer
 * ends in a weighted sum [K-ja 03, first paragraph], with a fixed floating
 * point order [RW "Rebuilding..."]. Formulas the pages leave open (router
 * arithmetic, top-k rule, weight normalisation, SwiGLU, MXFP8 encoding) follow
 * the readings written next to each function below.
 *
 * Arithmetic: fp64 everywhere, except the router logits, which are computed in
 * one fixed fp32 order (see orc_router_logits) because they decide integers
 * (top-k indices, counts, permutation) that must agree bit for bit with the
 * GPU. Operands of the expert GEMMs are quantised exactly as the GPU consumes
 * them (BF16, or MXFP8 blocks of 32 along the reduction dimension).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no -ffast-math).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <float.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR 1

/* ------------------------------------------------------------------------- */
/* BF16                                                                        */
/* ------------------------------------------------------------------------- */

/* BF16 is the upper half of an IEEE binary32; the value is exact in double. */
static double bf16_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static uint16_t f32_bits_hi(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* Round a double to the nearest BF16 value, ties to even, in one step (no
 * intermediate binary32 rounding). BF16 keeps 8 significant bits; its
 * smallest normal is 2^-126 and its subnormal spacing 2^-133. */
double orc_round_bf16(double d) {
    if (d == 0.0 || !isfinite(d)) return d;
    double a = fabs(d);
    int p;
    frexp(a, &p);                 /* a = m * 2^p, m in [0.5, 1) */
    int e = p - 1;                /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;       /* subnormal range: fixed spacing */
    double ulp = ldexp(1.0, e - 7);
    double q = rint(a / ulp);     /* default rounding mode: nearest-even */
    double r = q * ulp;
    return d < 0 ? -r : r;
}

uint16_t orc_f64_to_bf16_bits(double d) {
    double r = orc_round_bf16(d);
    return f32_bits_hi((float)r); /* exact: r is a BF16 value */
}

/* Element i of an input array that holds BF16 bit patterns (f64 == 0) or
 * doubles (f64 == 1). Every public entry that takes model inputs accepts both,
 * so finite-difference checks can perturb inputs in fp64. */
static double ld(const void* p, long i, int f64) {
    return f64 ? ((const double*)p)[i] : bf16_to_f64(((const uint16_t*)p)[i]);
}

/* ------------------------------------------------------------------------- */
/* MXFP8: E4M3 elements with one E8M0 scale per 32-element block.             */
/* Reading (pages name only "MXFP8"): OCP Microscaling Formats v1.0.          */
/*   E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; S.1111.111 is NaN,   */
/*         so the largest finite magnitude is 448; no infinities.             */
/*   E8M0: unsigned exponent, value 2^(code-127), code 255 is NaN.           */
/*   Block scale X = floor(log2(amax)) - 8 (8 = largest E4M3 exponent),       */
/*   clamped to [-127, 127]; amax = 0 gives code 0. Each element is v / 2^X   */
/*   rounded to nearest E4M3 (ties to even mantissa), saturating at +-448.    */
/* ------------------------------------------------------------------------- */

/* Value of an E4M3 code from the format's definition. NaN codes return NaN. */
double orc_e4m3_value(uint8_t code) {
    int s = (code >> 7) & 1;
    int ex = (code >> 3) & 0xF;
    int man = code & 7;
    double v;
    if (ex == 0xF && man == 7) return NAN;
    if (ex == 0) v = ldexp((double)man / 8.0, -6);           /* subnormal */
    else v = ldexp(1.0 + (double)man / 8.0, ex - 7);
    return s ? -v : v;
}

/* Nearest finite E4M3 code by exhaustive search over the 127 non-negative
 * finite codes; on a tie the code with the even mantissa (even code) wins.
 * Magnitudes beyond 448 saturate to 448. The sign bit follows the sign of the
 * input, so negative values that round to zero give the code 0x80. */
uint8_t orc_e4m3_encode(double v) {
    double a = fabs(v);
    if (a >= 448.0) return (uint8_t)(signbit(v) ? 0xFE : 0x7E);   /* saturate */
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double err = fabs(orc_e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(signbit(v) ? (0x80 | best) : best);
}

/* E8M0 code of a block with largest magnitude amax (see the reading above). */
int orc_e8m0_code(double amax) {
    if (!(amax > 0.0)) return 0;
    int p;
    frexp(amax, &p);              /* amax in [2^(p-1), 2^p) */
    int X = (p - 1) - 8;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    return X + 127;
}

/* Quantise one block of n <= 32 values; returns the scale code. */
static int mx_quantize_block(const double* v, int n, int stride, uint8_t* codes, int cstride) {
    double amax = 0.0;
    for (int i = 0; i < n; ++i) {
        double a = fabs(v[(long)i * stride]);
        if (a > amax) amax = a;
    }
    int sc = orc_e8m0_code(amax);
    double inv = ldexp(1.0, 127 - sc);                 /* 1 / 2^X, exact */
    for (int i = 0; i < n; ++i) codes[(long)i * cstride] = orc_e4m3_encode(v[(long)i * stride] * inv);
    return sc;
}

/* Quantise a row-major [rows, cols] matrix along its rows in blocks of 32
 * (cols % 32 == 0): codes [rows, cols], scales [rows, cols/32]. */
int orc_mx_quantize_rows(const double* v, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* scales) {
    if (cols % 32) return ORC_ERR;
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            scales[r * nb + b] = (uint8_t)mx_quantize_block(v + r * cols + b * 32, 32, 1,
                                                            codes + r * cols + b * 32, 1);
    return ORC_OK;
}

/* Same for BF16 input rows (the activations x): the GPU gather must produce
 * these bytes bit for bit. */
int orc_mx_quantize_bf16_rows(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* scales) {
    if (cols % 32) return ORC_ERR;
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double blk[32];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 32; ++i) blk[i] = bf16_to_f64(x[r * cols + b * 32 + i]);
            scales[r * nb + b] = (uint8_t)mx_quantize_block(blk, 32, 1, codes + r * cols + b * 32, 1);
        }
    }
    return ORC_OK;
}

/* Value a block-quantised element stands for: E4M3 value times 2^(code-127). */
static double mx_value(uint8_t code, uint8_t scale) {
    return orc_e4m3_value(code) * ldexp(1.0, (int)scale - 127);
}

/* Replace v (length n, stride 1) by its MXFP8 round trip, blocks of 32. */
static void mx_roundtrip_vec(double* v, int n) {
    uint8_t codes[32];
    for (int b = 0; b < n; b += 32) {
        int sc = mx_quantize_block(v + b, 32, 1, codes, 1);
        for (int i = 0; i < 32; ++i) v[b + i] = mx_value(codes[i], (uint8_t)sc);
    }
}

/* ------------------------------------------------------------------------- */
/* Router                                                                      */
/* ------------------------------------------------------------------------- */

/* Router logits l[t,e] = sum_h x[t,h] * W_r[h,e] (+ bias[e]) in fp32.
 *
 * The pages say only that a router picks experts per token each step
 * ([K-ja 01], second paragraph). Because the logits decide integers that the
 * GPU must reproduce bit for bit, the sum is defined in one fixed binary32
 * order, the same on both sides:
 *   - 32 partial sums ("chains") c = 0..31, each starting at +0.0f;
 *   - chain c accumulates h = 256*i + 8*c + m for i = 0,1,... and m = 0..7
 *     (h < H only), in that order, each step one fused multiply-add
 *     acc = fmaf(x[t,h], W_r[h,e], acc) rounded to nearest;
 *   - the chains are combined by five butterfly steps, off = 16,8,4,2,1:
 *     s[c] <- s[c] + s[c ^ off] for every c at once; the logit is s[0];
 *   - then logit <- logit + bias[e] (binary32 add) when a bias is given.
 * IEEE fma and add are correctly rounded, so any conforming machine gets the
 * same bits. */
int orc_router_logits(const uint16_t* x, const float* W_r, const float* bias,
                      int T, int H, int E, float* logits) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            float s[32];
            for (int c = 0; c < 32; ++c) {
                float acc = 0.0f;
                for (int i = 0; 256 * i < H; ++i)
                    for (int m = 0; m < 8; ++m) {
                        int h = 256 * i + 8 * c + m;
                        if (h < H) acc = fmaf((float)bf16_to_f64(x[(long)t * H + h]), W_r[(long)h * E + e], acc);
                    }
                s[c] = acc;
            }
            for (int off = 16; off >= 1; off >>= 1) {
                float n[32];
                for (int c = 0; c < 32; ++c) n[c] = s[c] + s[c ^ off];
                memcpy(s, n, sizeof(s));
            }
            float l = s[0];
            if (bias) l = l + bias[e];
            logits[(long)t * E + e] = l;
        }
    }
    return ORC_OK;
}

/* Same sum in fp64 (any order). Used only for finite-difference checks of the
 * backward pass, never for parity with the GPU. */
int orc_router_logits_f64(const double* x, const double* W_r, const double* bias,
                          int T, int H, int E, double* logits) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h) acc += x[(long)t * H + h] * W_r[(long)h * E + e];
            if (bias) acc += bias[e];
            logits[(long)t * E + e] = acc;
        }
    return ORC_OK;
}

/* Top-k selection and routing weights, from fp32 or fp64 logits.
 *
 * Reading: experts are ranked by (logit descending, index ascending), so ties
 * go to the lower index; slot j holds the j-th ranked expert. The weights are
 * the softmax over all E logits restricted to the selected experts and
 * renormalised to sum 1, which equals the softmax over the k selected logits:
 *   w_j = exp(l_j - l_0) / sum_{i<k} exp(l_i - l_0).
 * Selection uses the logits only (softmax is monotone). Logits must be finite. */
static int topk_common(const double* lg, int E, int k, int32_t* idx, double* w) {
    unsigned char used[4096];
    if (E > 4096) return ORC_ERR;
    memset(used, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (used[e]) continue;
            if (!isfinite(lg[e])) return ORC_ERR;
            if (best < 0 || lg[e] > lg[best]) best = e;   /* strict: lower index wins ties */
        }
        used[best] = 1;
        idx[j] = best;
    }
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += exp(lg[idx[j]] - lg[idx[0]]);
    for (int j = 0; j < k; ++j) w[j] = exp(lg[idx[j]] - lg[idx[0]]) / den;
    return ORC_OK;
}

int orc_topk_f32(const float* logits, int T, int E, int k, int32_t* idx, double* w) {
    if (k < 1 || k > E) return ORC_ERR;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(|:bad)
    for (int t = 0; t < T; ++t) {
        double lg[4096];
        if (E > 4096) { bad = 1; continue; }
        for (int e = 0; e < E; ++e) lg[e] = (double)logits[(long)t * E + e];
        bad |= topk_common(lg, E, k, idx + (long)t * k, w + (long)t * k);
    }
    return bad ? ORC_ERR : ORC_OK;
}

int orc_topk_f64(const double* logits, int T, int E, int k, int32_t* idx, double* w) {
    if (k < 1 || k > E) return ORC_ERR;
    int bad = 0;
    for (int t = 0; t < T; ++t) bad |= topk_common(logits + (long)t * E, E, k, idx + (long)t * k, w + (long)t * k);
    return bad ? ORC_ERR : ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Per-expert count and expert-contiguous placement                            */
/* ------------------------------------------------------------------------- */

/* The pages: count each expert's tokens, decide where each token lands, keep
 * the same expert's tokens adjacent so the grouped GEMM gets ordered input
 * ([K-ja 01], fourth paragraph). Reading: rows are ordered by (expert
 * ascending, token ascending); offsets are the exclusive prefix sum of the
 * counts (no padding); row_src[row] = t*k + j names the slot the row came
 * from and slot_row is its inverse. */
int orc_layout(const int32_t* idx, int T, int E, int k,
               int32_t* counts, int32_t* offsets, int32_t* row_src, int32_t* slot_row) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long s = 0; s < (long)T * k; ++s) {
        if (idx[s] < 0 || idx[s] >= E) return ORC_ERR;
        counts[idx[s]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t row = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j)
                if (idx[(long)t * k + j] == e) {
                    row_src[row] = t * k + j;
                    slot_row[(long)t * k + j] = row;
                    ++row;
                }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Expert FFN (SwiGLU) and the layer forward                                   */
/* ------------------------------------------------------------------------- */

/* Reading of "SwiGLU" ([K-ja 02], MXFP8 paragraph names it as a stage):
 *   G = a W_gate[e], U = a W_up[e], h = silu(G) * U, y = h W_down[e],
 *   silu(z) = z / (1 + exp(-z)); no biases, no extra scaling. */
static double silu(double z) { return z / (1.0 + exp(-z)); }

#define ORC_BF16 0
#define ORC_MXFP8 1
#define ORC_EXACT 2   /* no operand rounding at all (finite-difference checks) */

/* Operand values of one expert's weights, as the GEMMs consume them.
 * gate/up are [H, I] (reduction dim H: MXFP8 blocks run along H for each
 * column); down is [I, H] (blocks along I for each column). */
typedef struct { double *g, *u, *d; } expert_w;

static void load_expert(const void* Wg, const void* Wu, const void* Wd, int f64,
                        int e, int H, int I, int mode, expert_w* out) {
    long HI = (long)H * I;
    long base = (long)e * HI;
#pragma omp parallel for schedule(static)
    for (long i = 0; i < HI; ++i) {
        out->g[i] = ld(Wg, base + i, f64);
        out->u[i] = ld(Wu, base + i, f64);
        out->d[i] = ld(Wd, base + i, f64);
    }
    if (mode != ORC_MXFP8) return;
    /* Blocks of 32 along the reduction dimension, one scale per (block, column). */
#pragma omp parallel for schedule(static)
    for (int col = 0; col < I; ++col) {
        double blk[32];
        uint8_t codes[32];
        for (int kb = 0; kb < H; kb += 32) {
            double* mats[2] = {out->g, out->u};
            for (int q = 0; q < 2; ++q) {
                for (int r = 0; r < 32; ++r) blk[r] = mats[q][(long)(kb + r) * I + col];
                int sc = mx_quantize_block(blk, 32, 1, codes, 1);
                for (int r = 0; r < 32; ++r) mats[q][(long)(kb + r) * I + col] = mx_value(codes[r], (uint8_t)sc);
            }
        }
    }
#pragma omp parallel for schedule(static)
    for (int col = 0; col < H; ++col) {
        double blk[32];
        uint8_t codes[32];
        for (int kb = 0; kb < I; kb += 32) {
            for (int r = 0; r < 32; ++r) blk[r] = out->d[(long)(kb + r) * H + col];
            int sc = mx_quantize_block(blk, 32, 1, codes, 1);
            for (int r = 0; r < 32; ++r) out->d[(long)(kb + r) * H + col] = mx_value(codes[r], (uint8_t)sc);
        }
    }
}

/* One row through one expert: a [H] -> y [H]; optionally returns G, U, h
 * (h as the down GEMM consumes it). mode picks the h operand rounding. */
static void ffn_row(const double* a, const expert_w* W, int H, int I, int mode,
                    double* G, double* U, double* h, double* y) {
    for (int i = 0; i < I; ++i) { G[i] = 0.0; U[i] = 0.0; }
    for (int hh = 0; hh < H; ++hh) {
        double av = a[hh];
        if (av == 0.0) continue;
        const double* gr = W->g + (long)hh * I;
        const double* ur = W->u + (long)hh * I;
        for (int i = 0; i < I; ++i) { G[i] += av * gr[i]; U[i] += av * ur[i]; }
    }
    for (int i = 0; i < I; ++i) h[i] = silu(G[i]) * U[i];
    if (mode == ORC_BF16) for (int i = 0; i < I; ++i) h[i] = orc_round_bf16(h[i]);
    else if (mode == ORC_MXFP8) mx_roundtrip_vec(h, I);
    for (int c = 0; c < H; ++c) y[c] = 0.0;
    for (int i = 0; i < I; ++i) {
        double hv = h[i];
        if (hv == 0.0) continue;
        const double* dr = W->d + (long)i * H;
        for (int c = 0; c < H; ++c) y[c] += hv * dr[c];
    }
}

/* Activation operand of token t: BF16 x exactly, or its MXFP8 round trip. */
static void act_row(const void* x, int f64, int t, int H, int mode, double* a) {
    for (int h = 0; h < H; ++h) a[h] = ld(x, (long)t * H + h, f64);
    if (mode == ORC_MXFP8) mx_roundtrip_vec(a, H);
}

static int alloc_expert(expert_w* w, long HI) {
    w->g = (double*)malloc(sizeof(double) * HI);
    w->u = (double*)malloc(sizeof(double) * HI);
    w->d = (double*)malloc(sizeof(double) * HI);
    return (w->g && w->u && w->d) ? ORC_OK : ORC_ERR;
}
static void free_expert(expert_w* w) { free(w->g); free(w->u); free(w->d); }

/* Layer forward for the tokens listed in `tokens` (n_tok of them; NULL means
 * all T in order): out[n, :] = sum_j w[t,j] * y[t,j] + shared[t] in fp64.
 *
 * Routing (idx, w, layout) must already be computed (orc_topk_*, orc_layout).
 * The routed rows are visited expert by expert in layout order (row_src),
 * each row is pulled from its token, run through its expert, and its result
 * is pushed back to its (token, slot) - the plain, unfused form of the
 * dispatch -> grouped FFN -> combine -> weighted sum sequence the pages
 * describe ([K-ja 02] pull dispatch / push combine; [K-ja 03] weighted sum).
 * The sum over slots runs j = 0..k-1 ([RW "Rebuilding..."]: fixed order).
 *
 * mode: 0 BF16 operands (h rounded to BF16 before the down projection),
 *       1 MXFP8 operands (x, W_gate, W_up blocked along H; h, W_down along I),
 *       2 exact (no rounding of h; used by finite-difference checks).
 * Shared expert (optional, Wsg/Wsu [H, Is], Wsd [Is, H]): BF16 operands in
 * modes 0 and 1 (the pages keep shared experts in BF16 [RW "Rebuilding..."]),
 * weight 1, added after the routed sum. y_out (optional) receives the
 * unweighted per-slot results [n_tok, k, H]. Inputs are BF16 bit patterns
 * (f64 == 0) or doubles (f64 == 1). */
int orc_moe_forward(const void* x, const void* Wg, const void* Wu, const void* Wd, int f64,
                    int T, int H, int I, int E, int k,
                    const int32_t* idx, const double* w, const int32_t* offsets, const int32_t* row_src,
                    int mode, const int32_t* tokens, int n_tok,
                    const void* Wsg, const void* Wsu, const void* Wsd, int Is,
                    double* out, double* y_out) {
    (void)idx;
    if (mode < 0 || mode > 2) return ORC_ERR;
    if (mode == ORC_MXFP8 && (H % 32 || I % 32)) return ORC_ERR;
    int n = tokens ? n_tok : T;
    /* position of each token in the output (or -1 when not sampled) */
    int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)T);
    if (!pos) return ORC_ERR;
    for (int t = 0; t < T; ++t) pos[t] = tokens ? -1 : t;
    if (tokens) for (int q = 0; q < n_tok; ++q) { if (tokens[q] < 0 || tokens[q] >= T) { free(pos); return ORC_ERR; } pos[tokens[q]] = q; }
    double* yslots = (double*)calloc((size_t)n * k * H, sizeof(double));
    if (!yslots) { free(pos); return ORC_ERR; }
    long HI = (long)H * I;
    expert_w W;
    if (alloc_expert(&W, HI)) { free(pos); free(yslots); return ORC_ERR; }
    for (int e = 0; e < E; ++e) {
        int r0 = offsets[e], r1 = offsets[e + 1];
        int any = 0;
        for (int r = r0; r < r1 && !any; ++r) any = pos[row_src[r] / k] >= 0;
        if (!any) continue;
        load_expert(Wg, Wu, Wd, f64, e, H, I, mode, &W);
#pragma omp parallel
        {
            double* a = (double*)malloc(sizeof(double) * H);
            double* G = (double*)malloc(sizeof(double) * I);
            double* U = (double*)malloc(sizeof(double) * I);
            double* hb = (double*)malloc(sizeof(double) * I);
#pragma omp for schedule(dynamic, 1)
            for (int r = r0; r < r1; ++r) {
                int slot = row_src[r];
                int t = slot / k, j = slot % k;
                if (pos[t] < 0) continue;
                act_row(x, f64, t, H, mode, a);
                ffn_row(a, &W, H, I, mode, G, U, hb, yslots + ((long)pos[t] * k + j) * H);
            }
            free(a); free(G); free(U); free(hb);
        }
    }
    free_expert(&W);
    /* push-combine then fixed-order weighted sum */
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        if (pos[t] < 0) continue;
        double* o = out + (long)pos[t] * H;
        for (int c = 0; c < H; ++c) o[c] = 0.0;
        for (int j = 0; j < k; ++j) {
            double wj = w[(long)t * k + j];
            const double* y = yslots + ((long)pos[t] * k + j) * H;
            for (int c = 0; c < H; ++c) o[c] += wj * y[c];
        }
    }
    if (y_out) memcpy(y_out, yslots, sizeof(double) * (size_t)n * k * H);
    free(yslots);
    if (Wsg) {
        /* shared expert: BF16 operands (exact mode keeps h unrounded) */
        int smode = (mode == ORC_EXACT) ? ORC_EXACT : ORC_BF16;
        long HIs = (long)H * Is;
        expert_w S;
        if (alloc_expert(&S, HIs)) { free(pos); return ORC_ERR; }
        load_expert(Wsg, Wsu, Wsd, f64, 0, H, Is, smode, &S);
#pragma omp parallel
        {
            double* a = (double*)malloc(sizeof(double) * H);
            double* G = (double*)malloc(sizeof(double) * Is);
            double* U = (double*)malloc(sizeof(double) * Is);
            double* hb = (double*)malloc(sizeof(double) * Is);
            double* y = (double*)malloc(sizeof(double) * H);
#pragma omp for schedule(dynamic, 1)
            for (int t = 0; t < T; ++t) {
                if (pos[t] < 0) continue;
                act_row(x, f64, t, H, ORC_BF16, a);
                ffn_row(a, &S, H, Is, smode, G, U, hb, y);
                double* o = out + (long)pos[t] * H;
                for (int c = 0; c < H; ++c) o[c] += y[c];
            }
            free(a); free(G); free(U); free(hb); free(y);
        }
        free_expert(&S);
    }
    free(pos);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Backward                                                                    */
/* ------------------------------------------------------------------------- */

/* Backward of the layer for upstream gradient dY [T, H] (BF16), by the chain
 * rule applied to the forward above. The pages describe the backward only as
 * two reverse communications: pull on reverse-combine, push on
 * reverse-dispatch ([K-ja 02], paragraph on pull/push directions); the
 * arithmetic is the derivative of the forward:
 *   reverse-combine:  dy_j = w_j * dY[t],   gw_j = <dY[t], y_j>
 *   expert dgrad:     dh = dy_j W_down^T,  dG = dh * U * silu'(G),
 *                     dU = dh * silu(G),   da_j = dG W_gate^T + dU W_up^T
 *   expert wgrad:     dW_down[e] += h^T dy_j, dW_gate[e] += a^T dG,
 *                     dW_up[e] += a^T dU  (over the expert's rows, row order)
 *   router:           dl_j = w_j (gw_j - sum_i w_i gw_i) for selected experts,
 *                     zero for the others (the renormalised softmax over the
 *                     selected logits cancels the full-softmax denominator);
 *                     dW_r[h, e_j] += x[t,h] dl_j
 *   reverse-dispatch: dX[t] = sum_j da_j + sum_j dl_j W_r[:, e_j].
 * silu'(z) = s (1 + z (1 - s)), s = 1/(1+exp(-z)).
 * mode 0 (BF16): the GEMM operands the GPU stores in BF16 are rounded the same
 * way: h, dy, dG, dU. mode 2: no rounding. mode 1 (MXFP8): the forward as in
 * orc_moe_forward mode 1, the same BF16 roundings of dy, dG, dU and h, and
 * every backward GEMM operand quantised to MXFP8 along that GEMM's reduction
 * dimension: dy and W_down along H (dh), dG, dU, W_gate, W_up along I (da),
 * and x, h, dy, dG, dU along the expert's rows, 32 at a time (the weight
 * gradients).
 * Logits must be those the routing used (fp32 logits widened, or fp64).
 * Inputs are BF16 bits (W_r binary32) when f64 == 0, doubles when f64 == 1.
 * Outputs are fp64: dX [T,H], dWg/dWu [E,H,I], dWd [E,I,H], dWr [H,E].
 * The bias (if any) receives no gradient. */
/* Router weights are binary32 (f64 == 0) or doubles (f64 == 1). */
static double wr_at(const void* W_r, long i, int f64) {
    return f64 ? ((const double*)W_r)[i] : (double)((const float*)W_r)[i];
}

/* MXFP8 round trip of the rows of an [R, K] matrix along K (blocks of 32). */
static void mx_roundtrip_rows(double* v, long R, int K) {
#pragma omp parallel for schedule(static)
    for (long r = 0; r < R; ++r) mx_roundtrip_vec(v + r * K, K);
}

/* MXFP8 round trip of the columns of an [R, C] matrix along R, in blocks of
 * 32 consecutive rows starting at row 0 (the last block may be shorter: its
 * scale comes from its own rows). */
static void mx_roundtrip_cols(double* v, long R, int C) {
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; ++c) {
        double blk[32];
        uint8_t codes[32];
        for (long r0 = 0; r0 < R; r0 += 32) {
            int n = (int)(R - r0 < 32 ? R - r0 : 32);
            for (int q = 0; q < 32; ++q) blk[q] = q < n ? v[(r0 + q) * C + c] : 0.0;
            int sc = mx_quantize_block(blk, 32, 1, codes, 1);
            for (int q = 0; q < n; ++q) v[(r0 + q) * C + c] = mx_value(codes[q], (uint8_t)sc);
        }
    }
}

int orc_moe_backward(const void* x, const void* W_r, const void* Wg, const void* Wu,
                     const void* Wd, const void* dY, int f64, int T, int H, int I, int E, int k,
                     const int32_t* idx, const double* w, const int32_t* offsets, const int32_t* row_src,
                     int mode, double* dX, double* dWg, double* dWu, double* dWd, double* dWr) {
    if (mode != ORC_BF16 && mode != ORC_EXACT && mode != ORC_MXFP8) return ORC_ERR;
    if (mode == ORC_MXFP8 && (H % 32 || I % 32)) return ORC_ERR;
    const int mx = mode == ORC_MXFP8;
    /* the BF16 roundings of the stored backward operands (dy, dG, dU, and h
     * as the weight gradient reads it) apply in both quantised modes */
    const int round_bf = mode != ORC_EXACT;
    long HI = (long)H * I;
    double* gw = (double*)calloc((size_t)T * k, sizeof(double));
    double* da = (double*)calloc((size_t)T * k * H, sizeof(double));
    if (!gw || !da) { free(gw); free(da); return ORC_ERR; }
    memset(dWg, 0, sizeof(double) * (size_t)E * HI);
    memset(dWu, 0, sizeof(double) * (size_t)E * HI);
    memset(dWd, 0, sizeof(double) * (size_t)E * HI);
    expert_w W, WB;   /* forward operands; MXFP8: the backward's dgrad operands */
    if (alloc_expert(&W, HI)) { free(gw); free(da); return ORC_ERR; }
    if (mx && alloc_expert(&WB, HI)) { free_expert(&W); free(gw); free(da); return ORC_ERR; }
    for (int e = 0; e < E; ++e) {
        int r0 = offsets[e], r1 = offsets[e + 1];
        if (r1 == r0) continue;
        load_expert(Wg, Wu, Wd, f64, e, H, I, mode, &W);
        if (mx) {
            /* MXFP8 backward (reading of the pages' "MXFP8 backward", KuCoin
             * ja/fil article, section 03, and RuntimeWire "Cursor's benchmark
             * claims"): every backward GEMM takes MXFP8 operands blocked along
             * its own reduction dimension. dh = dy W_down^T reduces over H, so
             * W_down's rows are blocked along H; da = dG W_gate^T + dU W_up^T
             * reduces over I, so W_gate's and W_up's rows are blocked along I. */
            load_expert(Wg, Wu, Wd, f64, e, H, I, ORC_BF16, &WB);
            mx_roundtrip_rows(WB.g, H, I);
            mx_roundtrip_rows(WB.u, H, I);
            mx_roundtrip_rows(WB.d, I, H);
        }
        const expert_w* Wb = mx ? &WB : &W;
        int nr = r1 - r0;
        /* per-row forward intermediates and gradients of this expert */
        double* A = (double*)malloc(sizeof(double) * (size_t)nr * H);
        double* HB = (double*)malloc(sizeof(double) * (size_t)nr * I);
        double* DY = (double*)malloc(sizeof(double) * (size_t)nr * H);
        double* DG = (double*)malloc(sizeof(double) * (size_t)nr * I);
        double* DU = (double*)malloc(sizeof(double) * (size_t)nr * I);
        if (!A || !HB || !DY || !DG || !DU) return ORC_ERR;
#pragma omp parallel
        {
            double* G = (double*)malloc(sizeof(double) * I);
            double* U = (double*)malloc(sizeof(double) * I);
            double* hq = (double*)malloc(sizeof(double) * I);
            double* y = (double*)malloc(sizeof(double) * H);
            double* dh = (double*)malloc(sizeof(double) * I);
            double* af = (double*)malloc(sizeof(double) * H);
            double* dyq = (double*)malloc(sizeof(double) * H);
            double* dgq = (double*)malloc(sizeof(double) * I);
            double* duq = (double*)malloc(sizeof(double) * I);
#pragma omp for schedule(dynamic, 1)
            for (int q = 0; q < nr; ++q) {
                int slot = row_src[r0 + q];
                int t = slot / k;
                double* a = A + (long)q * H;
                act_row(x, f64, t, H, ORC_BF16, a);            /* x as stored (BF16) */
                act_row(x, f64, t, H, mode, af);               /* x as the forward GEMM reads it */
                ffn_row(af, &W, H, I, mode, G, U, hq, y);
                /* h as the weight gradient reads it: BF16 (mode 1 stores h in
                 * BF16 for the backward besides the MXFP8 copy the down GEMM
                 * reads), exact in mode 2 */
                for (int i = 0; i < I; ++i) {
                    double hv = silu(G[i]) * U[i];
                    HB[(long)q * I + i] = mode == ORC_BF16 ? hq[i] : (mx ? orc_round_bf16(hv) : hv);
                }
                /* reverse-combine */
                double wj = w[slot], g = 0.0;
                double* dyr = DY + (long)q * H;
                for (int c = 0; c < H; ++c) {
                    double dYv = ld(dY, (long)t * H + c, f64);
                    g += dYv * y[c];
                    dyr[c] = wj * dYv;
                    if (round_bf) dyr[c] = orc_round_bf16(dyr[c]);
                    dyq[c] = dyr[c];
                }
                if (mx) mx_roundtrip_vec(dyq, H);
                gw[slot] = g;
                /* dgrad of the down projection and of SwiGLU */
                for (int i = 0; i < I; ++i) {
                    double s = 0.0;
                    const double* dr = Wb->d + (long)i * H;
                    for (int c = 0; c < H; ++c) s += dyq[c] * dr[c];
                    dh[i] = s;
                }
                for (int i = 0; i < I; ++i) {
                    double sg = 1.0 / (1.0 + exp(-G[i]));
                    double dgv = dh[i] * U[i] * sg * (1.0 + G[i] * (1.0 - sg));
                    double duv = dh[i] * G[i] * sg;
                    if (round_bf) { dgv = orc_round_bf16(dgv); duv = orc_round_bf16(duv); }
                    DG[(long)q * I + i] = dgv;
                    DU[(long)q * I + i] = duv;
                    dgq[i] = dgv;
                    duq[i] = duv;
                }
                if (mx) { mx_roundtrip_vec(dgq, I); mx_roundtrip_vec(duq, I); }
                /* da = dG W_gate^T + dU W_up^T, pushed to slot (t, j) */
                double* dar = da + (long)slot * H;
                for (int c = 0; c < H; ++c) {
                    const double* gr = Wb->g + (long)c * I;
                    const double* ur = Wb->u + (long)c * I;
                    double s = 0.0;
                    for (int i = 0; i < I; ++i) s += dgq[i] * gr[i] + duq[i] * ur[i];
                    dar[c] = s;
                }
            }
            free(G); free(U); free(hq); free(y); free(dh); free(af); free(dyq); free(dgq); free(duq);
        }
        if (mx) {
            /* the weight gradients reduce over the expert's rows (layout
             * order): their operands are blocked along those rows, 32 at a
             * time from the expert's first row */
            mx_roundtrip_cols(A, nr, H);
            mx_roundtrip_cols(HB, nr, I);
            mx_roundtrip_cols(DY, nr, H);
            mx_roundtrip_cols(DG, nr, I);
            mx_roundtrip_cols(DU, nr, I);
        }
        /* wgrad: sums over the expert's rows in row order */
        double* dg = dWg + (long)e * HI;
        double* du = dWu + (long)e * HI;
        double* dd = dWd + (long)e * HI;
#pragma omp parallel for schedule(static)
        for (int hh = 0; hh < H; ++hh)
            for (int q = 0; q < nr; ++q) {
                double av = A[(long)q * H + hh];
                for (int i = 0; i < I; ++i) {
                    dg[(long)hh * I + i] += av * DG[(long)q * I + i];
                    du[(long)hh * I + i] += av * DU[(long)q * I + i];
                }
            }
#pragma omp parallel for schedule(static)
        for (int i = 0; i < I; ++i)
            for (int q = 0; q < nr; ++q) {
                double hv = HB[(long)q * I + i];
                for (int c = 0; c < H; ++c) dd[(long)i * H + c] += hv * DY[(long)q * H + c];
            }
        free(A); free(HB); free(DY); free(DG); free(DU);
    }
    free_expert(&W);
    if (mx) free_expert(&WB);
    /* router backward and reverse-dispatch */
    memset(dWr, 0, sizeof(double) * (size_t)H * E);
    double* dl = (double*)calloc((size_t)T * k, sizeof(double));
    if (!dl) return ORC_ERR;
    for (int t = 0; t < T; ++t) {
        double m = 0.0;
        for (int j = 0; j < k; ++j) m += w[(long)t * k + j] * gw[(long)t * k + j];
        for (int j = 0; j < k; ++j) dl[(long)t * k + j] = w[(long)t * k + j] * (gw[(long)t * k + j] - m);
    }
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int c = 0; c < H; ++c) {
            double s = 0.0;
            for (int j = 0; j < k; ++j) s += da[((long)t * k + j) * H + c];
            for (int j = 0; j < k; ++j) s += dl[(long)t * k + j] * wr_at(W_r, (long)c * E + idx[(long)t * k + j], f64);
            dX[(long)t * H + c] = s;
        }
#pragma omp parallel for schedule(static)
    for (int c = 0; c < H; ++c)
        for (int t = 0; t < T; ++t) {
            double xv = ld(x, (long)t * H + c, f64);
            for (int j = 0; j < k; ++j) dWr[(long)c * E + idx[(long)t * k + j]] += xv * dl[(long)t * k + j];
        }
    free(dl); free(gw); free(da);
    return ORC_OK;
}

/* Selected outputs of the backward above, computed one by one (for inputs
 * too large for the full backward): the same formulas restricted to
 *   dX rows of the tokens in `tok` (n_tok),
 *   dW_gate[e][:, i] and dW_up[e][:, i] columns for the (e, i) pairs in
 *   `col_e`/`col_i` (n_col), and dW_down[e][i][:] rows for the same pairs.
 * Inputs as in orc_moe_backward (BF16 bits, mode 0 rounds the operands the GPU
 * stores in BF16). Outputs: dX_s [n_tok, H], dWg_s/dWu_s [n_col, H],
 * dWd_s [n_col, H]. The router term of dX needs gw for the token's own slots
 * only, so no other token is touched. */
static void row_fwd_cols(const double* a, const uint16_t* Wg, const uint16_t* Wu, long base, int H, int I,
                         int i, double* G, double* U) {
    double g = 0.0, u = 0.0;
    for (int hh = 0; hh < H; ++hh) {
        g += a[hh] * bf16_to_f64(Wg[base + (long)hh * I + i]);
        u += a[hh] * bf16_to_f64(Wu[base + (long)hh * I + i]);
    }
    *G = g;
    *U = u;
}

int orc_moe_backward_sampled(const uint16_t* x, const float* W_r, const uint16_t* Wg, const uint16_t* Wu,
                             const uint16_t* Wd, const uint16_t* dY, int T, int H, int I, int E, int k,
                             const int32_t* idx, const double* w, const int32_t* offsets, const int32_t* row_src,
                             int mode, const int32_t* tok, int n_tok, const int32_t* col_e, const int32_t* col_i,
                             int n_col, double* dX_s, double* dWg_s, double* dWu_s, double* dWd_s) {
    if (mode != ORC_BF16 && mode != ORC_EXACT) return ORC_ERR;
    long HI = (long)H * I;
    /* ---- dX rows */
    for (int q = 0; q < n_tok; ++q) {
        int t = tok[q];
        if (t < 0 || t >= T) return ORC_ERR;
        double* o = dX_s + (long)q * H;
        double* gwv = (double*)calloc((size_t)k, sizeof(double));
        double* a = (double*)malloc(sizeof(double) * H);
        double* da = (double*)calloc((size_t)k * H, sizeof(double));
        if (!gwv || !a || !da) return ORC_ERR;
        for (int h = 0; h < H; ++h) a[h] = bf16_to_f64(x[(long)t * H + h]);
        for (int j = 0; j < k; ++j) {
            int e = idx[(long)t * k + j];
            long base = (long)e * HI;
            double wj = w[(long)t * k + j];
            double* G = (double*)malloc(sizeof(double) * I);
            double* U = (double*)malloc(sizeof(double) * I);
            double* hb = (double*)malloc(sizeof(double) * I);
            double* dyr = (double*)malloc(sizeof(double) * H);
            double* DG = (double*)malloc(sizeof(double) * I);
            double* DU = (double*)malloc(sizeof(double) * I);
#pragma omp parallel for schedule(static)
            for (int i = 0; i < I; ++i) row_fwd_cols(a, Wg, Wu, base, H, I, i, &G[i], &U[i]);
            for (int i = 0; i < I; ++i) {
                hb[i] = silu(G[i]) * U[i];
                if (mode == ORC_BF16) hb[i] = orc_round_bf16(hb[i]);
            }
            /* y and gw */
            double g = 0.0;
            for (int c = 0; c < H; ++c) {
                double y = 0.0;
                for (int i = 0; i < I; ++i) y += hb[i] * bf16_to_f64(Wd[base + (long)i * H + c]);
                double dYv = bf16_to_f64(dY[(long)t * H + c]);
                g += dYv * y;
                dyr[c] = wj * dYv;
                if (mode == ORC_BF16) dyr[c] = orc_round_bf16(dyr[c]);
            }
            gwv[j] = g;
#pragma omp parallel for schedule(static)
            for (int i = 0; i < I; ++i) {
                double dh = 0.0;
                for (int c = 0; c < H; ++c) dh += dyr[c] * bf16_to_f64(Wd[base + (long)i * H + c]);
                double sg = 1.0 / (1.0 + exp(-G[i]));
                double dgv = dh * U[i] * sg * (1.0 + G[i] * (1.0 - sg));
                double duv = dh * G[i] * sg;
                if (mode == ORC_BF16) { dgv = orc_round_bf16(dgv); duv = orc_round_bf16(duv); }
                DG[i] = dgv;
                DU[i] = duv;
            }
#pragma omp parallel for schedule(static)
            for (int c = 0; c < H; ++c) {
                double s = 0.0;
                for (int i = 0; i < I; ++i)
                    s += DG[i] * bf16_to_f64(Wg[base + (long)c * I + i]) + DU[i] * bf16_to_f64(Wu[base + (long)c * I + i]);
                da[(long)j * H + c] = s;
            }
            free(G); free(U); free(hb); free(dyr); free(DG); free(DU);
        }
        double m = 0.0;
        for (int j = 0; j < k; ++j) m += w[(long)t * k + j] * gwv[j];
        for (int c = 0; c < H; ++c) {
            double s = 0.0;
            for (int j = 0; j < k; ++j) s += da[(long)j * H + c];
            for (int j = 0; j < k; ++j) {
                double dl = w[(long)t * k + j] * (gwv[j] - m);
                s += dl * (double)W_r[(long)c * E + idx[(long)t * k + j]];
            }
            o[c] = s;
        }
        free(gwv); free(a); free(da);
    }
    /* ---- weight-gradient columns / rows */
    for (int q = 0; q < n_col; ++q) {
        int e = col_e[q], i = col_i[q];
        if (e < 0 || e >= E || i < 0 || i >= I) return ORC_ERR;
        long base = (long)e * HI;
        int r0 = offsets[e], r1 = offsets[e + 1];
        double* og = dWg_s + (long)q * H;
        double* ou = dWu_s + (long)q * H;
        double* od = dWd_s + (long)q * H;
        for (int c = 0; c < H; ++c) { og[c] = 0.0; ou[c] = 0.0; od[c] = 0.0; }
        int nr = r1 - r0;
        double* DGc = (double*)malloc(sizeof(double) * (nr > 0 ? nr : 1));
        double* DUc = (double*)malloc(sizeof(double) * (nr > 0 ? nr : 1));
        double* Hc = (double*)malloc(sizeof(double) * (nr > 0 ? nr : 1));
        if (!DGc || !DUc || !Hc) return ORC_ERR;
#pragma omp parallel
        {
            double* a = (double*)malloc(sizeof(double) * H);
#pragma omp for schedule(static)
            for (int rr = 0; rr < nr; ++rr) {
                int slot = row_src[r0 + rr];
                int t = slot / k;
                for (int h = 0; h < H; ++h) a[h] = bf16_to_f64(x[(long)t * H + h]);
                double G, U;
                row_fwd_cols(a, Wg, Wu, base, H, I, i, &G, &U);
                double hv = silu(G) * U;
                if (mode == ORC_BF16) hv = orc_round_bf16(hv);
                double dh = 0.0;
                for (int c = 0; c < H; ++c) {
                    double dyv = w[slot] * bf16_to_f64(dY[(long)t * H + c]);
                    if (mode == ORC_BF16) dyv = orc_round_bf16(dyv);
                    dh += dyv * bf16_to_f64(Wd[base + (long)i * H + c]);
                }
                double sg = 1.0 / (1.0 + exp(-G));
                double dgv = dh * U * sg * (1.0 + G * (1.0 - sg));
                double duv = dh * G * sg;
                if (mode == ORC_BF16) { dgv = orc_round_bf16(dgv); duv = orc_round_bf16(duv); }
                DGc[rr] = dgv;
                DUc[rr] = duv;
                Hc[rr] = hv;
            }
            free(a);
        }
        /* sums over the expert's rows, row order */
        for (int rr = 0; rr < nr; ++rr) {
            int slot = row_src[r0 + rr];
            int t = slot / k;
            for (int c = 0; c < H; ++c) {
                double av = bf16_to_f64(x[(long)t * H + c]);
                double dyv = w[slot] * bf16_to_f64(dY[(long)t * H + c]);
                if (mode == ORC_BF16) dyv = orc_round_bf16(dyv);
                og[c] += av * DGc[rr];
                ou[c] += av * DUc[rr];
                od[c] += Hc[rr] * dyv;
            }
        }
        free(DGc); free(DUc); free(Hc);
    }
    return ORC_OK;
}

/* The sampled outputs of orc_moe_backward_sampled in the MXFP8 mode of
 * orc_moe_backward (same arguments and outputs, BF16 inputs). Experts are
 * visited once each; an expert used by a sampled token or column has its
 * forward weights (W_gate, W_up blocked along H, W_down along I) and its
 * backward copies (W_down along H, W_gate and W_up along I) quantised once.
 * dX rows need only the token's own k rows; a weight-gradient column needs
 * the whole column of its operands over the expert's rows, blocked along
 * those rows 32 at a time from the expert's first row. */
int orc_moe_backward_sampled_mx(const uint16_t* x, const float* W_r, const uint16_t* Wg, const uint16_t* Wu,
                                const uint16_t* Wd, const uint16_t* dY, int T, int H, int I, int E, int k,
                                const int32_t* idx, const double* w, const int32_t* offsets, const int32_t* row_src,
                                const int32_t* tok, int n_tok, const int32_t* col_e, const int32_t* col_i, int n_col,
                                double* dX_s, double* dWg_s, double* dWu_s, double* dWd_s) {
    if (H % 32 || I % 32) return ORC_ERR;
    for (int q = 0; q < n_tok; ++q) if (tok[q] < 0 || tok[q] >= T) return ORC_ERR;
    for (int q = 0; q < n_col; ++q) if (col_e[q] < 0 || col_e[q] >= E || col_i[q] < 0 || col_i[q] >= I) return ORC_ERR;
    long HI = (long)H * I;
    double* gw = (double*)calloc((size_t)n_tok * k + 1, sizeof(double));
    double* da = (double*)calloc((size_t)n_tok * k * H + 1, sizeof(double));
    expert_w W, WB;
    if (!gw || !da || alloc_expert(&W, HI) || alloc_expert(&WB, HI)) return ORC_ERR;
    for (int e = 0; e < E; ++e) {
        int used = 0;
        for (int q = 0; q < n_tok && !used; ++q)
            for (int j = 0; j < k; ++j) used |= idx[(long)tok[q] * k + j] == e;
        for (int q = 0; q < n_col && !used; ++q) used |= col_e[q] == e;
        if (!used) continue;
        load_expert(Wg, Wu, Wd, 0, e, H, I, ORC_MXFP8, &W);
        load_expert(Wg, Wu, Wd, 0, e, H, I, ORC_BF16, &WB);
        mx_roundtrip_rows(WB.g, H, I);
        mx_roundtrip_rows(WB.u, H, I);
        mx_roundtrip_rows(WB.d, I, H);
        /* ---- the sampled tokens' rows through this expert */
        for (int q = 0; q < n_tok; ++q) {
            int t = tok[q];
            for (int j = 0; j < k; ++j) {
                if (idx[(long)t * k + j] != e) continue;
                double* af = (double*)malloc(sizeof(double) * H);
                double* G = (double*)malloc(sizeof(double) * I);
                double* U = (double*)malloc(sizeof(double) * I);
                double* hq = (double*)malloc(sizeof(double) * I);
                double* y = (double*)malloc(sizeof(double) * H);
                double* dyq = (double*)malloc(sizeof(double) * H);
                double* dg = (double*)malloc(sizeof(double) * I);
                double* du = (double*)malloc(sizeof(double) * I);
                act_row(x, 0, t, H, ORC_MXFP8, af);
                ffn_row(af, &W, H, I, ORC_MXFP8, G, U, hq, y);
                double wj = w[(long)t * k + j], g = 0.0;
                for (int c = 0; c < H; ++c) {
                    double dYv = bf16_to_f64(dY[(long)t * H + c]);
                    g += dYv * y[c];
                    dyq[c] = orc_round_bf16(wj * dYv);
                }
                gw[(long)q * k + j] = g;
                mx_roundtrip_vec(dyq, H);
#pragma omp parallel for schedule(static)
                for (int i = 0; i < I; ++i) {
                    double dh = 0.0;
                    const double* dr = WB.d + (long)i * H;
                    for (int c = 0; c < H; ++c) dh += dyq[c] * dr[c];
                    double sg = 1.0 / (1.0 + exp(-G[i]));
                    dg[i] = orc_round_bf16(dh * U[i] * sg * (1.0 + G[i] * (1.0 - sg)));
                    du[i] = orc_round_bf16(dh * G[i] * sg);
                }
                mx_roundtrip_vec(dg, I);
                mx_roundtrip_vec(du, I);
                double* dar = da + ((long)q * k + j) * H;
#pragma omp parallel for schedule(static)
                for (int c = 0; c < H; ++c) {
                    const double* gr = WB.g + (long)c * I;
                    const double* ur = WB.u + (long)c * I;
                    double sacc = 0.0;
                    for (int i = 0; i < I; ++i) sacc += dg[i] * gr[i] + du[i] * ur[i];
                    dar[c] = sacc;
                }
                free(af); free(G); free(U); free(hq); free(y); free(dyq); free(dg); free(du);
            }
        }
        /* ---- the sampled weight-gradient columns of this expert */
        int r0 = offsets[e], nr = offsets[e + 1] - offsets[e];
        for (int qc = 0; qc < n_col; ++qc) {
            if (col_e[qc] != e) continue;
            int i = col_i[qc];
            double* og = dWg_s + (long)qc * H;
            double* ou = dWu_s + (long)qc * H;
            double* od = dWd_s + (long)qc * H;
            for (int c = 0; c < H; ++c) { og[c] = 0.0; ou[c] = 0.0; od[c] = 0.0; }
            if (nr == 0) continue;
            double* A = (double*)malloc(sizeof(double) * (size_t)nr * H);
            double* DY = (double*)malloc(sizeof(double) * (size_t)nr * H);
            double* DGc = (double*)malloc(sizeof(double) * nr);
            double* DUc = (double*)malloc(sizeof(double) * nr);
            double* HBc = (double*)malloc(sizeof(double) * nr);
            if (!A || !DY || !DGc || !DUc || !HBc) return ORC_ERR;
#pragma omp parallel
            {
                double* af = (double*)malloc(sizeof(double) * H);
                double* dyq = (double*)malloc(sizeof(double) * H);
#pragma omp for schedule(static)
                for (int rr = 0; rr < nr; ++rr) {
                    int slot = row_src[r0 + rr];
                    int t = slot / k;
                    act_row(x, 0, t, H, ORC_BF16, A + (long)rr * H);
                    act_row(x, 0, t, H, ORC_MXFP8, af);
                    double Gv = 0.0, Uv = 0.0;
                    for (int hh = 0; hh < H; ++hh) {
                        Gv += af[hh] * W.g[(long)hh * I + i];
                        Uv += af[hh] * W.u[(long)hh * I + i];
                    }
                    HBc[rr] = orc_round_bf16(silu(Gv) * Uv);
                    for (int c = 0; c < H; ++c) {
                        DY[(long)rr * H + c] = orc_round_bf16(w[slot] * bf16_to_f64(dY[(long)t * H + c]));
                        dyq[c] = DY[(long)rr * H + c];
                    }
                    mx_roundtrip_vec(dyq, H);
                    double dh = 0.0;
                    for (int c = 0; c < H; ++c) dh += dyq[c] * WB.d[(long)i * H + c];
                    double sg = 1.0 / (1.0 + exp(-Gv));
                    DGc[rr] = orc_round_bf16(dh * Uv * sg * (1.0 + Gv * (1.0 - sg)));
                    DUc[rr] = orc_round_bf16(dh * Gv * sg);
                }
                free(af); free(dyq);
            }
            mx_roundtrip_cols(A, nr, H);
            mx_roundtrip_cols(DY, nr, H);
            mx_roundtrip_cols(DGc, nr, 1);
            mx_roundtrip_cols(DUc, nr, 1);
            mx_roundtrip_cols(HBc, nr, 1);
            for (int rr = 0; rr < nr; ++rr)
                for (int c = 0; c < H; ++c) {
                    og[c] += A[(long)rr * H + c] * DGc[rr];
                    ou[c] += A[(long)rr * H + c] * DUc[rr];
                    od[c] += HBc[rr] * DY[(long)rr * H + c];
                }
            free(A); free(DY); free(DGc); free(DUc); free(HBc);
        }
    }
    free_expert(&W);
    free_expert(&WB);
    /* ---- dX rows: the token's da rows plus the router term */
    for (int q = 0; q < n_tok; ++q) {
        int t = tok[q];
        double m = 0.0;
        for (int j = 0; j < k; ++j) m += w[(long)t * k + j] * gw[(long)q * k + j];
        double* o = dX_s + (long)q * H;
        for (int c = 0; c < H; ++c) {
            double sacc = 0.0;
            for (int j = 0; j < k; ++j) sacc += da[((long)q * k + j) * H + c];
            for (int j = 0; j < k; ++j) {
                double dl = w[(long)t * k + j] * (gw[(long)q * k + j] - m);
                sacc += dl * (double)W_r[(long)c * E + idx[(long)t * k + j]];
            }
            o[c] = sacc;
        }
    }
    free(gw);
    free(da);
    return ORC_OK;
}

/* Columns dW_r[:, e] of the router gradient for the experts listed in
 * `col_e` (n_col of them), computed for inputs too large for the full
 * backward. The column of expert e sums x[t] * dl[t, j] over the tokens t
 * whose slot j chose e, and dl[t, j] = w_j (gw_j - sum_i w_i gw_i) needs
 * gw[t, i] = <dY[t], y[t, i]> for all k slots of such a token: so every
 * routed row of every token that chose a listed expert is run through its
 * expert (the forward's own row step, with the BF16 rounding of h in mode 0),
 * expert by expert in layout order. Sums over tokens run in ascending token
 * order. Inputs as in orc_moe_backward_sampled; out: dWr_cols [n_col, H]. */
int orc_router_grad_columns(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                            const uint16_t* dY, int T, int H, int I, int E, int k, const int32_t* idx,
                            const double* w, const int32_t* offsets, const int32_t* row_src, int mode,
                            const int32_t* col_e, int n_col, double* dWr_cols) {
    if (mode != ORC_BF16 && mode != ORC_EXACT) return ORC_ERR;
    for (int q = 0; q < n_col; ++q)
        if (col_e[q] < 0 || col_e[q] >= E) return ORC_ERR;
    unsigned char* need = (unsigned char*)calloc((size_t)(T > 0 ? T : 1), 1);
    double* gw = (double*)calloc((size_t)T * k + 1, sizeof(double));
    if (!need || !gw) { free(need); free(gw); return ORC_ERR; }
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j)
            for (int q = 0; q < n_col; ++q)
                if (idx[(long)t * k + j] == col_e[q]) need[t] = 1;
    long HI = (long)H * I;
    expert_w W;
    if (alloc_expert(&W, HI)) { free(need); free(gw); return ORC_ERR; }
    for (int e = 0; e < E; ++e) {
        int r0 = offsets[e], r1 = offsets[e + 1];
        int any = 0;
        for (int r = r0; r < r1 && !any; ++r) any = need[row_src[r] / k];
        if (!any) continue;
        load_expert(Wg, Wu, Wd, 0, e, H, I, mode, &W);
#pragma omp parallel
        {
            double* a = (double*)malloc(sizeof(double) * H);
            double* G = (double*)malloc(sizeof(double) * I);
            double* U = (double*)malloc(sizeof(double) * I);
            double* hb = (double*)malloc(sizeof(double) * I);
            double* y = (double*)malloc(sizeof(double) * H);
#pragma omp for schedule(dynamic, 1)
            for (int r = r0; r < r1; ++r) {
                int slot = row_src[r];
                int t = slot / k;
                if (!need[t]) continue;
                act_row(x, 0, t, H, ORC_BF16, a);
                ffn_row(a, &W, H, I, mode, G, U, hb, y);
                double g = 0.0;
                for (int c = 0; c < H; ++c) g += bf16_to_f64(dY[(long)t * H + c]) * y[c];
                gw[slot] = g;
            }
            free(a); free(G); free(U); free(hb); free(y);
        }
    }
    free_expert(&W);
    for (int q = 0; q < n_col; ++q) {
        double* o = dWr_cols + (long)q * H;
        for (int c = 0; c < H; ++c) o[c] = 0.0;
    }
    for (int t = 0; t < T; ++t) {
        if (!need[t]) continue;
        double m = 0.0;
        for (int j = 0; j < k; ++j) m += w[(long)t * k + j] * gw[(long)t * k + j];
        for (int j = 0; j < k; ++j) {
            double dl = w[(long)t * k + j] * (gw[(long)t * k + j] - m);
            for (int q = 0; q < n_col; ++q) {
                if (idx[(long)t * k + j] != col_e[q]) continue;
                double* o = dWr_cols + (long)q * H;
                for (int c = 0; c < H; ++c) o[c] += bf16_to_f64(x[(long)t * H + c]) * dl;
            }
        }
    }
    free(need);
    free(gw);
    return ORC_OK;
}

/* Number of threads the OpenMP runtime will use. */
int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
