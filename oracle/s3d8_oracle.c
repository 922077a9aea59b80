/*
 * Plain CPU oracle for the S3D8 W2.7A8 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the package smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Everything here is a direct, slow, scalar restatement of the definitions on
 * two pages:
 *   [P]  "Llama-Mobile: Efficient 2.7-Bit Quantization of VLMs" (arXiv
 *        2608.21134), section 3.4 "The S3D8 Format", Equation 1 and the
 *        domains that follow it; section 4.3 for Y = X W^T.
 *   [B]  "11 billion parameters on a phone" (Graphcore Research blog), section
 *        "S3D8 design notes" -> "Bit layout" and "Output channel packing", and
 *        the fused matrix-vector example (scale dtypes and epilogue order).
 *
 * Readings taken where the pages leave a step open (each is listed with its
 * reason in the design notes of the repository):
 *   - bits 1..5 of a byte hold Q with Q0 at bit 1 (so I0 = 2Q + S0 and
 *     I1 = 32 S1 + Q are both plain indices, as [B] "Bit layout" states);
 *   - sign selector 0 means +, 1 means - ([B] "Bit layout");
 *   - byte (g, k) carries output channels 3g, 3g+1, 3g+2 at input column k,
 *     selector S_d and centroid column d going with channel 3g+d
 *     ([P] Eq. 1: C[q][i mod 3]; [B] "Output channel packing");
 *   - N is padded up to 3*ceil(N/3); the padded lanes never reach an output;
 *   - activations: one fp32 scale per token row, s = absmax / 127 (the same
 *     absmax rule [P] gives for the weight channel scale alpha), q =
 *     round-half-even(x / s) clamped to [-127, 127]; an all-zero row gives
 *     s = 0 and q = 0;
 *   - output: out[m,n] = xscale[m] * acc[m,n] * chan_scale[n], evaluated here
 *     in fp64 (the GPU evaluates it in fp32 and rounds once to bf16);
 *   - direct-cast encoder ([P] section 3.4 "Quantization", the forward-pass
 *     assignment with frozen centroids): alpha is rounded to bf16 (the stored
 *     scale) and the scaled magnitudes divide by that stored value; the
 *     squared distances are fp32 sums in the order d = 0, 1, 2, so that the
 *     GPU can take every argmin decision in the same arithmetic;
 *   - centroid fit ([P] section 3.4 "Quantization": Lloyd-Max with k-means++
 *     initialisation on the zero-padded |W|/alpha 3-vectors, then Round):
 *     the random draws are 32 caller-supplied 32-bit integers; D^2 weights
 *     and cluster sums are taken on a fixed-point grid of 2^-20 (floor), so
 *     that every sum is an exact integer and any summation order gives the
 *     same result; a mean is RN(RN(sum / count) * 2^-20) in fp64, then
 *     rounded to fp32; an empty cluster keeps its centroid; the iteration
 *     count is fixed by the caller; Round is to nearest, ties to even,
 *     clamped to 0..127;
 *   - fake-quant forward ([P] section 3.4, QAT: the weight is quantised in
 *     the forward pass and reconstructed by Eq. 1): W_hat = s alpha C[q][n mod
 *     3] from the direct cast, the product alpha C formed in fp32 (exact: at
 *     most 15 significant bits) and rounded once to bf16 (the training
 *     matmul's dtype); the straight-through backward passes the gradient of
 *     W_hat to the weights unchanged, so it needs no code here.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math, no
 * FMA contraction, so that the fp32 activation quantiser is plain IEEE
 * single-precision division and rounding on every host).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bfloat16 is the upper half of an IEEE binary32; widening is exact. */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ---------------------------------------------------------------------------
 * Byte layout, [B] "Bit layout": the byte is [S2 xor S0, S1, Q4..Q0, S0] from
 * bit 7 down to bit 0.
 * ------------------------------------------------------------------------- */

/* Split one packed byte into its centroid index Q and the three sign
 * selectors S0, S1, S2. */
void s3d8o_byte_fields(uint8_t b, int32_t *Q, int32_t *S0, int32_t *S1, int32_t *S2)
{
    int s0 = b & 1;                 /* bit 0            */
    int q = (b >> 1) & 31;          /* bits 1..5        */
    int s1 = (b >> 6) & 1;          /* bit 6            */
    int s2_xor_s0 = (b >> 7) & 1;   /* bit 7            */
    *Q = q;
    *S0 = s0;
    *S1 = s1;
    *S2 = s2_xor_s0 ^ s0;           /* recover S2       */
}

/* Inverse of s3d8o_byte_fields: build the byte from its fields. */
uint8_t s3d8o_pack_byte(int32_t Q, int32_t S0, int32_t S1, int32_t S2)
{
    return (uint8_t)((S0 & 1) | ((Q & 31) << 1) | ((S1 & 1) << 6) | (((S2 ^ S0) & 1) << 7));
}

/* One decoded INT8 weight: component d (0, 1, 2) of the byte, i.e. the
 * s * C[Q][d] factor of [P] Eq. 1 without the channel scale alpha.
 * C is the 32 x 3 absolute-value centroid table, row-major C[q*3 + d]. */
int32_t s3d8o_decode_component(uint8_t b, const int8_t *C, int32_t d)
{
    int32_t Q, S[3];
    s3d8o_byte_fields(b, &Q, &S[0], &S[1], &S[2]);
    int32_t c = C[Q * 3 + d];
    return S[d] ? -c : c;
}

/* Dense INT8 weight matrix W[n, k] (n < N) from packed[G, K], G = ceil(N/3).
 * Output row n comes from packed row n / 3, component n % 3 ([P] Eq. 1 with
 * q_{floor(i/3), j} and C_{q, i mod 3}). */
void s3d8o_decode(const uint8_t *packed, const int8_t *C, int64_t N, int64_t K, int8_t *w)
{
    for (int64_t n = 0; n < N; ++n) {
        int64_t g = n / 3;
        int32_t d = (int32_t)(n % 3);
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = (int8_t)s3d8o_decode_component(packed[g * K + k], C, d);
    }
}

/* Pack a dense sign/index description into bytes.
 *   Q[G, K]     centroid index per (group, column), 0..31
 *   S[3G, K]    sign selector per (channel, column), 0 or 1 (padded channels
 *               included, so that the caller controls every bit)
 * Output packed[G, K]. */
void s3d8o_pack(const int32_t *Q, const int32_t *S, int64_t G, int64_t K, uint8_t *packed)
{
    for (int64_t g = 0; g < G; ++g)
        for (int64_t k = 0; k < K; ++k)
            packed[g * K + k] = s3d8o_pack_byte(Q[g * K + k], S[(3 * g + 0) * K + k],
                                                S[(3 * g + 1) * K + k], S[(3 * g + 2) * K + k]);
}

/* ---------------------------------------------------------------------------
 * Activation quantisation (per-token absmax INT8), fp32 throughout.
 * x is bf16 bit patterns, row-major [M, K].
 * ------------------------------------------------------------------------- */
void s3d8o_quantize_act(const uint16_t *x, int64_t M, int64_t K, int8_t *xq, float *xscale)
{
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = x + m * K;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(bf16_bits_to_float(row[k]));
            if (a > amax)
                amax = a;
        }
        float s = amax / 127.0f;
        xscale[m] = s;
        for (int64_t k = 0; k < K; ++k) {
            int32_t q = 0;
            if (s != 0.0f) {
                float r = rintf(bf16_bits_to_float(row[k]) / s); /* ties to even */
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                q = (int32_t)r;
            }
            xq[m * K + k] = (int8_t)q;
        }
    }
}

/* ---------------------------------------------------------------------------
 * The linear layer, Y = X W^T ([P] section 4.3), split into the exact integer
 * accumulation and the scaled output.
 * ------------------------------------------------------------------------- */

/* acc[m, n] = sum_k xq[m, k] * Wq[n, k] in int64, Wq decoded byte by byte.
 * Returns the number of accumulators that fall outside int32. */
int64_t s3d8o_linear_acc(const uint8_t *packed, const int8_t *C, const int8_t *xq,
                         int64_t M, int64_t N, int64_t K, int64_t *acc)
{
    int64_t out_of_range = 0;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t g = n / 3;
            int32_t d = (int32_t)(n % 3);
            int64_t sum = 0;
            for (int64_t k = 0; k < K; ++k)
                sum += (int64_t)xq[m * K + k] *
                       (int64_t)s3d8o_decode_component(packed[g * K + k], C, d);
            acc[m * N + n] = sum;
            if (sum > INT32_MAX || sum < INT32_MIN)
                ++out_of_range;
        }
    }
    return out_of_range;
}

/* Same sum for a list of (m, n) pairs only, for spot checks at full size. */
void s3d8o_linear_acc_at(const uint8_t *packed, const int8_t *C, const int8_t *xq,
                         int64_t M, int64_t N, int64_t K,
                         const int64_t *ms, const int64_t *ns, int64_t count, int64_t *acc)
{
    (void)M;
    (void)N;
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = ms[i], n = ns[i];
        int64_t g = n / 3;
        int32_t d = (int32_t)(n % 3);
        int64_t sum = 0;
        for (int64_t k = 0; k < K; ++k)
            sum += (int64_t)xq[m * K + k] *
                   (int64_t)s3d8o_decode_component(packed[g * K + k], C, d);
        acc[i] = sum;
    }
}

/* out[m, n] = xscale[m] * acc[m, n] * alpha[n], in fp64 (exact products of the
 * stored fp32 / bf16 / integer values up to one fp64 rounding each).
 * chan_scale is bf16 bit patterns [N]. */
void s3d8o_linear_out(const int64_t *acc, const float *xscale, const uint16_t *chan_scale,
                      int64_t M, int64_t N, double *out)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            out[m * N + n] = (double)xscale[m] * (double)acc[m * N + n] *
                             (double)bf16_bits_to_float(chan_scale[n]);
}


/* ---------------------------------------------------------------------------
 * Direct-cast encoder, [P] section 3.4 "Quantization" (forward pass with the
 * centroids frozen).  w is bf16 bit patterns [N, K], row-major.
 *   alpha_n = max_k |W_nk| / 127 (fp32 division), stored as bf16 (round to
 *             nearest even): chan_scale[n];
 *   W'_{g,k,d} = |W_{3g+d,k}| / alpha_{3g+d}, with the stored alpha, in fp32;
 *             0 when that alpha is 0 and for the padded channels 3g+d >= N;
 *   s = +1 for W >= 0 (selector 0), -1 otherwise (selector 1); padded: 0;
 *   q = argmin over l of ((C[l][0] - W'_0)^2 + (C[l][1] - W'_1)^2)
 *       + (C[l][2] - W'_2)^2, each operation rounded in fp32, the lowest
 *       index winning a tie.
 * packed is [ceil(N/3), K]; the byte follows [B] "Bit layout".
 * ------------------------------------------------------------------------- */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float centroid_dist2(const int8_t *Crow, const float *wp)
{
    float t0 = (float)Crow[0] - wp[0];
    float t1 = (float)Crow[1] - wp[1];
    float t2 = (float)Crow[2] - wp[2];
    float s = t0 * t0;
    s = s + t1 * t1;
    s = s + t2 * t2;
    return s;
}

/* Returns 0, or -1 when the scratch for the scales cannot be allocated. */
int32_t s3d8o_encode(const uint16_t *w, const int8_t *C, int64_t N, int64_t K, uint8_t *packed,
                     uint16_t *chan_scale)
{
    float *alpha = (float *)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
    if (!alpha)
        return -1;
    for (int64_t n = 0; n < N; ++n) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(bf16_bits_to_float(w[n * K + k]));
            if (a > amax)
                amax = a;
        }
        chan_scale[n] = float_to_bf16_rne(amax / 127.0f);
        alpha[n] = bf16_bits_to_float(chan_scale[n]);
    }
    const int64_t G = (N + 2) / 3;
    for (int64_t g = 0; g < G; ++g)
        for (int64_t k = 0; k < K; ++k) {
            float wp[3];
            int32_t sel[3];
            for (int d = 0; d < 3; ++d) {
                const int64_t n = 3 * g + d;
                wp[d] = 0.0f;
                sel[d] = 0;
                if (n < N) {
                    const float v = bf16_bits_to_float(w[n * K + k]);
                    sel[d] = (v >= 0.0f) ? 0 : 1;
                    if (alpha[n] != 0.0f)
                        wp[d] = fabsf(v) / alpha[n];
                }
            }
            int32_t best = 0;
            float bestd = centroid_dist2(C, wp);
            for (int32_t l = 1; l < 32; ++l) {
                const float dl = centroid_dist2(C + 3 * l, wp);
                if (dl < bestd) {
                    bestd = dl;
                    best = l;
                }
            }
            packed[g * K + k] = s3d8o_pack_byte(best, sel[0], sel[1], sel[2]);
        }
    free(alpha);
    return 0;
}


/* ---------------------------------------------------------------------------
 * Centroid fit, [P] section 3.4 "Quantization": C = Round(Lloyd-Max({W'})),
 * Lloyd-Max started from k-means++ (Arthur and Vassilvitskii, "k-means++: the
 * advantages of careful seeding", SODA 2007).
 *
 * Points: p = g K + k for packed row g and column k, W'_p = (|W[3g+d,k]| /
 * alpha_{3g+d})_{d=0,1,2} exactly as in the encoder (alpha stored as bf16;
 * padded channels and alpha = 0 give 0).  Np = ceil(N/3) K points.
 *
 * k-means++: centre 0 is point floor(r[0] Np / 2^32).  For t = 1..31, with
 * D2_p the fp32 squared distance from p to its nearest chosen centre and
 * w_p = floor(D2_p 2^20), S = sum w_p: centre t is the first point whose
 * inclusive prefix sum of w exceeds floor(r[t] S / 2^32), i.e. point p with
 * probability w_p / S; if S = 0 it is point floor(r[t] Np / 2^32).
 *
 * Lloyd: `iters` times, assign every point to its nearest centroid (fp32
 * distance as in the encoder, lowest index on a tie), then move each centroid
 * with a nonempty cluster to the mean of its points: per component,
 * float(RN(RN(sum_p floor(W'_pd 2^20) / n) 2^-20)) with the division in fp64.
 *
 * Outputs the fp32 centroids (cf, 32 x 3) and C = clamp(rint(cf), 0, 127).
 * Returns 0, or -1 when scratch cannot be allocated.
 * ------------------------------------------------------------------------- */
static float fdist2(const float *c, const float *w)
{
    float t0 = c[0] - w[0];
    float t1 = c[1] - w[1];
    float t2 = c[2] - w[2];
    float s = t0 * t0;
    s = s + t1 * t1;
    s = s + t2 * t2;
    return s;
}

/* floor(r x / 2^32) for r < 2^32, x < 2^62, in 64-bit integers */
static uint64_t scale_draw(uint32_t r, uint64_t x)
{
    const uint64_t hi = x >> 32, lo = x & 0xFFFFFFFFu;
    return (uint64_t)r * hi + (((uint64_t)r * lo) >> 32);
}

static void scaled_points(const uint16_t *w, int64_t N, int64_t K, float *P)
{
    const int64_t G = (N + 2) / 3;
    float alpha[3];
    for (int64_t g = 0; g < G; ++g) {
        for (int d = 0; d < 3; ++d) {
            const int64_t n = 3 * g + d;
            alpha[d] = 0.0f;
            if (n < N) {
                float amax = 0.0f;
                for (int64_t k = 0; k < K; ++k) {
                    float a = fabsf(bf16_bits_to_float(w[n * K + k]));
                    if (a > amax)
                        amax = a;
                }
                alpha[d] = bf16_bits_to_float(float_to_bf16_rne(amax / 127.0f));
            }
        }
        for (int64_t k = 0; k < K; ++k)
            for (int d = 0; d < 3; ++d) {
                const int64_t n = 3 * g + d;
                float v = 0.0f;
                if (n < N && alpha[d] != 0.0f)
                    v = fabsf(bf16_bits_to_float(w[n * K + k])) / alpha[d];
                P[3 * (g * K + k) + d] = v;
            }
    }
}

int32_t s3d8o_fit_centroids(const uint16_t *w, int64_t N, int64_t K, const uint32_t *r,
                            int32_t iters, float *cf, int8_t *C)
{
    const int64_t Np = ((N + 2) / 3) * K;
    float *P = (float *)malloc((size_t)Np * 3 * sizeof(float));
    float *D2 = (float *)malloc((size_t)Np * sizeof(float));
    if (!P || !D2) {
        free(P);
        free(D2);
        return -1;
    }
    scaled_points(w, N, K, P);

    /* k-means++ */
    int64_t idx = (int64_t)scale_draw(r[0], (uint64_t)Np);
    memcpy(cf, P + 3 * idx, 3 * sizeof(float));
    for (int64_t p = 0; p < Np; ++p)
        D2[p] = fdist2(cf, P + 3 * p);
    for (int t = 1; t < 32; ++t) {
        uint64_t S = 0;
        for (int64_t p = 0; p < Np; ++p)
            S += (uint64_t)(D2[p] * 1048576.0f);
        if (S == 0) {
            idx = (int64_t)scale_draw(r[t], (uint64_t)Np);
        } else {
            const uint64_t target = scale_draw(r[t], S);
            uint64_t run = 0;
            idx = Np - 1;
            for (int64_t p = 0; p < Np; ++p) {
                run += (uint64_t)(D2[p] * 1048576.0f);
                if (run > target) {
                    idx = p;
                    break;
                }
            }
        }
        memcpy(cf + 3 * t, P + 3 * idx, 3 * sizeof(float));
        for (int64_t p = 0; p < Np; ++p) {
            const float d = fdist2(cf + 3 * t, P + 3 * p);
            if (d < D2[p])
                D2[p] = d;
        }
    }

    /* Lloyd-Max */
    for (int32_t it = 0; it < iters; ++it) {
        uint64_t sum[32][3];
        uint64_t cnt[32];
        memset(sum, 0, sizeof sum);
        memset(cnt, 0, sizeof cnt);
        for (int64_t p = 0; p < Np; ++p) {
            int best = 0;
            float bestd = fdist2(cf, P + 3 * p);
            for (int l = 1; l < 32; ++l) {
                const float d = fdist2(cf + 3 * l, P + 3 * p);
                if (d < bestd) {
                    bestd = d;
                    best = l;
                }
            }
            cnt[best] += 1;
            for (int d = 0; d < 3; ++d)
                sum[best][d] += (uint64_t)(P[3 * p + d] * 1048576.0f);
        }
        for (int l = 0; l < 32; ++l)
            if (cnt[l] > 0)
                for (int d = 0; d < 3; ++d) {
                    const double mean = (double)sum[l][d] / (double)cnt[l];
                    cf[3 * l + d] = (float)(mean * 0x1p-20);
                }
    }
    for (int i = 0; i < 96; ++i) {
        float v = rintf(cf[i]);
        if (v < 0.0f)
            v = 0.0f;
        if (v > 127.0f)
            v = 127.0f;
        C[i] = (int8_t)v;
    }
    free(P);
    free(D2);
    return 0;
}


/* ---------------------------------------------------------------------------
 * Fake-quant forward, [P] section 3.4 "Quantization" (QAT phase: quantise in
 * the forward pass with the centroids frozen, reconstruct by Eq. 1):
 * w_hat[n,k] = bf16_rn(s * alpha_n * C[q][n mod 3]) with (alpha, s, q) from
 * s3d8o_encode.  Returns 0, or -1 when scratch cannot be allocated.
 * ------------------------------------------------------------------------- */
int32_t s3d8o_fake_quant(const uint16_t *w, const int8_t *C, int64_t N, int64_t K,
                         uint16_t *w_hat)
{
    const int64_t G = (N + 2) / 3;
    uint8_t *packed = (uint8_t *)malloc((size_t)(G > 0 ? G : 1) * (size_t)K);
    uint16_t *cs = (uint16_t *)malloc((size_t)(N > 0 ? N : 1) * sizeof(uint16_t));
    if (!packed || !cs || s3d8o_encode(w, C, N, K, packed, cs) != 0) {
        free(packed);
        free(cs);
        return -1;
    }
    for (int64_t n = 0; n < N; ++n) {
        const float alpha = bf16_bits_to_float(cs[n]);
        for (int64_t k = 0; k < K; ++k) {
            const int32_t wq = s3d8o_decode_component(packed[(n / 3) * K + k], C, (int32_t)(n % 3));
            w_hat[n * K + k] = float_to_bf16_rne(alpha * (float)wq);
        }
    }
    free(packed);
    free(cs);
    return 0;
}
