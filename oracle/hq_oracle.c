/*
 * hq_oracle.c -- plain, slow, scalar CPU reference of the quantized
 * speculative-verify linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU baseline of the
 * benchmark do.  It shares no code, header, table or constant generator with
 * the CUDA library; every value it needs it derives here from the definitions
 * below.
 *
 * Source of the method: "Karpathy's Trick for Faster Local LLMs Finally Has
 * Proper Tooling" (blog.dailydoseofds.com), section "How Uzu optimizes bytes
 * and tokens per pass":
 *   - Medium checkpoint: 4-bit asymmetric integer weights, grouped;
 *   - Large checkpoint: 8-bit symmetric integer weights;
 *   - activations quantized to 8 bits on the fly, so both matmul operands are
 *     integers;
 *   - a block-diagonal random Hadamard transform is applied before
 *     quantization: +1/-1 entries plus one overall scale, random sign flips
 *     before the mixing, blocks of 32 values, exactly invertible;
 *   - the transform block and the quantization group are independent sizes.
 * The page gives no formula.  The readings taken here (all plain):
 *   R1  the overall scale is the orthonormal one, 1/sqrt(32), rounded to fp32
 *       (bit pattern 0x3E3504F3) and applied after the +-1 butterfly;
 *   R2  one sign per input feature k, shared by weight rows and activation
 *       rows, so that (x R)(W R)^T = x W^T;
 *   R3  butterfly order: strides 1, 2, 4, 8, 16, every add/sub rounded to
 *       fp32, no fused multiply-add (compile with -ffp-contract=off);
 *   R4  activations: one scale per row over all K, symmetric range
 *       [-127, 127], round half to even, IEEE division;
 *   R5  Medium: per (output channel, group of G along K), range widened to
 *       include 0, scale = (hi-lo)/15, integer zero point z in [0, 15];
 *   R6  Large: per (output channel, group of G along K), scale = absmax/127;
 *   R7  all-zero rows / groups get scale 0 and codes 0 (no NaN);
 *   R8  per-group integer partial sums, then an fp32 epilogue that sums the
 *       scaled groups in ascending group order and multiplies by the row
 *       scale of the activations.
 *
 * Build: gcc -std=c99 -O2 -ffp-contract=off -fno-fast-math (optionally
 * -fopenmp; the pragmas below only split independent output rows).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_BLOCK 32

/* ------------------------------------------------------------------------ */
/* Signs: SplitMix64 (Steele, Lea & Flood, OOPSLA 2014; constants as in     */
/* Vigna's public splitmix64.c).  Output i decides the sign of feature i:   */
/* top bit set => -1.  Packed: bit (i % 32) of word i / 32.                 */
/* ------------------------------------------------------------------------ */
uint64_t or_splitmix64_next(uint64_t *state)
{
    uint64_t z;
    *state += 0x9E3779B97F4A7C15ULL;
    z = *state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

int or_make_signs(uint64_t seed, int K, uint32_t *signs)
{
    uint64_t st = seed;
    int i;
    if (K <= 0 || K % OR_BLOCK != 0 || !signs) return 1;
    for (i = 0; i < K / OR_BLOCK; ++i) signs[i] = 0u;
    for (i = 0; i < K; ++i) {
        uint64_t r = or_splitmix64_next(&st);
        if (r >> 63) signs[i / 32] |= (1u << (i % 32));
    }
    return 0;
}

static float or_sign_of(const uint32_t *signs, int k)
{
    return ((signs[k / 32] >> (k % 32)) & 1u) ? -1.0f : 1.0f;
}

static float or_hadamard_scale(void)
{
    /* fp32 nearest to 1/sqrt(32), given by its bit pattern (reading R1). */
    const uint32_t bits = 0x3E3504F3u;
    float c;
    memcpy(&c, &bits, sizeof c);
    return c;
}

/* Unnormalized Walsh-Hadamard butterfly on one block of 32, in place.
 * Stage h pairs index j (bit h clear) with j + h:
 *   (u_j, u_{j+h}) <- (u_j + u_{j+h}, u_j - u_{j+h}).
 * After the five stages u = v H with H the Sylvester matrix
 * H[i][j] = (-1)^popcount(i & j).                                          */
void or_fwht32(float *u)
{
    int h, j;
    for (h = 1; h < OR_BLOCK; h <<= 1) {
        for (j = 0; j < OR_BLOCK; ++j) {
            if ((j & h) == 0) {
                float a = u[j];
                float b = u[j + h];
                float s = a + b;
                float d = a - b;
                u[j] = s;
                u[j + h] = d;
            }
        }
    }
}

/* Forward rotation of one length-K vector: for every block of 32,
 * u = c * H (s o v)  (sign flip, butterfly, overall scale).                */
void or_rotate_vec(const float *v, int K, const uint32_t *signs, float *out)
{
    const float c = or_hadamard_scale();
    int b, j;
    for (b = 0; b < K / OR_BLOCK; ++b) {
        float u[OR_BLOCK];
        for (j = 0; j < OR_BLOCK; ++j) {
            int k = b * OR_BLOCK + j;
            u[j] = v[k] * or_sign_of(signs, k);
        }
        or_fwht32(u);
        for (j = 0; j < OR_BLOCK; ++j) out[b * OR_BLOCK + j] = u[j] * c;
    }
}

/* Inverse rotation: butterfly, overall scale, then the same sign flip
 * (H is symmetric and H H = 32 I, c^2 = 1/32).                             */
void or_rotate_inverse_vec(const float *u, int K, const uint32_t *signs, float *out)
{
    const float c = or_hadamard_scale();
    int b, j;
    for (b = 0; b < K / OR_BLOCK; ++b) {
        float t[OR_BLOCK];
        for (j = 0; j < OR_BLOCK; ++j) t[j] = u[b * OR_BLOCK + j];
        or_fwht32(t);
        for (j = 0; j < OR_BLOCK; ++j) {
            int k = b * OR_BLOCK + j;
            float y = t[j] * c;
            out[k] = y * or_sign_of(signs, k);
        }
    }
}

void or_rotate_rows(const float *V, int R, int K, const uint32_t *signs, float *out)
{
    int r;
    for (r = 0; r < R; ++r) or_rotate_vec(V + (size_t)r * K, K, signs, out + (size_t)r * K);
}

/* ------------------------------------------------------------------------ */
/* Quantizers on already-rotated values.                                     */
/* ------------------------------------------------------------------------ */

/* Round to nearest, ties to even, then clamp; NaN maps to 0. */
static float or_round_clamp(float x, float lo, float hi)
{
    float r = rintf(x);
    if (r != r) return 0.0f;
    if (r < lo) r = lo;
    if (r > hi) r = hi;
    return r;
}

/* Activation row (reading R4): a = max |u|; s = a / 127; q = rint(u / s). */
void or_quant_row_act(const float *u, int K, int8_t *q, float *s_out)
{
    float a = 0.0f, s;
    int k;
    for (k = 0; k < K; ++k) {
        float t = fabsf(u[k]);
        if (t > a) a = t;
    }
    if (a == 0.0f) {
        *s_out = 0.0f;
        for (k = 0; k < K; ++k) q[k] = 0;
        return;
    }
    s = a / 127.0f;
    *s_out = s;
    for (k = 0; k < K; ++k) q[k] = (int8_t)or_round_clamp(u[k] / s, -127.0f, 127.0f);
}

/* Medium group (reading R5): lo = min(0, min w), hi = max(0, max w),
 * scale = (hi - lo) / 15, z = rint(-lo / scale), q = rint(w / scale) + z.  */
void or_quant_group_asym4(const float *w, int n, uint8_t *q, float *scale_out, uint8_t *zero_out)
{
    float lo = 0.0f, hi = 0.0f, scale, z;
    int i;
    for (i = 0; i < n; ++i) {
        if (w[i] < lo) lo = w[i];
        if (w[i] > hi) hi = w[i];
    }
    scale = (hi - lo) / 15.0f;
    if (scale == 0.0f) {
        *scale_out = 0.0f;
        *zero_out = 0;
        for (i = 0; i < n; ++i) q[i] = 0;
        return;
    }
    z = or_round_clamp(-lo / scale, 0.0f, 15.0f);
    *scale_out = scale;
    *zero_out = (uint8_t)z;
    for (i = 0; i < n; ++i) {
        float r = rintf(w[i] / scale);
        if (r != r) r = 0.0f;
        q[i] = (uint8_t)or_round_clamp(r + z, 0.0f, 15.0f);
    }
}

/* Large group (reading R6): scale = absmax / 127, q = rint(w / scale). */
void or_quant_group_sym8(const float *w, int n, int8_t *q, float *scale_out)
{
    float a = 0.0f, scale;
    int i;
    for (i = 0; i < n; ++i) {
        float t = fabsf(w[i]);
        if (t > a) a = t;
    }
    if (a == 0.0f) {
        *scale_out = 0.0f;
        for (i = 0; i < n; ++i) q[i] = 0;
        return;
    }
    scale = a / 127.0f;
    *scale_out = scale;
    for (i = 0; i < n; ++i) q[i] = (int8_t)or_round_clamp(w[i] / scale, -127.0f, 127.0f);
}

/* ------------------------------------------------------------------------ */
/* The three stages of the layer.                                            */
/* ------------------------------------------------------------------------ */

static int or_shape_ok(int R, int K, int G)
{
    return R >= 0 && K > 0 && K % OR_BLOCK == 0 && G > 0 && K % G == 0;
}

/* Activations: rotate each row, quantize it, and sum the codes per group.
 * X [M][K] fp32 -> qx [M][K] int8, sx [M], gsum [M][K/G] int32.           */
int or_quant_act(const float *X, int M, int K, int G, const uint32_t *signs,
                 int8_t *qx, float *sx, int32_t *gsum)
{
    int m;
    if (!or_shape_ok(M, K, G)) return 1;
    for (m = 0; m < M; ++m) {
        float *u = (float *)malloc(sizeof(float) * (size_t)K);
        int8_t *q = qx + (size_t)m * K;
        int g, k;
        if (!u) return 2;
        or_rotate_vec(X + (size_t)m * K, K, signs, u);
        or_quant_row_act(u, K, q, &sx[m]);
        for (g = 0; g < K / G; ++g) {
            int32_t t = 0;
            for (k = g * G; k < (g + 1) * G; ++k) t += q[k];
            gsum[(size_t)m * (K / G) + g] = t;
        }
        free(u);
    }
    return 0;
}

/* Medium weights: W [N][K] fp32 -> codes [N][K] (0..15), scales [N][K/G],
 * zeros [N][K/G] (0..15).                                                   */
int or_quant_w4(const float *W, int N, int K, int G, const uint32_t *signs,
                uint8_t *codes, float *scales, uint8_t *zeros)
{
    int n;
    if (!or_shape_ok(N, K, G)) return 1;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (n = 0; n < N; ++n) {
        float *u = (float *)malloc(sizeof(float) * (size_t)K);
        int g;
        if (!u) continue;
        or_rotate_vec(W + (size_t)n * K, K, signs, u);
        for (g = 0; g < K / G; ++g) {
            size_t pi = (size_t)n * (K / G) + g;
            or_quant_group_asym4(u + (size_t)g * G, G, codes + (size_t)n * K + (size_t)g * G,
                                 &scales[pi], &zeros[pi]);
        }
        free(u);
    }
    return 0;
}

/* Large weights: W [N][K] fp32 -> codes [N][K] int8, scales [N][K/G]. */
int or_quant_w8(const float *W, int N, int K, int G, const uint32_t *signs,
                int8_t *codes, float *scales)
{
    int n;
    if (!or_shape_ok(N, K, G)) return 1;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (n = 0; n < N; ++n) {
        float *u = (float *)malloc(sizeof(float) * (size_t)K);
        int g;
        if (!u) continue;
        or_rotate_vec(W + (size_t)n * K, K, signs, u);
        for (g = 0; g < K / G; ++g) {
            size_t pi = (size_t)n * (K / G) + g;
            or_quant_group_sym8(u + (size_t)g * G, G, codes + (size_t)n * K + (size_t)g * G, &scales[pi]);
        }
        free(u);
    }
    return 0;
}

/* Per-group integer partial sums (reading R8), by brute force in int64:
 *   Medium: P[m][n][g] = sum_{k in g} qx[m][k] * (q[n][k] - z[n][g])
 *   Large:  P[m][n][g] = sum_{k in g} qx[m][k] * q[n][k]
 * codes is uint8 (Medium) or int8 (Large) viewed through `is_w4`.
 * Returns 3 if a partial does not fit in int32.                             */
int or_partials(const int8_t *qx, int M, const void *codes, const uint8_t *zeros,
                int N, int K, int G, int is_w4, int32_t *P)
{
    int m, overflow = 0;
    const int NG = K / G;
    if (!or_shape_ok(N, K, G) || M < 0) return 1;
    for (m = 0; m < M; ++m) {
        int n;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) reduction(| : overflow)
#endif
        for (n = 0; n < N; ++n) {
            int g;
            for (g = 0; g < NG; ++g) {
                int64_t acc = 0;
                int k;
                for (k = g * G; k < (g + 1) * G; ++k) {
                    int64_t a = qx[(size_t)m * K + k];
                    int64_t w;
                    if (is_w4)
                        w = (int64_t)((const uint8_t *)codes)[(size_t)n * K + k] - (int64_t)zeros[(size_t)n * NG + g];
                    else
                        w = (int64_t)((const int8_t *)codes)[(size_t)n * K + k];
                    acc += a * w;
                }
                if (acc > INT32_MAX || acc < INT32_MIN) overflow = 1;
                P[((size_t)m * N + n) * NG + g] = (int32_t)acc;
            }
        }
    }
    return overflow ? 3 : 0;
}

/* fp32 epilogue (reading R8): acc = sum over g ascending of
 * (scale[n][g] * float(P[m][n][g])), each product and sum rounded to fp32;
 * Y[m][n] = sx[m] * acc.                                                    */
int or_output(const int32_t *P, const float *sx, const float *scales, int M, int N, int NG, float *Y)
{
    int m;
    if (M < 0 || N < 0 || NG <= 0) return 1;
    for (m = 0; m < M; ++m) {
        int n;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (n = 0; n < N; ++n) {
            float acc = 0.0f;
            int g;
            for (g = 0; g < NG; ++g) {
                float p = (float)P[((size_t)m * N + n) * NG + g];
                float t = scales[(size_t)n * NG + g] * p;
                acc = acc + t;
            }
            Y[(size_t)m * N + n] = sx[m] * acc;
        }
    }
    return 0;
}

/* The integer GEMM and the epilogue in one call, without storing P: the
 * same arithmetic as or_partials followed by or_output, one output at a
 * time.  Used to time the reference on large shapes.                        */
int or_verify_gemm(const int8_t *qx, const float *sx, int M, const void *codes, const float *scales,
                   const uint8_t *zeros, int N, int K, int G, int is_w4, float *Y)
{
    int m, overflow = 0;
    const int NG = K / G;
    if (!or_shape_ok(N, K, G) || M < 0) return 1;
    for (m = 0; m < M; ++m) {
        int n;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) reduction(| : overflow)
#endif
        for (n = 0; n < N; ++n) {
            float acc = 0.0f;
            int g;
            for (g = 0; g < NG; ++g) {
                int64_t p = 0;
                int k;
                float t;
                for (k = g * G; k < (g + 1) * G; ++k) {
                    int64_t a = qx[(size_t)m * K + k];
                    int64_t w;
                    if (is_w4)
                        w = (int64_t)((const uint8_t *)codes)[(size_t)n * K + k] - (int64_t)zeros[(size_t)n * NG + g];
                    else
                        w = (int64_t)((const int8_t *)codes)[(size_t)n * K + k];
                    p += a * w;
                }
                if (p > INT32_MAX || p < INT32_MIN) overflow = 1;
                t = scales[(size_t)n * NG + g] * (float)(int32_t)p;
                acc = acc + t;
            }
            Y[(size_t)m * N + n] = sx[m] * acc;
        }
    }
    return overflow ? 3 : 0;
}

/* Number of OpenMP threads the oracle library uses (1 without OpenMP). */
/* ------------------------------------------------------------------------ */
/* Tree acceptance (section "Producing several tokens from one model pass"  */
/* and "Verifying a draft tree without restoring model state": the main    */
/* model checks the drafted positions together, accepts the valid prefix,  */
/* adds its own token at the first position it did not confirm; on a tree  */
/* it accepts the longest valid path).  Readings:                          */
/*   T1  node 0 is the root (the last committed token); every other node i */
/*       has a parent p[i] < i and a drafted token t[i];                   */
/*   T2  row i of the logits is the main model's output after node i; its  */
/*       greedy token g[i] = argmax_v logits[i][v], the lowest index among */
/*       equal maxima; a NaN counts as larger than every number (the first */
/*       NaN wins);                                                        */
/*   T3  node i >= 1 is valid when its parent is valid (the root is) and   */
/*       t[i] == g[p[i]];                                                  */
/*   T4  the accepted node is the deepest valid node, the lowest index     */
/*       among equally deep ones; the sequence advances by its depth (the  */
/*       accepted drafted tokens) plus one: the main model's own token g   */
/*       at the accepted node.                                             */
/* ------------------------------------------------------------------------ */
int or_argmax_rows(const float *logits, int M, int V, int32_t *g)
{
    if (M < 0 || V <= 0) return 1;
    for (int i = 0; i < M; ++i) {
        const float *row = logits + (size_t)i * (size_t)V;
        int best = 0;
        for (int v = 1; v < V; ++v) {
            const float a = row[v], b = row[best];
            if (isnan(b)) break;                 /* the first NaN wins */
            if (isnan(a) || a > b) best = v;     /* strictly greater: lowest index on ties */
        }
        g[i] = best;
    }
    return 0;
}

/* path[0..depth-1]: the accepted drafted nodes from the root's child down to
   the accepted node; *n_accept = depth; *bonus = g[accepted node]. */
int or_tree_accept(const int32_t *g, const int32_t *parent, const int32_t *tokens, int M, int32_t *path,
                   int32_t *n_accept, int32_t *bonus)
{
    if (M <= 0) return 1;
    int *valid = (int *)malloc(sizeof(int) * (size_t)M);
    int *depth = (int *)malloc(sizeof(int) * (size_t)M);
    if (!valid || !depth) { free(valid); free(depth); return 2; }
    valid[0] = 1;
    depth[0] = 0;
    for (int i = 1; i < M; ++i) {
        const int p = parent[i];
        if (p < 0 || p >= i) { free(valid); free(depth); return 1; }
        valid[i] = valid[p] && tokens[i] == g[p];
        depth[i] = depth[p] + 1;
    }
    int best = 0;
    for (int i = 1; i < M; ++i)
        if (valid[i] && depth[i] > depth[best]) best = i;
    *n_accept = depth[best];
    *bonus = g[best];
    for (int i = best, d = depth[best]; d > 0; i = parent[i], --d) path[d - 1] = i;
    free(valid);
    free(depth);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Tree-masked verify attention (section "Verifying a draft tree without    */
/* restoring model state": an attention layer keeps a cache of every past  */
/* token; the main model checks every branch of the draft tree in one pass */
/* and changes its committed state only for the accepted path).  The page  */
/* gives no mask and no formula.  Readings:                                */
/*   A1  the M tree nodes are processed in this pass; their keys and values */
/*       sit in the cache right after the L committed positions (node j at  */
/*       position L + j);                                                   */
/*   A2  node i attends to the L committed positions, to every ancestor of  */
/*       i and to i itself: exactly the prefix its own branch would have    */
/*       had if decoded alone (the plainest mask; siblings and cousins are  */
/*       not visible);                                                      */
/*   A3  the ancestor walk follows parent[] while the parent lies in        */
/*       [0, node); a parent outside that range ends the walk (the root,    */
/*       node 0, has none);                                                 */
/*   A4  attention itself is the textbook one: s = scale * (q . k),         */
/*       softmax over the visible positions, output = sum_j p_j v_j, with   */
/*       grouped heads: query head h reads key/value head h / (Hq / Hkv);   */
/*   A5  q, k, v are IEEE binary16 values; the arithmetic here is double.   */
/* Commit (section above: state is committed only along the chosen path):  */
/*   A6  the root stays at position L; accepted node path[d] (depth d + 1)  */
/*       moves to position L + 1 + d, for d < n_accept; nothing moves when  */
/*       n_accept <= 0.                                                     */
/* ------------------------------------------------------------------------ */
double or_half_to_double(uint16_t h)
{
    const int sgn = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);   /* (1 + m/1024) * 2^(e-15) */
    return sgn ? -v : v;
}

/* vis[i * M + j] = 1 when tree node j is visible to node i (A2, A3). */
static void or_tree_visibility(const int32_t *parent, int M, unsigned char *vis)
{
    for (int i = 0; i < M; ++i) {
        for (int j = 0; j < M; ++j) vis[(size_t)i * M + j] = 0;
        vis[(size_t)i * M + i] = 1;
        int cur = i;
        while (cur > 0) {
            const int p = parent[cur];
            if (p < 0 || p >= cur) break;
            vis[(size_t)i * M + p] = 1;
            cur = p;
        }
    }
}

/* q [M][Hq][D], k and v [Hkv][cap][D] (binary16 bit patterns), out [M][Hq][D]. */
int or_tree_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, int cap, int L, int M, int Hq,
                      int Hkv, int D, const int32_t *parent, double scale, double *out)
{
    if (M < 1 || L < 0 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0 || cap < L + M) return 1;
    const int G = Hq / Hkv;
    unsigned char *vis = (unsigned char *)malloc((size_t)M * (size_t)M);
    if (!vis) return 2;
    or_tree_visibility(parent, M, vis);
    int fail = 0;
#pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < M * Hq; ++r) {
        const int i = r / Hq, h = r % Hq, hk = h / G;
        double *s = (double *)malloc(sizeof(double) * (size_t)(L + M));
        int *pos = (int *)malloc(sizeof(int) * (size_t)(L + M));
        if (!s || !pos) {
            free(s);
            free(pos);
            fail = 1;
            continue;
        }
        int n = 0;
        for (int t = 0; t < L; ++t) pos[n++] = t;
        for (int j = 0; j < M; ++j)
            if (vis[(size_t)i * M + j]) pos[n++] = L + j;
        const uint16_t *qr = q + ((size_t)i * Hq + h) * D;
        double m = -INFINITY;
        for (int a = 0; a < n; ++a) {
            const uint16_t *kr = k + ((size_t)hk * cap + pos[a]) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += or_half_to_double(qr[d]) * or_half_to_double(kr[d]);
            s[a] = scale * dot;
            if (s[a] > m) m = s[a];
        }
        double den = 0.0;
        for (int a = 0; a < n; ++a) {
            s[a] = exp(s[a] - m);
            den += s[a];
        }
        double *o = out + ((size_t)i * Hq + h) * D;
        for (int d = 0; d < D; ++d) {
            double num = 0.0;
            for (int a = 0; a < n; ++a) num += s[a] * or_half_to_double(v[((size_t)hk * cap + pos[a]) * D + d]);
            o[d] = num / den;
        }
        free(s);
        free(pos);
    }
    free(vis);
    return fail ? 2 : 0;
}

/* In place on k and v [Hkv][cap][D] (A6). */
int or_tree_commit_kv(uint16_t *k, uint16_t *v, int cap, int L, int Hkv, int D, const int32_t *path, int n_accept)
{
    if (n_accept <= 0) return 0;
    if (L < 0 || Hkv < 1 || D < 1 || L + 1 + n_accept > cap) return 1;
    for (int d = 0; d < n_accept; ++d)
        if (path[d] < 1 || L + path[d] >= cap) return 1;
    uint16_t *tmp = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n_accept * (size_t)D);
    if (!tmp) return 2;
    for (int which = 0; which < 2; ++which) {
        uint16_t *c = which == 0 ? k : v;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < n_accept; ++d)
                memcpy(tmp + (size_t)d * D, c + ((size_t)h * cap + L + path[d]) * D, sizeof(uint16_t) * (size_t)D);
            for (int d = 0; d < n_accept; ++d)
                memcpy(c + ((size_t)h * cap + L + 1 + d) * D, tmp + (size_t)d * D, sizeof(uint16_t) * (size_t)D);
        }
    }
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Rollback-free DeltaNet tree pass (section "Verifying a draft tree        */
/* without restoring model state": a Gated DeltaNet layer compresses the   */
/* past into a fixed-size state that every accepted token changes; the     */
/* verify pass computes the outputs of every tree branch without changing  */
/* the live state, which is then updated only along the accepted path).    */
/* The page gives no equations.  Readings:                                 */
/*   D1  the recurrence is the published gated delta rule (Yang, Kautz and  */
/*       Hatamizadeh, "Gated Delta Networks", ICLR 2025), per head:         */
/*         S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T */
/*         o_t = S_t q_t                                                    */
/*       S is D x D (rows: value dimensions, columns: key dimensions);      */
/*       q, k, v, alpha, beta are inputs (their projections, gates and     */
/*       normalizations come before this step);                            */
/*   D2  on the tree, node i's state follows from its parent's state by one */
/*       step with node i's inputs; the root (node 0) and any node whose    */
/*       parent lies outside [0, i) follow from the committed state;        */
/*   D3  the committed state is only read; commit replaces it by the state  */
/*       of the accepted node, i.e. one step for the root and one for each  */
/*       accepted node path[0..n_accept) in order; nothing changes when     */
/*       n_accept < 0 (a malformed tree).                                   */
/* ------------------------------------------------------------------------ */
/* One step on a D x D state (row-major), in place. */
static void or_delta_step(double *S, int D, const float *k, const float *v, double alpha, double beta)
{
    double *u = (double *)malloc(sizeof(double) * (size_t)D);
    for (int r = 0; r < D; ++r) {
        double t = 0.0;
        for (int c = 0; c < D; ++c) t += S[(size_t)r * D + c] * (double)k[c];
        u[r] = t;                                   /* (S k)_r */
    }
    for (int r = 0; r < D; ++r)
        for (int c = 0; c < D; ++c)                 /* alpha S (I - beta k k^T) + beta v k^T */
            S[(size_t)r * D + c] = alpha * (S[(size_t)r * D + c] - beta * u[r] * (double)k[c]) +
                                   beta * (double)v[r] * (double)k[c];
    free(u);
}

/* state [H][D][D]; q, k, v [M][H][D]; alpha, beta [M][H]; out [M][H][D]. */
int or_delta_tree(const float *state, const float *q, const float *k, const float *v, const float *alpha,
                  const float *beta, const int32_t *parent, int M, int H, int D, double *out)
{
    if (M < 1 || H < 1 || D < 1) return 1;
    int fail = 0;
#pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < M * H; ++r) {
        const int i = r / H, h = r % H;
        int *chain = (int *)malloc(sizeof(int) * (size_t)M);
        double *S = (double *)malloc(sizeof(double) * (size_t)D * D);
        if (!chain || !S) { free(chain); free(S); fail = 1; continue; }
        int n = 0, cur = i;
        chain[n++] = cur;
        while (cur > 0) {
            const int p = parent[cur];
            if (p < 0 || p >= cur) break;
            chain[n++] = p;
            cur = p;
        }
        for (size_t e = 0; e < (size_t)D * D; ++e) S[e] = (double)state[(size_t)h * D * D + e];
        for (int a = n - 1; a >= 0; --a) {            /* from the top of the chain down to node i */
            const int j = chain[a];
            const size_t b = ((size_t)j * H + h) * D;
            or_delta_step(S, D, k + b, v + b, (double)alpha[(size_t)j * H + h], (double)beta[(size_t)j * H + h]);
        }
        const float *qi = q + ((size_t)i * H + h) * D;
        for (int rr = 0; rr < D; ++rr) {
            double t = 0.0;
            for (int c = 0; c < D; ++c) t += S[(size_t)rr * D + c] * (double)qi[c];
            out[((size_t)i * H + h) * D + rr] = t;
        }
        free(chain);
        free(S);
    }
    return fail ? 2 : 0;
}

/* state [H][D][D] in place (double); the root, then path[0..n_accept). */
int or_delta_commit(double *state, const float *k, const float *v, const float *alpha, const float *beta,
                    const int32_t *path, int n_accept, int M, int H, int D)
{
    if (n_accept < 0) return 0;
    if (n_accept >= M || H < 1 || D < 1) return 1;
    for (int d = 0; d < n_accept; ++d)
        if (path[d] < 1 || path[d] >= M) return 1;
    for (int h = 0; h < H; ++h) {
        double *S = state + (size_t)h * D * D;
        for (int a = -1; a < n_accept; ++a) {
            const int j = a < 0 ? 0 : path[a];
            const size_t b = ((size_t)j * H + h) * D;
            or_delta_step(S, D, k + b, v + b, (double)alpha[(size_t)j * H + h], (double)beta[(size_t)j * H + h]);
        }
    }
    return 0;
}

int or_num_threads(void)
{
#ifdef _OPENMP
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
#else
    return 1;
#endif
}
