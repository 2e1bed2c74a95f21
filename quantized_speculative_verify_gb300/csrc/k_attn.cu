// k_attn.cu -- tree-masked verify attention and the accepted-path KV commit.
//
// Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
// section "Verifying a draft tree without restoring model state": an
// attention layer keeps a cache of every past token; the main model checks
// every branch of the draft tree in one pass, and its state is committed only
// along the accepted path.  The page gives no mask: here node i attends to
// the L committed positions, to its ancestors and to itself (the prefix its
// branch would have had if decoded alone); an ancestor walk ends at a parent
// outside [0, node).
//
// Layout: q fp16 [M][Hq][D]; k, v fp16 [Hkv][cap][D], committed positions
// [0, L), tree node j at position L + j; out fp32 [M][Hq][D].  Grouped heads:
// query head h reads key/value head h / G, G = Hq / Hkv.  The query rows of
// one key/value head are r = node * G + g (query head hk * G + g); a thread
// block takes 64 of them and one contiguous chunk of key positions (split
// KV), and a second kernel merges the chunks.
//
// Split kernel: one producer thread loads each 64-key tile of K and V with
// four TMA tiled copies (boxes of 64 dimensions x 64 positions of one head,
// 128-byte swizzle, L2 evict-first) into a ring of shared-memory stages; in a
// swizzled box the 16-byte chunk c of row r sits at chunk c ^ (r mod 8), so
// the ldmatrix reads of eight rows hit eight different bank groups.  The
// tensor maps end at position L + M: rows past it arrive as zeros.  Four
// consumer warps each own 16 query rows: S = Q K^T and
// O += P V on fp16 tensor cores with fp32 accumulation, online softmax in
// base-2 units (s * scale * log2 e), P rounded to fp16 for the second
// product.  Each block writes its unnormalized O, running maximum and sum;
// the merge rescales and adds the chunks in ascending order.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "hq_internal.cuh"

namespace hq {
namespace {

constexpr int AD = HQ_ATTN_HEAD_DIM;          // head dimension
constexpr int AROWS = 64;                     // query rows per thread block
constexpr int AKEYS = 64;                     // key positions per stage
constexpr int ASTAGES = 3;
constexpr int ABOX_DIMS = 64;                 // dimensions per TMA box (128 bytes: the swizzle span)
constexpr int ABOX_BYTES = AKEYS * ABOX_DIMS * 2;  // 8 KB, a multiple of the 1024-byte swizzle atom
constexpr int ATILE_BYTES = (AD / ABOX_DIMS) * ABOX_BYTES;
constexpr int ASTAGE_BYTES = 2 * ATILE_BYTES;  // K tile, then V tile
constexpr int ACW = 4;                         // consumer warps, 16 rows each
constexpr int ATHREADS = (ACW + 1) * 32;
constexpr int AMAX_ROWS_SPLITS = 4096;         // splits x padded rows, per key/value head (workspace)
constexpr int AMAX_SPLITS = 64;
// the ring starts at the first 1024-byte boundary of the dynamic shared memory
constexpr size_t ASMEM = 1024 + (size_t)ASTAGES * ASTAGE_BYTES + 2 * ASTAGES * 8 + AROWS * 16 + HQ_MAX_M * 4;

struct AttnArgs {
    const __half *q, *k, *v;
    const int32_t *parent;
    float *ws_o;   // [NS][Hkv][rows_pad][AD]
    float *ws_ml;  // [NS][Hkv][rows_pad][2]: running maximum (base-2 units), sum
    int *err;
    int cap, L, M, Hq, Hkv, G, NS, chunk, rows_pad;
    float c_log2;  // scale * log2(e)
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16, fp16) * B(16x8, fp16) + D, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 3-D TMA tiled load (dimension, position, head) into shared memory,
// completing on `bar`.  x * 2 bytes is a multiple of 16 (x in {0, 64}).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// Byte offset of 16-byte chunk c (dimensions 8c .. 8c+7 of a box) of row r in
// a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__global__ void __launch_bounds__(ATHREADS, 2)
    k_tree_attn_split(const AttnArgs a, const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *ring = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + (size_t)ASTAGES * ASTAGE_BYTES);  // full[S], empty[S]
    uint32_t *s_anc = reinterpret_cast<uint32_t *>(bars + 2 * ASTAGES);                   // [AROWS][4]
    int32_t *s_par = reinterpret_cast<int32_t *>(s_anc + AROWS * 4);                      // [HQ_MAX_M]

    const int split = blockIdx.x, hk = blockIdx.y, rt = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = a.L + a.M;                      // key positions
    const int k0 = split * a.chunk;
    const int k1 = k0 + a.chunk < total ? k0 + a.chunk : total;
    const int ntiles = (k1 - k0 + AKEYS - 1) / AKEYS;
    const int npt = AROWS / a.G;                      // tree nodes per block
    const int node0 = rt * npt;

    if (threadIdx.x == 0) {
        for (int i = 0; i < ASTAGES; ++i) {
            mbar_init(smem_addr(&bars[i]), 1);
            mbar_init(smem_addr(&bars[ASTAGES + i]), ACW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == ACW) {
        // ------------------------------------------------------ producer ---
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            auto issue = [&](int i) {
                const int st = i % ASTAGES;
                const uint32_t kt = smem_addr(ring + (size_t)st * ASTAGE_BYTES);
                const uint32_t bar = smem_addr(&bars[st]);
                mbar_arrive_expect_tx(bar, (uint32_t)ASTAGE_BYTES);
#pragma unroll
                for (int bx = 0; bx < AD / ABOX_DIMS; ++bx) {
                    tma_load_3d(kt + bx * ABOX_BYTES, &tk, bx * ABOX_DIMS, k0 + i * AKEYS, hk, bar, pol);
                    tma_load_3d(kt + ATILE_BYTES + bx * ABOX_BYTES, &tv, bx * ABOX_DIMS, k0 + i * AKEYS, hk, bar, pol);
                }
            };
            // Committed positions are not written by the kernel before this
            // one (only the tree rows are): the first stages' tiles that lie
            // below L are loaded before waiting for it.
            int i = 0;
            for (; i < ntiles && i < ASTAGES && k0 + (i + 1) * AKEYS <= a.L; ++i) issue(i);
            pdl_wait();
            for (; i < ntiles; ++i) {
                const int st = i % ASTAGES;
                const uint32_t ph = (uint32_t)((i / ASTAGES) & 1);
                if (i >= ASTAGES && !mbar_wait_bounded(smem_addr(&bars[ASTAGES + st]), ph ^ 1u, a.err)) break;
                issue(i);
            }
            // no copy may still be landing in shared memory when the block exits
            for (int j = i > ASTAGES ? i - ASTAGES : 0; j < i; ++j)
                mbar_wait_bounded(smem_addr(&bars[j % ASTAGES]), (uint32_t)((j / ASTAGES) & 1), a.err);
        }
        return;
    }

    // ---------------------------------------------------------- consumers ---
    pdl_wait();
    const int g8 = lane >> 2, t4 = lane & 3;
    const int rA = warp * 16 + g8, rB = rA + 8;  // this lane's two query rows (block-local)
    const int nA = node0 + rA / a.G, nB = node0 + rB / a.G;
    uint32_t qa[AD / 16][4];
    {
        const int hA = hk * a.G + rA % a.G, hB = hk * a.G + rB % a.G;
        const uint32_t *qA = reinterpret_cast<const uint32_t *>(a.q + ((size_t)nA * a.Hq + hA) * AD);
        const uint32_t *qB = reinterpret_cast<const uint32_t *>(a.q + ((size_t)nB * a.Hq + hB) * AD);
        const bool vA = nA < a.M, vB = nB < a.M;
#pragma unroll
        for (int ks = 0; ks < AD / 16; ++ks) {
            const int c = ks * 8 + t4;  // 32-bit column: dims 2c, 2c + 1
            qa[ks][0] = vA ? __ldg(qA + c) : 0u;
            qa[ks][1] = vB ? __ldg(qB + c) : 0u;
            qa[ks][2] = vA ? __ldg(qA + c + 4) : 0u;
            qa[ks][3] = vB ? __ldg(qB + c + 4) : 0u;
        }
    }
    // Ancestor sets of this block's nodes, only where the chunk reaches the
    // tree positions: bit j of word j / 32 = tree node j visible.
    if (k1 > a.L) {
        for (int i = threadIdx.x; i < a.M; i += ACW * 32) s_par[i] = a.parent[i];
        named_barrier(1, ACW * 32);
        if (threadIdx.x < npt) {
            uint32_t m4[4] = {0u, 0u, 0u, 0u};
            const int node = node0 + threadIdx.x;
            if (node < a.M) {
                m4[node >> 5] |= 1u << (node & 31);
                int cur = node;
                for (int step = 0; step < HQ_MAX_M && cur > 0; ++step) {
                    const int p = s_par[cur];
                    if (p < 0 || p >= cur) break;
                    m4[p >> 5] |= 1u << (p & 31);
                    cur = p;
                }
            }
#pragma unroll
            for (int w = 0; w < 4; ++w) s_anc[threadIdx.x * 4 + w] = m4[w];
        }
        named_barrier(1, ACW * 32);
    }
    const uint32_t *ancA = s_anc + (rA / a.G) * 4, *ancB = s_anc + (rB / a.G) * 4;  // this lane's rows' ancestor sets

    float o[AD / 8][4];
#pragma unroll
    for (int j = 0; j < AD / 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[j][e] = 0.0f;
    float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.0f, 0.0f};
    bool ok = true;

    // ldmatrix rows of this lane: K (non-transposed) row (lane >> 4) * 8 + (lane & 7)
    // and chunk half (lane >> 3) & 1; V (transposed) row ((lane >> 3) & 1) * 8 +
    // (lane & 7) and chunk half lane >> 4.  Every row index is r = 8m + (lane & 7).
    const int k_row = (lane >> 4) * 8 + (lane & 7), k_half = (lane >> 3) & 1;
    const int v_row = ((lane >> 3) & 1) * 8 + (lane & 7), v_half = lane >> 4;

    for (int i = 0; i < ntiles; ++i) {
        const int st = i % ASTAGES;
        const uint32_t ph = (uint32_t)((i / ASTAGES) & 1);
        if (ok) ok = mbar_wait_bounded(smem_addr(&bars[st]), ph, a.err);
        const uint32_t kt = smem_addr(ring + (size_t)st * ASTAGE_BYTES);
        const uint32_t vt = kt + ATILE_BYTES;
        const int p0 = k0 + i * AKEYS;

        // S = Q K^T: 16 rows x 64 keys per warp
        float s[AKEYS / 8][4];
#pragma unroll
        for (int j = 0; j < AKEYS / 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[j][e] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < AD / 16; ++ks)
#pragma unroll
            for (int np = 0; np < AKEYS / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kt + (uint32_t)((ks >> 2) * ABOX_BYTES) + swz(np * 16 + k_row, 2 * (ks & 3) + k_half), b0, b1,
                        b2, b3);
                mma16816(s[2 * np], qa[ks], b0, b1);
                mma16816(s[2 * np + 1], qa[ks], b2, b3);
            }

        // mask, scale to base-2 units, running maximum
        const bool full = p0 + AKEYS <= a.L && p0 + AKEYS <= k1;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < AKEYS / 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int pos = p0 + j * 8 + 2 * t4 + (e & 1);
                float x = s[j][e] * a.c_log2;
                if (!full) {
                    bool vis = pos < k1;
                    if (vis && pos >= a.L) {
                        const int tn = pos - a.L;
                        const uint32_t *anc = (e >> 1) ? ancB : ancA;
                        vis = (anc[tn >> 5] >> (tn & 31)) & 1u;
                    }
                    if (!vis) x = -INFINITY;
                }
                s[j][e] = x;
                mx[e >> 1] = fmaxf(mx[e >> 1], x);
            }
        float alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            const float mnew = fmaxf(mrun[h], mx[h]);
            // no visible key yet for this row: nothing to scale, probabilities 0
            alpha[h] = mnew == -INFINITY ? 1.0f : exp2f(mrun[h] - mnew);
            mx[h] = mnew == -INFINITY ? 0.0f : mnew;  // subtrahend for the probabilities
            mrun[h] = mnew;
        }
        float rs[2] = {0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < AKEYS / 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p = exp2f(s[j][e] - mx[e >> 1]);
                s[j][e] = p;
                rs[e >> 1] += p;
            }
#pragma unroll
        for (int h = 0; h < 2; ++h) lrun[h] = lrun[h] * alpha[h] + rs[h];
        // once the maxima settle (alpha == 1 exactly) the rescale is skipped
        if (!__all_sync(0xffffffffu, alpha[0] == 1.0f && alpha[1] == 1.0f)) {
#pragma unroll
            for (int j = 0; j < AD / 8; ++j) {
                o[j][0] *= alpha[0];
                o[j][1] *= alpha[0];
                o[j][2] *= alpha[1];
                o[j][3] *= alpha[1];
            }
        }

        // O += P V: P (fp16) as the A operand, V through transposed ldmatrix
#pragma unroll
        for (int kk = 0; kk < AKEYS / 16; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_half2(s[2 * kk][0], s[2 * kk][1]);
            pa[1] = pack_half2(s[2 * kk][2], s[2 * kk][3]);
            pa[2] = pack_half2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pa[3] = pack_half2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int dp = 0; dp < AD / 16; ++dp) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vt + (uint32_t)((dp >> 2) * ABOX_BYTES) + swz(kk * 16 + v_row, 2 * (dp & 3) + v_half), b0,
                          b1, b2, b3);
                mma16816(o[2 * dp], pa, b0, b1);
                mma16816(o[2 * dp + 1], pa, b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bars[ASTAGES + st]));
    }

    // partial results of this chunk: unnormalized O, running maximum and sum
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        lrun[h] += __shfl_xor_sync(0xffffffffu, lrun[h], 1);
        lrun[h] += __shfl_xor_sync(0xffffffffu, lrun[h], 2);
    }
    const size_t base = ((size_t)split * a.Hkv + hk) * (size_t)a.rows_pad + (size_t)rt * AROWS;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const size_t row = base + (size_t)(h ? rB : rA);
        float *dst = a.ws_o + row * AD;
#pragma unroll
        for (int j = 0; j < AD / 8; ++j)
            *reinterpret_cast<float2 *>(dst + j * 8 + 2 * t4) = make_float2(o[j][2 * h], o[j][2 * h + 1]);
        if (t4 == 0) *reinterpret_cast<float2 *>(a.ws_ml + row * 2) = make_float2(mrun[h], lrun[h]);
    }
}

// One thread block per (node, query head), one thread per dimension.  The
// chunks' maxima and sums are read once into shared memory (one load per
// thread), the weights exp2(m_s - max) computed once, and the partial outputs
// loaded 32 chunks at a time; chunks are added in ascending order.
__global__ void __launch_bounds__(AD) k_tree_attn_merge(const float *__restrict__ ws_o, const float *__restrict__ ws_ml,
                                                        int NS, int Hkv, int Hq, int G, int rows_pad,
                                                        float *__restrict__ out) {
    __shared__ float s_m[AMAX_SPLITS], s_l[AMAX_SPLITS], s_w[AMAX_SPLITS];
    pdl_launch_dependents();
    pdl_wait();
    const int node = blockIdx.x / Hq, h = blockIdx.x % Hq;
    const int hk = h / G, row = node * G + (h % G);
    const int d = threadIdx.x;
    const size_t split_stride = (size_t)Hkv * rows_pad;  // rows between consecutive chunks
    const size_t r0 = (size_t)hk * rows_pad + row;
    if (d < NS) {
        const float2 ml = *reinterpret_cast<const float2 *>(ws_ml + (r0 + d * split_stride) * 2);
        s_m[d] = ml.x;
        s_l[d] = ml.y;
    }
    __syncthreads();
    float mg = -INFINITY;
    for (int sp = 0; sp < NS; ++sp) mg = fmaxf(mg, s_m[sp]);
    if (d < NS) s_w[d] = exp2f(s_m[d] - mg);  // 0 for a chunk in which the row saw no key
    __syncthreads();
    float num = 0.0f, den = 0.0f;
    const float *o = ws_o + r0 * AD + d;
    for (int s0 = 0; s0 < NS; s0 += 32) {
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = s0 + j < NS ? o[(size_t)(s0 + j) * split_stride * AD] : 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (s0 + j < NS) {
                num += s_w[s0 + j] * x[j];
                den += s_w[s0 + j] * s_l[s0 + j];
            }
    }
    out[((size_t)node * Hq + h) * AD + d] = num / den;
}

// One thread block per (key/value head, K or V): the accepted rows are read
// into shared memory first, because a destination row may be another
// accepted node's source row.
__global__ void __launch_bounds__(256) k_tree_commit(__half *k, __half *v, int cap, int L, int M,
                                                     const int32_t *__restrict__ path,
                                                     const int32_t *__restrict__ n_accept) {
    __shared__ __align__(16) uint4 s_rows[HQ_MAX_M][AD * 2 / 16];
    __shared__ int s_src[HQ_MAX_M];
    pdl_launch_dependents();
    pdl_wait();
    const int n = *n_accept;
    if (n <= 0 || n >= M || L + 1 + n > cap) return;
    uint4 *c = reinterpret_cast<uint4 *>((blockIdx.y == 0 ? k : v) + (size_t)blockIdx.x * cap * AD);
    constexpr int RW = AD * 2 / 16;  // uint4 per row
    for (int d = threadIdx.x; d < n; d += blockDim.x) {
        const int p = path[d];
        s_src[d] = (p >= 1 && p < M) ? p : -1;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < n * RW; idx += blockDim.x) {
        const int d = idx / RW, w = idx % RW;
        if (s_src[d] >= 0) s_rows[d][w] = c[(size_t)(L + s_src[d]) * RW + w];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < n * RW; idx += blockDim.x) {
        const int d = idx / RW, w = idx % RW;
        if (s_src[d] >= 0) c[(size_t)(L + 1 + d) * RW + w] = s_rows[d][w];
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Tensor map of a cache [Hkv][cap][AD] fp16 that ends at position `rows`:
// boxes of 64 dimensions x AKEYS positions x 1 head, 128-byte swizzle,
// out-of-range positions filled with zeros.
cudaError_t cache_map(CUtensorMap *m, const void *base, int rows, int cap, int Hkv) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)AD, (cuuint64_t)rows, (cuuint64_t)Hkv};
    const cuuint64_t strides[2] = {(cuuint64_t)AD * 2, (cuuint64_t)cap * AD * 2};
    const cuuint32_t box[3] = {ABOX_DIMS, AKEYS, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaLaunchConfig_t attn_config(dim3 grid, dim3 block, size_t smem, bool pdl, cudaStream_t s,
                               cudaLaunchAttribute (&attr)[1]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

}  // namespace

size_t attn_workspace_bytes(int Hkv) {
    return 16 + (size_t)Hkv * AMAX_ROWS_SPLITS * (size_t)(AD + 2) * 4;
}

cudaError_t launch_tree_attention(const void *q, const void *k, const void *v, int cap, int L, int M, int Hq, int Hkv,
                                  const int32_t *parent, float scale, float *out, void *workspace, bool pdl,
                                  cudaStream_t s) {
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorNoDevice;
    const int G = Hq / Hkv;
    const int row_tiles = (M * G + AROWS - 1) / AROWS;
    const int rows_pad = row_tiles * AROWS;
    const int total = L + M;
    // about two resident blocks per SM, at most AMAX_ROWS_SPLITS / rows_pad chunks
    int ns_cap = AMAX_ROWS_SPLITS / rows_pad;
    if (ns_cap > AMAX_SPLITS) ns_cap = AMAX_SPLITS;
    if (ns_cap < 1) ns_cap = 1;
    int ns = (2 * sms + Hkv * row_tiles - 1) / (Hkv * row_tiles);
    if (ns > ns_cap) ns = ns_cap;
    if (ns < 1) ns = 1;
    int chunk = (total + ns - 1) / ns;
    chunk = (chunk + AKEYS - 1) / AKEYS * AKEYS;
    ns = (total + chunk - 1) / chunk;

    AttnArgs a;
    a.q = static_cast<const __half *>(q);
    a.k = static_cast<const __half *>(k);
    a.v = static_cast<const __half *>(v);
    a.parent = parent;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.err = reinterpret_cast<int *>(ws);
    a.ws_o = reinterpret_cast<float *>(ws + 16);
    a.ws_ml = a.ws_o + (size_t)ns * Hkv * rows_pad * AD;
    a.cap = cap;
    a.L = L;
    a.M = M;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = G;
    a.NS = ns;
    a.chunk = chunk;
    a.rows_pad = rows_pad;
    a.c_log2 = scale * 1.4426950408889634f;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<int> configured[CACHE_DEVICES];
    int done = 0;
    e = cached_per_device(configured, dev, &done, [&](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(k_tree_attn_split, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ASMEM);
    });
    if (e != cudaSuccess) return e;
    CUtensorMap tk, tv;
    e = cache_map(&tk, k, total, cap, Hkv);
    if (e != cudaSuccess) return e;
    e = cache_map(&tv, v, total, cap, Hkv);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg =
        attn_config(dim3((unsigned)ns, (unsigned)Hkv, (unsigned)row_tiles), dim3(ATHREADS), ASMEM, pdl, s, attr);
    e = cudaLaunchKernelEx(&cfg, k_tree_attn_split, a, tk, tv);
    if (e != cudaSuccess) return e;
    cfg = attn_config(dim3((unsigned)(M * Hq)), dim3(AD), 0, true, s, attr);
    return cudaLaunchKernelEx(&cfg, k_tree_attn_merge, (const float *)a.ws_o, (const float *)a.ws_ml, ns, Hkv, Hq, G,
                              rows_pad, out);
}

cudaError_t launch_tree_commit_kv(void *k, void *v, int cap, int L, int M, int Hkv, const int32_t *path,
                                  const int32_t *n_accept, bool pdl, cudaStream_t s) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = attn_config(dim3((unsigned)Hkv, 2), dim3(256), 0, pdl, s, attr);
    return cudaLaunchKernelEx(&cfg, k_tree_commit, static_cast<__half *>(k), static_cast<__half *>(v), cap, L, M,
                              path, n_accept);
}

}  // namespace hq
