// k_delta.cu -- rollback-free DeltaNet tree pass and the accepted-path state
// commit.
//
// Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
// section "Verifying a draft tree without restoring model state": a Gated
// DeltaNet layer keeps a fixed-size state that every accepted token changes;
// the verify pass computes the outputs of every branch of the draft tree in
// one pass without changing the live state, and the state is then updated
// only along the accepted path.  The page gives no equations; the recurrence
// is the published gated delta rule (Yang, Kautz and Hatamizadeh, "Gated
// Delta Networks", ICLR 2025), per head with a D x D state S:
//     S_i = alpha_i S_p (I - beta_i k_i k_i^T) + beta_i v_i k_i^T,  o_i = S_i q_i
// where p is node i's parent (the committed state for the root, or where the
// parent link is not a tree link).
//
// Tree pass without a recurrence over states: for any vector q,
//     S_i q = S_p w' + c v_i,  c = beta_i (k_i . q),  w' = alpha_i (q - c k_i),
// so walking from node i up to the root with a D-vector w (starting at q_i)
// gives o_i = S_committed w + sum of c_j v_j over the path.  Each node costs
// O(depth * D) vector work plus one product with the committed state, and no
// state is ever written.  Grid (head, 16-row block), 16 warps: every block
// stages its committed-state rows (padded rows: conflict-free reads), the
// nodes' q, k, gates and its value rows in shared memory (one round of
// loads), walks the nodes (one warp per node, lanes hold 4 dimensions each,
// dot products by warp shuffles in a fixed order), then, in the warp that
// walked a node, forms its 16 rows of S_c w (a thread per row and half row,
// four accumulators).  The committed state is read before waiting for the
// previous kernel of the stream: only the commit of the previous step
// writes it.
//
// Commit: one warp per state row applies the root's step and the accepted
// nodes' steps in order (a row evolves independently of the others).
#include <cuda_runtime.h>

#include "hq_internal.cuh"

namespace hq {
namespace {

constexpr int DD = HQ_DELTA_HEAD_DIM;  // state is DD x DD per head
constexpr int DROWS = 16;              // state rows per thread block of the tree pass
constexpr int DTREE_THREADS = 512;     // 16 warps: one node per warp per round
constexpr int DSTRIDE = DD + 4;        // padded shared-memory row of the state block (floats)
constexpr int DTHREADS = 256;          // commit

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__global__ void __launch_bounds__(DTREE_THREADS, 2) k_delta_tree(const float *__restrict__ state,
                                                              const float *__restrict__ q,
                                                              const float *__restrict__ k,
                                                              const float *__restrict__ v,
                                                              const float *__restrict__ alpha,
                                                              const float *__restrict__ beta,
                                                              const int32_t *__restrict__ parent, int M, int H,
                                                              float *__restrict__ out) {
    extern __shared__ __align__(16) float dsm[];
    float *s_S = dsm;                                 // [DROWS][DSTRIDE] this block's committed-state rows
    float *s_w = s_S + DROWS * DSTRIDE;               // [M][DD] walked vectors (start: q)
    float *s_k = s_w + (size_t)M * DD;                // [M][DD] keys of this head
    float *s_v = s_k + (size_t)M * DD;                // [M][DROWS] this block's value rows
    float *s_vs = s_v + (size_t)M * DROWS;            // [M][DROWS] value sums of this block's rows
    float *s_a = s_vs + (size_t)M * DROWS;            // [M] gates
    float *s_b = s_a + M;                             // [M] write strengths
    int *s_par = reinterpret_cast<int *>(s_b + M);    // [M]
    const int h = blockIdx.x, rb = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int NW = DTREE_THREADS / 32;

    // the committed-state rows of this block (not written by the previous kernel)
    for (int x = threadIdx.x; x < DROWS * (DD / 4); x += DTREE_THREADS) {
        const int r = x / (DD / 4), c4 = x % (DD / 4);
        reinterpret_cast<float4 *>(s_S + r * DSTRIDE)[c4] =
            __ldg(reinterpret_cast<const float4 *>(state + ((size_t)h * DD + rb * DROWS + r) * DD) + c4);
    }
    pdl_launch_dependents();
    pdl_wait();
    // every node's q, k, gates and this block's value rows, in one round of loads
    for (int x = threadIdx.x; x < M * (DD / 4); x += DTREE_THREADS) {
        const int i = x / (DD / 4), c4 = x % (DD / 4);
        const size_t b = ((size_t)i * H + h) * DD;
        reinterpret_cast<float4 *>(s_w)[x] = __ldg(reinterpret_cast<const float4 *>(q + b) + c4);
        reinterpret_cast<float4 *>(s_k)[x] = __ldg(reinterpret_cast<const float4 *>(k + b) + c4);
    }
    for (int x = threadIdx.x; x < M * DROWS; x += DTREE_THREADS) {
        const int i = x / DROWS, r = x % DROWS;
        s_v[x] = __ldg(v + ((size_t)i * H + h) * DD + rb * DROWS + r);
    }
    for (int i = threadIdx.x; i < M; i += DTREE_THREADS) {
        s_a[i] = __ldg(alpha + (size_t)i * H + h);
        s_b[i] = __ldg(beta + (size_t)i * H + h);
        s_par[i] = parent[i];
    }
    __syncthreads();

    // one warp per node: walk from the node up to the root (or to a link
    // that is not a tree link), lanes holding 4 dimensions each
    for (int i = warp; i < M; i += NW) {
        float4 w = reinterpret_cast<const float4 *>(s_w + (size_t)i * DD)[lane];
        float vs = 0.0f;  // sum of c_j v_j for row rb*DROWS + lane (lanes < DROWS)
        int j = i;
        for (int step = 0; step < M; ++step) {
            const float4 kj = reinterpret_cast<const float4 *>(s_k + (size_t)j * DD)[lane];
            const float dot = warp_sum(kj.x * w.x + kj.y * w.y + kj.z * w.z + kj.w * w.w);
            const float c = s_b[j] * dot;
            const float a = s_a[j];
            if (lane < DROWS) vs += c * s_v[(size_t)j * DROWS + lane];
            w.x = a * (w.x - c * kj.x);
            w.y = a * (w.y - c * kj.y);
            w.z = a * (w.z - c * kj.z);
            w.w = a * (w.w - c * kj.w);
            if (j == 0) break;
            const int p = s_par[j];
            if (p < 0 || p >= j) break;  // the chain starts at the committed state
            j = p;
        }
        reinterpret_cast<float4 *>(s_w + (size_t)i * DD)[lane] = w;
        if (lane < DROWS) s_vs[(size_t)i * DROWS + lane] = vs;
    }
    // the products below take node i in the warp that walked it (the same
    // node-to-warp assignment): no block barrier, warps do not wait for the
    // deepest walk
    __syncwarp();

    // o_i[row] = S_c[row] . w_i + vs_i[row]: thread (node slot, half, row)
    // sums 64 columns with four accumulators (a quarter warp reads eight
    // different padded rows: no bank conflict), one shuffle joins the halves
    const int r = threadIdx.x & (DROWS - 1), half = (threadIdx.x >> 4) & 1, slot = warp;
    const float4 *srow = reinterpret_cast<const float4 *>(s_S + r * DSTRIDE + half * (DD / 2));
    for (int i = slot; i < M; i += NW) {
        const float4 *wp = reinterpret_cast<const float4 *>(s_w + (size_t)i * DD + half * (DD / 2));
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int e = 0; e < DD / 8; ++e) {
            const float4 sv = srow[e], wv = wp[e];
            acc[e & 3] += sv.x * wv.x + sv.y * wv.y + sv.z * wv.z + sv.w * wv.w;
        }
        float t = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        t += __shfl_xor_sync(0xffffffffu, t, 16);
        if (half == 0) out[((size_t)i * H + h) * DD + rb * DROWS + r] = t + s_vs[(size_t)i * DROWS + r];
    }
}

// One warp per state row (8 rows per block): the root's step, then the
// accepted nodes' steps; path entries outside [1, M) are skipped; nothing
// changes when *n_accept < 0.
__global__ void __launch_bounds__(DTHREADS) k_delta_commit(float *__restrict__ state, const float *__restrict__ k,
                                                           const float *__restrict__ v,
                                                           const float *__restrict__ alpha,
                                                           const float *__restrict__ beta,
                                                           const int32_t *__restrict__ path,
                                                           const int32_t *__restrict__ n_accept, int M, int H) {
    pdl_launch_dependents();
    pdl_wait();
    const int n = *n_accept;
    if (n < 0 || n >= M) return;
    const int h = blockIdx.x, row = blockIdx.y * (DTHREADS / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    float4 *sp = reinterpret_cast<float4 *>(state + ((size_t)h * DD + row) * DD) + lane;
    float4 s = *sp;
    for (int a = -1; a < n; ++a) {
        const int j = a < 0 ? 0 : path[a];
        if (a >= 0 && (j < 1 || j >= M)) continue;
        const size_t b = (size_t)j * H + h;
        const float4 kj = __ldg(reinterpret_cast<const float4 *>(k + b * DD) + lane);
        const float u = warp_sum(s.x * kj.x + s.y * kj.y + s.z * kj.z + s.w * kj.w);  // (S k)_row
        const float al = __ldg(alpha + b), be = __ldg(beta + b);
        const float bu = be * u, bv = be * __ldg(v + b * DD + row);
        s.x = al * (s.x - bu * kj.x) + bv * kj.x;
        s.y = al * (s.y - bu * kj.y) + bv * kj.y;
        s.z = al * (s.z - bu * kj.z) + bv * kj.z;
        s.w = al * (s.w - bu * kj.w) + bv * kj.w;
    }
    *sp = s;
}

cudaLaunchConfig_t delta_config(dim3 grid, dim3 block, size_t smem, bool pdl, cudaStream_t s,
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

cudaError_t launch_delta_tree(const float *state, const float *q, const float *k, const float *v, const float *alpha,
                              const float *beta, const int32_t *parent, int M, int H, float *out, bool pdl,
                              cudaStream_t s) {
    const size_t smem = (size_t)DROWS * DSTRIDE * 4 + (size_t)M * (2 * DD + 2 * DROWS + 3) * 4;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<int> configured[CACHE_DEVICES];
    int done = 0;
    e = cached_per_device(configured, dev, &done, [&](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(k_delta_tree, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)((size_t)DROWS * DSTRIDE * 4 + (size_t)HQ_MAX_M * (2 * DD + 2 * DROWS + 3) * 4));
    });
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = delta_config(dim3((unsigned)H, DD / DROWS), dim3(DTREE_THREADS), smem, pdl, s, attr);
    return cudaLaunchKernelEx(&cfg, k_delta_tree, state, q, k, v, alpha, beta, parent, M, H, out);
}

cudaError_t launch_delta_commit(float *state, const float *k, const float *v, const float *alpha, const float *beta,
                                const int32_t *path, const int32_t *n_accept, int M, int H, bool pdl, cudaStream_t s) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = delta_config(dim3((unsigned)H, DD / (DTHREADS / 32)), dim3(DTHREADS), 0, pdl, s, attr);
    return cudaLaunchKernelEx(&cfg, k_delta_commit, state, k, v, alpha, beta, path, n_accept, M, H);
}

}  // namespace hq
