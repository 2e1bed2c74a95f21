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
// state is ever written.  Grid (head, 32-row block): every block walks all
// nodes (one warp per node, lanes hold 4 dimensions each, dot products by
// warp shuffles in a fixed order) and then forms its 32 rows of S_c w for all
// nodes (8 threads per row, 16 columns each).  The committed state is read
// before waiting for the previous kernel of the stream: only the commit of
// the previous step writes it.
//
// Commit: one warp per state row applies the root's step and the accepted
// nodes' steps in order (a row evolves independently of the others).
#include <cuda_runtime.h>

#include "hq_internal.cuh"

namespace hq {
namespace {

constexpr int DD = HQ_DELTA_HEAD_DIM;  // state is DD x DD per head
constexpr int DROWS = 32;              // state rows per thread block of the tree pass
constexpr int DTHREADS = 256;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__global__ void __launch_bounds__(DTHREADS) k_delta_tree(const float *__restrict__ state, const float *__restrict__ q,
                                                         const float *__restrict__ k, const float *__restrict__ v,
                                                         const float *__restrict__ alpha,
                                                         const float *__restrict__ beta,
                                                         const int32_t *__restrict__ parent, int M, int H,
                                                         float *__restrict__ out) {
    extern __shared__ __align__(16) float dsm[];
    float *s_w = dsm;                                     // [M][DD] walked vectors
    float *s_vs = s_w + (size_t)M * DD;                   // [M][DROWS] value sums of this block's rows
    int *s_par = reinterpret_cast<int *>(s_vs + (size_t)M * DROWS);
    const int h = blockIdx.x, rb = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this thread's 16 committed-state values: row rb*32 + t/8, columns 16*(t%8) ..
    const int row = rb * DROWS + (threadIdx.x >> 3), seg = threadIdx.x & 7;
    float srow[16];
    {
        const float4 *sp = reinterpret_cast<const float4 *>(state + ((size_t)h * DD + row) * DD + seg * 16);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 t = __ldg(sp + e);
            srow[4 * e] = t.x;
            srow[4 * e + 1] = t.y;
            srow[4 * e + 2] = t.z;
            srow[4 * e + 3] = t.w;
        }
    }
    pdl_launch_dependents();
    pdl_wait();
    for (int i = threadIdx.x; i < M; i += DTHREADS) s_par[i] = parent[i];
    __syncthreads();

    for (int i = warp; i < M; i += DTHREADS / 32) {
        float4 w = __ldg(reinterpret_cast<const float4 *>(q + ((size_t)i * H + h) * DD) + lane);
        float vs = 0.0f;  // sum of c_j v_j for row rb*32 + lane
        int j = i;
        for (int step = 0; step < M; ++step) {
            const size_t b = (size_t)j * H + h;
            const float4 kj = __ldg(reinterpret_cast<const float4 *>(k + b * DD) + lane);
            const float dot = warp_sum(kj.x * w.x + kj.y * w.y + kj.z * w.z + kj.w * w.w);
            const float c = __ldg(beta + b) * dot;
            const float a = __ldg(alpha + b);
            vs += c * __ldg(v + b * DD + rb * DROWS + lane);
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
        s_vs[(size_t)i * DROWS + lane] = vs;
    }
    __syncthreads();

    // o_i[row] = S_c[row] . w_i + vs_i[row]; 8 threads per row, 16 columns each
    for (int i = 0; i < M; ++i) {
        const float4 *wp = reinterpret_cast<const float4 *>(s_w + (size_t)i * DD + seg * 16);
        float acc = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 t = wp[e];
            acc += srow[4 * e] * t.x + srow[4 * e + 1] * t.y + srow[4 * e + 2] * t.z + srow[4 * e + 3] * t.w;
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (seg == 0) out[((size_t)i * H + h) * DD + row] = acc + s_vs[(size_t)i * DROWS + (row - rb * DROWS)];
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

cudaLaunchConfig_t delta_config(dim3 grid, size_t smem, bool pdl, cudaStream_t s, cudaLaunchAttribute (&attr)[1]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(DTHREADS);
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
    const size_t smem = (size_t)M * (DD + DROWS) * 4 + (size_t)M * 4;
    static int configured_for = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_for != dev) {
        e = cudaFuncSetAttribute(k_delta_tree, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)((size_t)HQ_MAX_M * (DD + DROWS) * 4 + (size_t)HQ_MAX_M * 4));
        if (e != cudaSuccess) return e;
        configured_for = dev;
    }
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = delta_config(dim3((unsigned)H, DD / DROWS), smem, pdl, s, attr);
    return cudaLaunchKernelEx(&cfg, k_delta_tree, state, q, k, v, alpha, beta, parent, M, H, out);
}

cudaError_t launch_delta_commit(float *state, const float *k, const float *v, const float *alpha, const float *beta,
                                const int32_t *path, const int32_t *n_accept, int M, int H, bool pdl, cudaStream_t s) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = delta_config(dim3((unsigned)H, DD / (DTHREADS / 32)), 0, pdl, s, attr);
    return cudaLaunchKernelEx(&cfg, k_delta_commit, state, k, v, alpha, beta, path, n_accept, M, H);
}

}  // namespace hq
