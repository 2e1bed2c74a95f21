// k_accept.cu -- the main model's greedy token per row of its logits, and the
// acceptance of a draft tree.
//
// Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
// sections "Producing several tokens from one model pass" (the main model
// checks the drafted positions together, accepts the valid prefix and adds
// its own token at the first position it does not confirm) and "Verifying a
// draft tree without restoring model state" (on a tree, the longest valid
// path is accepted).  Node 0 is the root (the last committed token); node
// i > 0 has parent p[i] < i and drafted token t[i]; row i of the logits is the
// main model's output after node i, g[i] its greedy token (lowest index among
// equal maxima, a NaN larger than every number).  Node i is valid when its
// parent is and t[i] == g[p[i]]; the deepest valid node is accepted (lowest
// index among equally deep ones) and g at that node is the bonus token.
//
// Kernel 1: C thread blocks per row, each reduces a contiguous chunk of the
// row to one 64-bit key (value mapped to a monotone unsigned integer in the
// high word, the inverted index in the low word: the maximum key is the
// maximum value at the lowest index).  Kernel 2: one block reduces the C keys
// of every row in a fixed order and walks the tree (M <= 128 nodes).
#include <cuda_runtime.h>

#include "hq_internal.cuh"

namespace hq {
namespace {

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    uint32_t u = __float_as_uint(v);
    if (v != v) u = 0x7FC00000u;  // every NaN ranks above +inf
    if (v == 0.0f) u = 0u;        // -0 and +0 are equal
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ unsigned long long max_u64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

constexpr int ARGMAX_THREADS = 256;

__global__ void __launch_bounds__(ARGMAX_THREADS) k_argmax_partial(const float *__restrict__ logits, int V,
                                                                   int chunk, int C,
                                                                   unsigned long long *__restrict__ partial) {
    __shared__ unsigned long long s_red[ARGMAX_THREADS / 32];
    pdl_launch_dependents();
    pdl_wait();
    const int row = blockIdx.x / C, part = blockIdx.x % C;
    const int lo = part * chunk;
    const int hi = lo + chunk < V ? lo + chunk : V;
    const float *r = logits + (size_t)row * (size_t)V;
    unsigned long long best = 0ull;  // below every real key
    // float4 loads where the row and the chunk allow it, scalar elsewhere
    const bool vec = ((reinterpret_cast<uintptr_t>(r) & 15u) == 0) && (lo % 4 == 0);
    int k = lo;
    if (vec) {
        const int hi4 = lo + ((hi - lo) / 4) * 4;
        for (int j = lo / 4 + threadIdx.x; j < hi4 / 4; j += ARGMAX_THREADS) {
            const float4 q = __ldg(reinterpret_cast<const float4 *>(r) + j);
            best = max_u64(best, argmax_key(q.x, 4 * j));
            best = max_u64(best, argmax_key(q.y, 4 * j + 1));
            best = max_u64(best, argmax_key(q.z, 4 * j + 2));
            best = max_u64(best, argmax_key(q.w, 4 * j + 3));
        }
        k = hi4;
    }
    for (int j = k + threadIdx.x; j < hi; j += ARGMAX_THREADS) best = max_u64(best, argmax_key(__ldg(r + j), j));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max_u64(best, __shfl_xor_sync(0xffffffffu, best, o));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long b = s_red[0];
        for (int w = 1; w < ARGMAX_THREADS / 32; ++w) b = max_u64(b, s_red[w]);
        partial[blockIdx.x] = b;
    }
}

__global__ void __launch_bounds__(128) k_tree_accept(const unsigned long long *__restrict__ partial, int M, int C,
                                                     const int32_t *__restrict__ parent,
                                                     const int32_t *__restrict__ tokens, int32_t *__restrict__ g_out,
                                                     int32_t *__restrict__ path, int32_t *__restrict__ n_accept,
                                                     int32_t *__restrict__ bonus) {
    __shared__ int32_t s_g[HQ_MAX_M];
    __shared__ int32_t s_valid[HQ_MAX_M];
    __shared__ int32_t s_depth[HQ_MAX_M];
    pdl_launch_dependents();
    pdl_wait();
    for (int i = threadIdx.x; i < M; i += blockDim.x) {
        unsigned long long b = partial[(size_t)i * C];
        for (int c = 1; c < C; ++c) b = max_u64(b, partial[(size_t)i * C + c]);
        const int32_t gi = (int32_t)(0xFFFFFFFFu - (uint32_t)(b & 0xFFFFFFFFull));
        s_g[i] = gi;
        g_out[i] = gi;
        path[i] = -1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // parents precede children, so one pass in index order sees every parent first
        bool tree = true;
        s_valid[0] = 1;
        s_depth[0] = 0;
        for (int i = 1; i < M; ++i) {
            const int p = parent[i];
            if (p < 0 || p >= i) {
                tree = false;
                break;
            }
            s_valid[i] = s_valid[p] && tokens[i] == s_g[p];
            s_depth[i] = s_depth[p] + 1;
        }
        if (!tree) {
            *n_accept = -1;
            *bonus = -1;
        } else {
            int best = 0;
            for (int i = 1; i < M; ++i)
                if (s_valid[i] && s_depth[i] > s_depth[best]) best = i;
            *n_accept = s_depth[best];
            *bonus = s_g[best];
            for (int i = best, d = s_depth[best]; d > 0; i = parent[i], --d) path[d - 1] = i;
        }
    }
}

cudaError_t launch_pdl(const cudaLaunchConfig_t &base, bool pdl, cudaLaunchConfig_t &cfg,
                       cudaLaunchAttribute (&attr)[1]) {
    cfg = base;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaSuccess;
}

}  // namespace

int accept_chunks(int V) { return (V + ACCEPT_CHUNK - 1) / ACCEPT_CHUNK; }

cudaError_t launch_tree_accept(const float *logits, int M, int V, const int32_t *parent, const int32_t *tokens,
                               int32_t *g_out, int32_t *path, int32_t *n_accept, int32_t *bonus, void *workspace,
                               bool pdl, cudaStream_t s) {
    const int C = accept_chunks(V);
    unsigned long long *partial = static_cast<unsigned long long *>(workspace);
    cudaLaunchConfig_t base = {}, cfg;
    cudaLaunchAttribute attr[1];
    base.stream = s;
    base.gridDim = dim3((unsigned)(M * C));
    base.blockDim = dim3(ARGMAX_THREADS);
    launch_pdl(base, pdl, cfg, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_argmax_partial, logits, V, (int)ACCEPT_CHUNK, C, partial);
    if (e != cudaSuccess) return e;
    base.gridDim = dim3(1);
    base.blockDim = dim3(128);
    launch_pdl(base, pdl, cfg, attr);
    return cudaLaunchKernelEx(&cfg, k_tree_accept, (const unsigned long long *)partial, M, C, parent, tokens, g_out,
                              path, n_accept, bonus);
}

}  // namespace hq
