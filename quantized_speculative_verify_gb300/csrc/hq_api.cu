// hq_api.cu -- the C ABI declared in include/hq.h: argument validation (done
// before anything is launched), blob/workspace geometry and kernel dispatch.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "hq_internal.cuh"
#include "k_gemm.cuh"

namespace hq {

int device_sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {

__global__ void k_wait_selftest(int *err, long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    // Nothing arrives on this barrier: the bounded wait must give up.
    mbar_wait_bounded(b, 0u, err, (unsigned long long)limit_ns);
}

}  // namespace

cudaError_t launch_wait_selftest(void *workspace, long long limit_ns, cudaStream_t s) {
    k_wait_selftest<<<1, 1, 0, s>>>(static_cast<int *>(workspace), limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_verify_gemm(const Geom &g, const void *blob, const uint8_t *qop, const float *sx, int M, float *Y,
                               int32_t *partials, void *workspace, uint32_t flags, cudaStream_t s, int wait_extra,
                               long long wait_ns) {
    const bool pdl = (flags & HQ_LAUNCH_PDL) != 0;
    const bool exact = (flags & HQ_LAUNCH_EXACT_ORDER) != 0;
    const bool det = exact || (flags & HQ_LAUNCH_DETERMINISTIC) != 0;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorNoDevice;
    GemmArgs a;
    a.blob = static_cast<const uint8_t *>(blob);
    a.qop = qop;
    a.sx = sx;
    a.Y = Y;
    a.partials = partials;
    a.ws = static_cast<uint8_t *>(workspace);
    a.det = det ? 1 : 0;
    a.nb_align = exact ? 1 : 0;
    a.wait_extra = wait_extra;
    a.wait_ns = wait_ns > 0 ? wait_ns : (long long)WAIT_LIMIT_NS;
    a.M = M;
    a.N = g.N;
    a.K = g.K;
    a.G = g.G;
    a.KT = g.KT;
    a.GPT = g.GPT;
    a.NGK = g.NGK;
    a.NB = g.NB;
    a.KTILES = g.KTILES;
    a.T = g.NB * g.KTILES;
    // One thread block per SM (each owns all of its SM's tensor memory).
    // Small layers get fewer blocks so that every block streams at least
    // MIN_TILES tiles and an n-block is split between few blocks.
    constexpr int MIN_TILES = 4;
    // the register-resident GEMM (up to 32 rows) runs rs_bps(rows) blocks per SM
    const bool rs = act_rs(g.fmt, M);
    int bps = 1;
    if (rs) {
        // rs_bps(rows), fewer where two stages of a unit do not fit in a
        // block's share of the SM's 228 KB (less 1 KB per block)
        const int stage = ((RS_UNIT * g.tile_bytes + 127) / 128 * 128 + RS_UNIT * act_tile_bytes(M, g.G, g.fmt) + 127) /
                          128 * 128;
        bps = rs_bps(act_rows(M));
        while (bps > 1 && 1024 + 2 * stage > 228 * 1024 / bps - 1024) --bps;
    }
    int grid = sms * bps;
    if (exact) {
        // whole n-blocks per block: every output is summed by one block
        if (grid > g.NB) grid = g.NB;
    } else if (grid > a.T / MIN_TILES) {
        grid = a.T / MIN_TILES;
    }
    if (grid < 1) grid = 1;
    if (grid > MAX_CTAS) grid = MAX_CTAS;
    a.grid = grid;
    a.tile_bytes = g.tile_bytes;
    a.code_bytes = g.code_bytes;
    a.scale_bytes = g.scale_bytes;
    const int MT = act_rows(M);
    const bool e4 = act_e4(g.fmt, M, g.G);
    // stage: U weight tiles, then the U activation K tiles (codes, group sums)
    a.act_bytes = act_tile_code_bytes(M, g.G, g.fmt);
    a.s_bytes = act_tile_sum_bytes(M, g.G, g.fmt);
    a.act_tile_bytes = act_tile_bytes(M, g.G, g.fmt);
    auto stage_layout = [&](int U, int header, int budget) {
        a.U = U;
        a.act_off = (U * g.tile_bytes + 127) / 128 * 128;
        a.stage_bytes = (a.act_off + U * a.act_tile_bytes + 127) / 128 * 128;
        // Stage ring: as many units as fit in the block's shared memory beside the barriers.
        int stages = (budget - header) / a.stage_bytes;
        if (stages > MAX_STAGES) stages = MAX_STAGES;
        if (stages < 2) stages = 2;
        a.stages = stages;
        return header + (size_t)stages * a.stage_bytes <= (size_t)budget;
    };
    if (rs) {
        // Register-resident kernel (warp-level fp16 MMAs): up to 32 rows, where
        // the per-group fold of every output is a few register operations.  Units of RS_UNIT tiles.
        a.V = a.na = a.nd = 0;
        // the SM's 228 KB of shared memory, less 1 KB per block, shared by its blocks
        const int budget = 228 * 1024 / bps - 1024;
        if (!stage_layout(RS_UNIT, 1024, budget)) return cudaErrorInvalidConfiguration;
        return g.fmt == HQ_W4_ASYM ? launch_gemm_w4_rs(a, pdl, s) : launch_gemm_w8_rs(a, pdl, s);
    }
    const int dc = e4 ? 2 * MT : MT;             // TMEM columns of one group's accumulator
    const int acols = e4 ? g.KT / 4 : g.KT / 2;  // TMEM columns of one tile's widened weights
    // Pipeline unit: U consecutive tiles, one weight copy and one
    // activation copy (fewer, larger copies stream faster); four tiles up to
    // 32 rows where tensor memory allows, else two, else one.  Tensor memory
    // (512 columns): two A buffers of a unit, then accumulator units of V
    // groups (as many as fit twice, up to a unit's groups), up to MAX_ND.
    int U = MT <= 32 ? 4 : 1, V = 1, nd = 0;
    const int na = 2;
    for (;;) {
        const int rem = TMEM_COLS - na * U * acols;
        nd = 0;
        if (rem > 0) {
            V = U * g.GPT;
            while (V > 1 && 2 * V * dc > rem) V /= 2;
            nd = rem / (V * dc);
        }
        if (nd >= 2 || U == 1) break;
        U /= 2;
    }
    if (nd > MAX_ND) nd = MAX_ND;
    a.V = V;
    a.na = na;
    a.nd = nd;
    if (!stage_layout(U, 2048, GEMM_SMEM_LIMIT) || nd < 2 || na * U * acols + nd * V * dc > TMEM_COLS)
        return cudaErrorInvalidConfiguration;
    return g.fmt == HQ_W4_ASYM ? launch_gemm_w4(a, pdl, s) : launch_gemm_w8(a, pdl, s);
}

}  // namespace hq

using hq::Geom;

namespace {

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

using hq::desc_ok;

Geom geom_of(const hq_layer_desc *d) { return hq::make_geom(d->K, d->N, d->group, d->format); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? HQ_OK : HQ_ERR_CUDA; }

// SplitMix64 (Steele, Lea & Flood 2014): state += golden gamma, then the
// two xor-shift-multiply finalizer rounds.
uint64_t splitmix64_next(uint64_t &state) {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

}  // namespace

extern "C" {

const char *hq_status_string(int status) {
    switch (status) {
        case HQ_OK: return "HQ_OK";
        case HQ_ERR_INVALID_ARG: return "HQ_ERR_INVALID_ARG";
        case HQ_ERR_UNSUPPORTED: return "HQ_ERR_UNSUPPORTED";
        case HQ_ERR_CUDA: return "HQ_ERR_CUDA";
        case HQ_ERR_TIMEOUT: return "HQ_ERR_TIMEOUT";
        default: return "HQ_ERR_UNKNOWN";
    }
}

int32_t hq_version(void) { return (2 << 16) | 0; }  // 2.0: tensor-memory GEMM, one launch up to 128 rows; opaque activation operand with group sums

size_t hq_packed_bytes(const hq_layer_desc *desc) {
    if (!desc_ok(desc)) return 0;
    return hq::blob_bytes(geom_of(desc));
}

size_t hq_workspace_bytes(const hq_layer_desc *desc, int32_t M) {
    if (!desc_ok(desc) || M < 0 || M > HQ_MAX_M) return 0;
    return hq::ws_bytes(geom_of(desc));
}

int hq_make_signs(uint64_t seed, int32_t K, uint32_t *signs_host) {
    if (!signs_host || K <= 0 || K % 32 != 0) return HQ_ERR_INVALID_ARG;
    uint64_t st = seed;
    for (int32_t w = 0; w < K / 32; ++w) {
        uint32_t bits = 0;
        for (int j = 0; j < 32; ++j)
            if (splitmix64_next(st) >> 63) bits |= 1u << j;
        signs_host[w] = bits;
    }
    return HQ_OK;
}

int hq_pack_weights(const hq_layer_desc *desc, const float *W, const uint32_t *signs, void *blob, void *stream) {
    if (!desc_ok(desc) || !W || !signs || !blob) return HQ_ERR_INVALID_ARG;
    if (!aligned(W, 4) || !aligned(signs, 4) || !aligned(blob, 16)) return HQ_ERR_INVALID_ARG;
    const Geom g = geom_of(desc);
    return cuda_status(hq::launch_pack(g, W, g.N, 0, signs, blob, static_cast<cudaStream_t>(stream)));
}

int hq_pack_weights_at(const hq_layer_desc *desc, int32_t n0, int32_t rows, const float *W, const uint32_t *signs,
                       void *blob, void *stream) {
    if (!desc_ok(desc) || !W || !signs || !blob) return HQ_ERR_INVALID_ARG;
    if (n0 < 0 || n0 % hq::BN != 0 || rows <= 0 || (long long)n0 + rows > desc->N) return HQ_ERR_INVALID_ARG;
    if (!aligned(W, 4) || !aligned(signs, 4) || !aligned(blob, 16)) return HQ_ERR_INVALID_ARG;
    const Geom g = geom_of(desc);
    return cuda_status(hq::launch_pack(g, W, rows, n0 / hq::BN, signs, blob, static_cast<cudaStream_t>(stream)));
}

size_t hq_act_operand_bytes(const hq_layer_desc *desc, int32_t M) {
    if (!desc_ok(desc) || M <= 0 || M > HQ_MAX_M) return 0;
    return hq::act_operand_bytes(M, desc->K, desc->group, desc->format);
}

int hq_rotate_quant_act(const hq_layer_desc *desc, const float *X, int32_t M, const uint32_t *signs, int8_t *qx,
                        int32_t *gsum, void *qop, float *sx, uint32_t flags, void *stream) {
    if (!desc_ok(desc)) return HQ_ERR_INVALID_ARG;
    if (M < 0 || M > HQ_MAX_M) return HQ_ERR_INVALID_ARG;
    if ((flags & ~HQ_LAUNCH_PDL) != 0) return HQ_ERR_INVALID_ARG;
    if (M == 0) return HQ_OK;
    if (!X || !signs || !sx || (!qx && !qop && !gsum)) return HQ_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(sx, 4) || !aligned(signs, 4) || (qx && !aligned(qx, 4)) ||
        (gsum && !aligned(gsum, 4)) || (qop && !aligned(qop, 16)))
        return HQ_ERR_INVALID_ARG;
    const int K = desc->K, G = desc->group;
    return cuda_status(hq::launch_rotate_quant_act(X, M, K, G, hq::act_rs(desc->format, M), hq::act_e4(desc->format, M, G), hq::act_sums(desc->format, M), signs, qx, gsum,
                                                   static_cast<uint8_t *>(qop), sx, (flags & HQ_LAUNCH_PDL) != 0,
                                                   static_cast<cudaStream_t>(stream)));
}

int hq_verify_gemm(const hq_layer_desc *desc, const void *blob, const void *qop, const float *sx, int32_t M, float *Y,
                   int32_t *partials, void *workspace, uint32_t flags, void *stream) {
    if (!desc_ok(desc)) return HQ_ERR_INVALID_ARG;
    if (M < 0 || M > HQ_MAX_M) return HQ_ERR_INVALID_ARG;
    if ((flags & ~(HQ_LAUNCH_PDL | HQ_LAUNCH_DETERMINISTIC | HQ_LAUNCH_EXACT_ORDER)) != 0) return HQ_ERR_INVALID_ARG;
    if (M == 0) return HQ_OK;
    if (!blob || !qop || !sx || !Y || !workspace) return HQ_ERR_INVALID_ARG;
    if (!aligned(blob, 16) || !aligned(qop, 16) || !aligned(sx, 4) || !aligned(Y, 4) || !aligned(workspace, 16) ||
        (partials && !aligned(partials, 4)))
        return HQ_ERR_INVALID_ARG;
    const Geom g = geom_of(desc);
    return cuda_status(hq::launch_verify_gemm(g, blob, static_cast<const uint8_t *>(qop), sx, M, Y, partials, workspace,
                                              flags, static_cast<cudaStream_t>(stream)));
}

static size_t q8_operand_offset(const hq_layer_desc *desc, int32_t M) {
    return (hq_workspace_bytes(desc, M) + 255) / 256 * 256;
}

size_t hq_workspace_q8_bytes(const hq_layer_desc *desc, int32_t M) {
    if (!desc_ok(desc) || M < 0 || M > HQ_MAX_M) return 0;
    return q8_operand_offset(desc, M) + (M > 0 ? hq::act_operand_bytes(M, desc->K, desc->group, desc->format) : 0);
}

int hq_verify_gemm_q8(const hq_layer_desc *desc, const void *blob, const int8_t *qx, const float *sx,
                      const int32_t *gsum, int32_t M, float *Y, int32_t *partials, void *workspace, uint32_t flags,
                      void *stream) {
    (void)gsum;  // the group sums are formed from qx itself
    if (!desc_ok(desc)) return HQ_ERR_INVALID_ARG;
    if (M < 0 || M > HQ_MAX_M) return HQ_ERR_INVALID_ARG;
    if ((flags & ~(HQ_LAUNCH_PDL | HQ_LAUNCH_DETERMINISTIC | HQ_LAUNCH_EXACT_ORDER)) != 0) return HQ_ERR_INVALID_ARG;
    if (M == 0) return HQ_OK;
    if (!blob || !qx || !sx || !Y || !workspace) return HQ_ERR_INVALID_ARG;
    if (!aligned(blob, 16) || !aligned(qx, 4) || !aligned(sx, 4) || !aligned(Y, 4) || !aligned(workspace, 16) ||
        (partials && !aligned(partials, 4)))
        return HQ_ERR_INVALID_ARG;
    const int fmt = desc->format, K = desc->K, G = desc->group;
    uint8_t *qop = static_cast<uint8_t *>(workspace) + q8_operand_offset(desc, M);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = hq::launch_codes_to_operand(qx, M, K, G, hq::act_rs(fmt, M), hq::act_e4(fmt, M, G),
                                                hq::act_sums(fmt, M), qop, (flags & HQ_LAUNCH_PDL) != 0, s);
    if (e != cudaSuccess) return HQ_ERR_CUDA;
    // the GEMM follows the conversion on the stream (programmatic launch: its
    // weight stream starts before the operand is complete)
    const Geom g = geom_of(desc);
    return cuda_status(hq::launch_verify_gemm(g, blob, qop, sx, M, Y, partials, workspace, flags | HQ_LAUNCH_PDL, s));
}

int hq_unpack_codes(const hq_layer_desc *desc, const void *blob, uint8_t *codes, float *scales, uint8_t *zeros,
                    void *stream) {
    if (!desc_ok(desc) || !blob || !codes || !scales) return HQ_ERR_INVALID_ARG;
    if (desc->format == HQ_W4_ASYM && !zeros) return HQ_ERR_INVALID_ARG;
    if (!aligned(blob, 16) || !aligned(scales, 4)) return HQ_ERR_INVALID_ARG;
    const Geom g = geom_of(desc);
    return cuda_status(hq::launch_unpack(g, blob, codes, scales, desc->format == HQ_W4_ASYM ? zeros : nullptr,
                                         static_cast<cudaStream_t>(stream)));
}

int hq_workspace_status(void *workspace, void *stream) {
    if (!workspace || !aligned(workspace, 16)) return HQ_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return HQ_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return HQ_ERR_CUDA;
    if (v == 0) return HQ_OK;
    const int zero = 0;
    if (cudaMemcpy(workspace, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return HQ_ERR_CUDA;
    return HQ_ERR_TIMEOUT;
}

int hq_selftest_gemm_wait_timeout(const hq_layer_desc *desc, const void *blob, const void *qop, const float *sx,
                                  int32_t M, float *Y, void *workspace, int64_t limit_ns, void *stream) {
    if (!desc_ok(desc) || M <= 0 || M > HQ_MAX_M) return HQ_ERR_INVALID_ARG;
    if (limit_ns < 1000 || limit_ns > 100000000) return HQ_ERR_INVALID_ARG;
    if (!blob || !qop || !sx || !Y || !workspace) return HQ_ERR_INVALID_ARG;
    if (!aligned(blob, 16) || !aligned(qop, 16) || !aligned(sx, 4) || !aligned(Y, 4) || !aligned(workspace, 16))
        return HQ_ERR_INVALID_ARG;
    const Geom g = geom_of(desc);
    // the deterministic mode waits for one arrival more than there are
    // contributors: every wait between thread blocks runs out after limit_ns
    return cuda_status(hq::launch_verify_gemm(g, blob, static_cast<const uint8_t *>(qop), sx, M, Y, nullptr, workspace,
                                              HQ_LAUNCH_DETERMINISTIC, static_cast<cudaStream_t>(stream), 1,
                                              (long long)limit_ns));
}

int hq_selftest_wait_timeout(void *workspace, int64_t limit_ns, void *stream) {
    if (!workspace || !aligned(workspace, 16)) return HQ_ERR_INVALID_ARG;
    if (limit_ns < 1000 || limit_ns > 100000000) return HQ_ERR_INVALID_ARG;
    return cuda_status(hq::launch_wait_selftest(workspace, limit_ns, static_cast<cudaStream_t>(stream)));
}

size_t hq_tree_attention_workspace_bytes(int32_t Hkv) {
    if (Hkv <= 0 || Hkv > 4096) return 0;
    return hq::attn_workspace_bytes(Hkv);
}

int hq_tree_attention(const void *q, const void *k_cache, const void *v_cache, int32_t cap, int32_t L, int32_t M,
                      int32_t Hq, int32_t Hkv, int32_t D, const int32_t *parent, float scale, float *out,
                      void *workspace, uint32_t flags, void *stream) {
    if (M <= 0 || M > HQ_MAX_M || L < 0 || Hq <= 0 || Hkv <= 0 || Hkv > 4096 || Hq % Hkv != 0) return HQ_ERR_INVALID_ARG;
    if ((long long)L + M > (long long)cap || (long long)cap * Hkv > (1ll << 40)) return HQ_ERR_INVALID_ARG;
    if ((flags & ~HQ_LAUNCH_PDL) != 0 || !(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
        return HQ_ERR_INVALID_ARG;
    if (!q || !k_cache || !v_cache || !parent || !out || !workspace) return HQ_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(parent, 4) ||
        !aligned(out, 16) || !aligned(workspace, 16))
        return HQ_ERR_INVALID_ARG;
    if (D != HQ_ATTN_HEAD_DIM || 64 % (Hq / Hkv) != 0) return HQ_ERR_UNSUPPORTED;
    if ((long long)M * Hq > (1ll << 30)) return HQ_ERR_UNSUPPORTED;
    return cuda_status(hq::launch_tree_attention(q, k_cache, v_cache, cap, L, M, Hq, Hkv, parent, scale, out,
                                                 workspace, (flags & HQ_LAUNCH_PDL) != 0,
                                                 static_cast<cudaStream_t>(stream)));
}

int hq_tree_commit_kv(void *k_cache, void *v_cache, int32_t cap, int32_t L, int32_t M, int32_t Hkv, int32_t D,
                      const int32_t *path, const int32_t *n_accept, uint32_t flags, void *stream) {
    if (M <= 0 || M > HQ_MAX_M || L < 0 || Hkv <= 0 || Hkv > 65535 || (long long)L + M > (long long)cap)
        return HQ_ERR_INVALID_ARG;
    if ((flags & ~HQ_LAUNCH_PDL) != 0) return HQ_ERR_INVALID_ARG;
    if (!k_cache || !v_cache || !path || !n_accept) return HQ_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(path, 4) || !aligned(n_accept, 4))
        return HQ_ERR_INVALID_ARG;
    if (D != HQ_ATTN_HEAD_DIM) return HQ_ERR_UNSUPPORTED;
    return cuda_status(hq::launch_tree_commit_kv(k_cache, v_cache, cap, L, M, Hkv, path, n_accept,
                                                 (flags & HQ_LAUNCH_PDL) != 0, static_cast<cudaStream_t>(stream)));
}

int hq_delta_tree(const float *state, const float *q, const float *k, const float *v, const float *alpha,
                  const float *beta, const int32_t *parent, int32_t M, int32_t H, int32_t D, float *out,
                  uint32_t flags, void *stream) {
    if (M <= 0 || M > HQ_MAX_M || H <= 0 || H > 65535) return HQ_ERR_INVALID_ARG;
    if ((flags & ~HQ_LAUNCH_PDL) != 0) return HQ_ERR_INVALID_ARG;
    if (!state || !q || !k || !v || !alpha || !beta || !parent || !out) return HQ_ERR_INVALID_ARG;
    if (!aligned(state, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(alpha, 4) ||
        !aligned(beta, 4) || !aligned(parent, 4) || !aligned(out, 16))
        return HQ_ERR_INVALID_ARG;
    if (D != HQ_DELTA_HEAD_DIM) return HQ_ERR_UNSUPPORTED;
    return cuda_status(hq::launch_delta_tree(state, q, k, v, alpha, beta, parent, M, H, out,
                                             (flags & HQ_LAUNCH_PDL) != 0, static_cast<cudaStream_t>(stream)));
}

int hq_delta_commit(float *state, const float *k, const float *v, const float *alpha, const float *beta,
                    const int32_t *path, const int32_t *n_accept, int32_t M, int32_t H, int32_t D, uint32_t flags,
                    void *stream) {
    if (M <= 0 || M > HQ_MAX_M || H <= 0 || H > 65535) return HQ_ERR_INVALID_ARG;
    if ((flags & ~HQ_LAUNCH_PDL) != 0) return HQ_ERR_INVALID_ARG;
    if (!state || !k || !v || !alpha || !beta || !path || !n_accept) return HQ_ERR_INVALID_ARG;
    if (!aligned(state, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(alpha, 4) || !aligned(beta, 4) ||
        !aligned(path, 4) || !aligned(n_accept, 4))
        return HQ_ERR_INVALID_ARG;
    if (D != HQ_DELTA_HEAD_DIM) return HQ_ERR_UNSUPPORTED;
    return cuda_status(hq::launch_delta_commit(state, k, v, alpha, beta, path, n_accept, M, H,
                                               (flags & HQ_LAUNCH_PDL) != 0, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

extern "C" {

size_t hq_tree_accept_workspace_bytes(int32_t M, int32_t V) {
    if (M <= 0 || M > HQ_MAX_M || V <= 0) return 0;
    return ((size_t)M * (size_t)hq::accept_chunks(V) * 8 + 15) / 16 * 16;
}

int hq_tree_accept(const float *logits, int32_t M, int32_t V, const int32_t *parent, const int32_t *tokens,
                   int32_t *greedy, int32_t *path, int32_t *n_accept, int32_t *bonus, void *workspace, uint32_t flags,
                   void *stream) {
    if (M <= 0 || M > HQ_MAX_M || V <= 0) return HQ_ERR_INVALID_ARG;
    if ((flags & ~HQ_LAUNCH_PDL) != 0) return HQ_ERR_INVALID_ARG;
    if (!logits || !parent || !tokens || !greedy || !path || !n_accept || !bonus || !workspace)
        return HQ_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(parent, 4) || !aligned(tokens, 4) || !aligned(greedy, 4) ||
        !aligned(path, 4) || !aligned(n_accept, 4) || !aligned(bonus, 4) || !aligned(workspace, 16))
        return HQ_ERR_INVALID_ARG;
    return cuda_status(hq::launch_tree_accept(logits, M, V, parent, tokens, greedy, path, n_accept, bonus, workspace,
                                              (flags & HQ_LAUNCH_PDL) != 0, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
