// k_pack.cu -- offline rotate + quantize + pack of a layer's weights, and the
// inverse view (canonical codes / scales / zero points) used for checking.
//
// Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
// section "How Uzu optimizes bytes and tokens per pass": the Medium
// checkpoint stores 4-bit asymmetric integers, the Large checkpoint 8-bit
// symmetric integers; the randomized Hadamard transform (32-element blocks)
// is applied before quantization; the quantization group is independent of
// the transform block.
//
// One thread block per blob tile (128 channels x KT features).  Phase 1: each
// warp rotates rows of the tile, one 32-block per warp instruction (lane j
// holds feature j; butterfly stride h = lane exchange xor h), and quantizes
// each (channel, group).  Phase 2: the tile is written in the lane-fragment
// order the GEMM consumes (layout described in hq_internal.cuh).
#include <cuda_runtime.h>

#include "hq_internal.cuh"

namespace hq {
namespace {

__device__ __forceinline__ float round_clamp(float x, float lo, float hi) {
    float r = rintf(x);
    if (r != r) return 0.0f;
    return fminf(fmaxf(r, lo), hi);
}

// Reduce over the lanes of one group: `width` lanes (32 or 16).
__device__ __forceinline__ float warp_min(float v, int width) {
    for (int o = width / 2; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_max(float v, int width) {
    for (int o = width / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int KT>
__global__ void __launch_bounds__(256) k_pack(Geom g, const float *__restrict__ W, const uint32_t *__restrict__ signs,
                                              uint8_t *__restrict__ blob) {
    constexpr int NBLK = KT / 32;
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *codes_s = smem;                                    // [BN][KT]
    float *scales_s = reinterpret_cast<float *>(smem + BN * KT); // [BN][GPT]
    uint8_t *zeros_s = smem + BN * KT + BN * g.GPT * 4;         // [BN][GPT]

    const int kt = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float c = __int_as_float((int)HADAMARD_SCALE_BITS);
    const int G = g.G;
    const bool w4 = g.fmt == HQ_W4_ASYM;

    for (int r = warp; r < BN; r += 8) {
        const int n = b * BN + r;
        float u[NBLK];
#pragma unroll
        for (int blk = 0; blk < NBLK; ++blk) {
            const int k = kt * KT + blk * 32 + lane;
            float v = 0.0f;
            if (n < g.N && k < g.K) {
                v = __ldg(W + (size_t)n * g.K + k);
                const uint32_t sb = (__ldg(signs + (k >> 5)) >> lane) & 1u;
                v = __int_as_float(__float_as_int(v) ^ (int)(sb << 31));
            }
#pragma unroll
            for (int h = 1; h < 32; h <<= 1) {
                const float p = __shfl_xor_sync(0xffffffffu, v, h);
                v = (lane & h) ? __fsub_rn(p, v) : __fadd_rn(v, p);
            }
            u[blk] = __fmul_rn(v, c);
        }
        // per-group parameters, then codes
#pragma unroll
        for (int blk = 0; blk < NBLK; ++blk) {
            const int kl = blk * 32 + lane;  // feature within the tile
            const int gl = kl / G;           // group within the tile
            const int width = G >= 32 ? 32 : 16;
            // reduce over the lane's values of group gl, then across lanes
            float lo = 0.0f, hi = 0.0f, am = 0.0f;
            if (G >= 32) {
                const int b0 = gl * (G / 32), b1 = b0 + G / 32;
#pragma unroll
                for (int bb = 0; bb < NBLK; ++bb) {
                    if (bb >= b0 && bb < b1) {
                        lo = fminf(lo, u[bb]);
                        hi = fmaxf(hi, u[bb]);
                        am = fmaxf(am, fabsf(u[bb]));
                    }
                }
            } else {
                lo = fminf(lo, u[blk]);
                hi = fmaxf(hi, u[blk]);
                am = fmaxf(am, fabsf(u[blk]));
            }
            lo = warp_min(lo, width);
            hi = warp_max(hi, width);
            am = warp_max(am, width);
            uint8_t code;
            float scale;
            uint8_t zero = 0;
            if (w4) {
                scale = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
                if (scale == 0.0f) {
                    code = 0;
                } else {
                    const float z = round_clamp(__fdiv_rn(-lo, scale), 0.0f, 15.0f);
                    float r0 = rintf(__fdiv_rn(u[blk], scale));
                    if (r0 != r0) r0 = 0.0f;
                    code = (uint8_t)round_clamp(__fadd_rn(r0, z), 0.0f, 15.0f);
                    zero = (uint8_t)z;
                }
            } else {
                if (am == 0.0f) {
                    scale = 0.0f;
                    code = 0;
                } else {
                    scale = __fdiv_rn(am, 127.0f);
                    code = (uint8_t)(int8_t)round_clamp(__fdiv_rn(u[blk], scale), -127.0f, 127.0f);
                }
            }
            codes_s[r * KT + kl] = code;
            if ((kl % G) == 0) {
                scales_s[r * g.GPT + gl] = scale;
                zeros_s[r * g.GPT + gl] = zero;
            }
        }
    }
    __syncthreads();

    uint8_t *tile = blob + ((size_t)b * g.KTILES + kt) * (size_t)g.tile_bytes;
    const int nchunks = g.code_bytes / 16;
    for (int q = threadIdx.x; q < nchunks; q += blockDim.x) {
        const int ch = q >> 8, j = (q >> 5) & 7, t = q & 31;
        const int r0 = j * 16 + (t >> 2), r1 = r0 + 8, tig = t & 3;
        uint8_t out[16];
        if (w4) {
            // word (c2, s2): features b = ch*64 + c2*32 + tig*8 + 4*s2 .. b+3;
            // nibbles n0..n7 = (r0,b) (r1,b) (r0,b+2) (r1,b+2) (r0,b+1) (r1,b+1) (r0,b+3) (r1,b+3)
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
                const int b = ch * 64 + (wd >> 1) * 32 + tig * 8 + 4 * (wd & 1);
                const uint8_t *p0 = codes_s + r0 * KT + b, *p1 = codes_s + r1 * KT + b;
                const uint32_t word = (uint32_t)p0[0] | ((uint32_t)p1[0] << 4) | ((uint32_t)p0[2] << 8) |
                                      ((uint32_t)p1[2] << 12) | ((uint32_t)p0[1] << 16) | ((uint32_t)p1[1] << 20) |
                                      ((uint32_t)p0[3] << 24) | ((uint32_t)p1[3] << 28);
                out[4 * wd + 0] = (uint8_t)word;
                out[4 * wd + 1] = (uint8_t)(word >> 8);
                out[4 * wd + 2] = (uint8_t)(word >> 16);
                out[4 * wd + 3] = (uint8_t)(word >> 24);
            }
        } else {
            const int kb = ch * 32 + tig * 8;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                out[e] = codes_s[r0 * KT + kb + e];
                out[4 + e] = codes_s[r1 * KT + kb + e];
                out[8 + e] = codes_s[r0 * KT + kb + 4 + e];
                out[12 + e] = codes_s[r1 * KT + kb + 4 + e];
            }
        }
        uint4 w;
        w.x = out[0] | (out[1] << 8) | (out[2] << 16) | ((uint32_t)out[3] << 24);
        w.y = out[4] | (out[5] << 8) | (out[6] << 16) | ((uint32_t)out[7] << 24);
        w.z = out[8] | (out[9] << 8) | (out[10] << 16) | ((uint32_t)out[11] << 24);
        w.w = out[12] | (out[13] << 8) | (out[14] << 16) | ((uint32_t)out[15] << 24);
        reinterpret_cast<uint4 *>(tile)[q] = w;
    }
    float *sc = reinterpret_cast<float *>(tile + g.code_bytes);
    for (int q = threadIdx.x; q < g.GPT * BN; q += blockDim.x) {
        const int gl = q / BN, rem = q % BN, j = rem / 16, pos = rem % 16;
        const int r = j * 16 + (pos >> 1) + 8 * (pos & 1);
        sc[q] = scales_s[r * g.GPT + gl];
    }
    if (w4) {
        uint8_t *zp = tile + g.code_bytes + g.scale_bytes;
        for (int q = threadIdx.x; q < g.GPT * BN / 2; q += blockDim.x) {
            const int gl = q / (BN / 2), rem = q % (BN / 2), j = rem / 8, rr = rem % 8;
            zp[q] = (uint8_t)(zeros_s[(j * 16 + rr) * g.GPT + gl] | (zeros_s[(j * 16 + rr + 8) * g.GPT + gl] << 4));
        }
    }
}

__global__ void __launch_bounds__(256) k_unpack(Geom g, const uint8_t *__restrict__ blob, uint8_t *__restrict__ codes,
                                                float *__restrict__ scales, uint8_t *__restrict__ zeros) {
    const int kt = blockIdx.x, b = blockIdx.y;
    const uint8_t *tile = blob + ((size_t)b * g.KTILES + kt) * (size_t)g.tile_bytes;
    const bool w4 = g.fmt == HQ_W4_ASYM;
    const int nchunks = g.code_bytes / 16;
    for (int q = threadIdx.x; q < nchunks; q += blockDim.x) {
        const int ch = q >> 8, j = (q >> 5) & 7, t = q & 31;
        const int r0 = j * 16 + (t >> 2), r1 = r0 + 8, tig = t & 3;
        const uint8_t *in = tile + (size_t)q * 16;
        const int n0 = b * BN + r0, n1 = b * BN + r1;
        for (int e = 0; e < 16; ++e) {
            int k;
            if (w4) {
                if (e >= 4) continue;  // one 32-bit word per iteration
                const int wd = e;
                const uint32_t word = (uint32_t)in[4 * wd] | ((uint32_t)in[4 * wd + 1] << 8) |
                                      ((uint32_t)in[4 * wd + 2] << 16) | ((uint32_t)in[4 * wd + 3] << 24);
                const int b = kt * g.KT + ch * 64 + (wd >> 1) * 32 + tig * 8 + 4 * (wd & 1);
                // nibble i -> (row, feature offset)
                const int rowsel[8] = {0, 1, 0, 1, 0, 1, 0, 1};
                const int foff[8] = {0, 0, 2, 2, 1, 1, 3, 3};
                for (int nb = 0; nb < 8; ++nb) {
                    const int kk = b + foff[nb];
                    const int n = rowsel[nb] ? n1 : n0;
                    if (kk < g.K && n < g.N) codes[(size_t)n * g.K + kk] = (uint8_t)((word >> (4 * nb)) & 15u);
                }
            } else {
                const int quarter = e / 4, off = e % 4;
                k = kt * g.KT + ch * 32 + tig * 8 + (quarter >= 2 ? 4 : 0) + off;
                const int n = (quarter & 1) ? n1 : n0;
                if (k < g.K && n < g.N) codes[(size_t)n * g.K + k] = in[e];
            }
        }
    }
    const float *sc = reinterpret_cast<const float *>(tile + g.code_bytes);
    for (int q = threadIdx.x; q < g.GPT * BN; q += blockDim.x) {
        const int gl = q / BN, rem = q % BN, j = rem / 16, pos = rem % 16;
        const int n = b * BN + j * 16 + (pos >> 1) + 8 * (pos & 1);
        const int gg = kt * g.GPT + gl;
        if (n < g.N && gg < g.NGK) scales[(size_t)n * g.NGK + gg] = sc[q];
    }
    if (w4 && zeros) {
        const uint8_t *zp = tile + g.code_bytes + g.scale_bytes;
        for (int q = threadIdx.x; q < g.GPT * BN / 2; q += blockDim.x) {
            const int gl = q / (BN / 2), rem = q % (BN / 2), j = rem / 8, rr = rem % 8;
            const int gg = kt * g.GPT + gl;
            const int n0 = b * BN + j * 16 + rr, n1 = n0 + 8;
            if (gg < g.NGK) {
                if (n0 < g.N) zeros[(size_t)n0 * g.NGK + gg] = zp[q] & 15;
                if (n1 < g.N) zeros[(size_t)n1 * g.NGK + gg] = zp[q] >> 4;
            }
        }
    }
}

template <int KT>
cudaError_t launch_pack_t(const Geom &g, const float *W, const uint32_t *signs, void *blob, cudaStream_t s) {
    const size_t smem = (size_t)BN * KT + (size_t)BN * g.GPT * 5;
    cudaError_t e = cudaFuncSetAttribute(k_pack<KT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_pack<KT><<<dim3(g.KTILES, g.NB), 256, smem, s>>>(g, W, signs, static_cast<uint8_t *>(blob));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack(const Geom &g, const float *W, const uint32_t *signs, void *blob, cudaStream_t s) {
    if (g.KT == 128) return launch_pack_t<128>(g, W, signs, blob, s);
    if (g.KT == 256) return launch_pack_t<256>(g, W, signs, blob, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_unpack(const Geom &g, const void *blob, uint8_t *codes, float *scales, uint8_t *zeros,
                          cudaStream_t s) {
    k_unpack<<<dim3(g.KTILES, g.NB), 256, 0, s>>>(g, static_cast<const uint8_t *>(blob), codes, scales, zeros);
    return cudaGetLastError();
}

}  // namespace hq
