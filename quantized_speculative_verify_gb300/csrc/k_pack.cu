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
// each (channel, group).  Phase 2: the tile is written in the channel-per-
// thread order the GEMM consumes (layout described in hq_internal.cuh).
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
// Packs `rows` rows of W into the n-blocks nb0, nb0 + 1, ... of the blob of
// layer g (rows past `rows` are zero).
__global__ void __launch_bounds__(256) k_pack(Geom g, const float *__restrict__ W, int rows, int nb0,
                                              const uint32_t *__restrict__ signs, uint8_t *__restrict__ blob) {
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
            if (n < rows && k < g.K) {
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

    uint8_t *tile = blob + ((size_t)(nb0 + b) * g.KTILES + kt) * (size_t)g.tile_bytes;
    const int nchunks = g.code_bytes / 16;
    for (int q = threadIdx.x; q < nchunks; q += blockDim.x) {
        const int cp = q / BN, r = q % BN;  // 16-byte run cp of channel r
        const uint8_t *src = codes_s + r * KT;
        uint32_t wv[4];
        if (w4) {
            // word t: nibble i = feature 2 t + 8 i, nibble i + 4 = feature 2 t + 8 i + 1 (i = 0..3)
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const uint8_t *p8 = src + cp * 32 + 2 * t;
                uint32_t word = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    word |= ((uint32_t)(p8[8 * i] & 15u) << (4 * i)) | ((uint32_t)(p8[8 * i + 1] & 15u) << (4 * i + 16));
                wv[t] = word;
            }
        } else {
            // word t: features 2 t, 2 t + 1, 2 t + 8, 2 t + 9 of the run 16 cp ..
            const uint8_t *p8 = src + cp * 16;
#pragma unroll
            for (int t = 0; t < 4; ++t)
                wv[t] = (uint32_t)p8[2 * t] | ((uint32_t)p8[2 * t + 1] << 8) | ((uint32_t)p8[2 * t + 8] << 16) |
                        ((uint32_t)p8[2 * t + 9] << 24);
        }
        reinterpret_cast<uint4 *>(tile)[q] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
    float *sc = reinterpret_cast<float *>(tile + g.code_bytes);
    for (int q = threadIdx.x; q < g.GPT * BN; q += blockDim.x) sc[q] = scales_s[q];  // [channel][group]
    if (w4) {
        uint8_t *zp = tile + g.code_bytes + g.scale_bytes;
        // nibble i = (channel i / GPT, group i % GPT), low nibble first
        for (int q = threadIdx.x; q < g.GPT * BN / 2; q += blockDim.x) zp[q] = (uint8_t)(zeros_s[2 * q] | (zeros_s[2 * q + 1] << 4));
    }
}

__global__ void __launch_bounds__(256) k_unpack(Geom g, const uint8_t *__restrict__ blob, uint8_t *__restrict__ codes,
                                                float *__restrict__ scales, uint8_t *__restrict__ zeros) {
    const int kt = blockIdx.x, b = blockIdx.y;
    const uint8_t *tile = blob + ((size_t)b * g.KTILES + kt) * (size_t)g.tile_bytes;
    const bool w4 = g.fmt == HQ_W4_ASYM;
    const int nchunks = g.code_bytes / 16;
    for (int q = threadIdx.x; q < nchunks; q += blockDim.x) {
        const int cp = q / BN, r = q % BN;
        const int n = b * BN + r;
        const uint4 u = reinterpret_cast<const uint4 *>(tile)[q];
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
        if (n >= g.N) continue;
        for (int j = 0; j < 4; ++j) {
            if (w4) {
                for (int i = 0; i < 8; ++i) {  // nibble i of word j: feature 2 j + 8 (i % 4) + i / 4
                    const int k = kt * g.KT + cp * 32 + 2 * j + 8 * (i & 3) + (i >> 2);
                    if (k < g.K) codes[(size_t)n * g.K + k] = (uint8_t)((wv[j] >> (4 * i)) & 15u);
                }
            } else {
                for (int e = 0; e < 4; ++e) {  // byte e of word j: feature 2 j + (e & 1) + 8 (e >> 1)
                    const int k = kt * g.KT + cp * 16 + 2 * j + (e & 1) + 8 * (e >> 1);
                    if (k < g.K) codes[(size_t)n * g.K + k] = (uint8_t)(wv[j] >> (8 * e));
                }
            }
        }
    }
    const float *sc = reinterpret_cast<const float *>(tile + g.code_bytes);
    for (int q = threadIdx.x; q < g.GPT * BN; q += blockDim.x) {
        const int n = b * BN + q / g.GPT, gg = kt * g.GPT + q % g.GPT;
        if (n < g.N && gg < g.NGK) scales[(size_t)n * g.NGK + gg] = sc[q];
    }
    if (w4 && zeros) {
        const uint8_t *zp = tile + g.code_bytes + g.scale_bytes;
        for (int i = threadIdx.x; i < g.GPT * BN; i += blockDim.x) {
            const int n = b * BN + i / g.GPT, gg = kt * g.GPT + i % g.GPT;
            if (n < g.N && gg < g.NGK) zeros[(size_t)n * g.NGK + gg] = (zp[i >> 1] >> (4 * (i & 1))) & 15;
        }
    }
}

template <int KT>
cudaError_t launch_pack_t(const Geom &g, const float *W, int rows, int nb0, const uint32_t *signs, void *blob,
                          cudaStream_t s) {
    const size_t smem = (size_t)BN * KT + (size_t)BN * g.GPT * 5;
    cudaError_t e = cudaFuncSetAttribute(k_pack<KT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_pack<KT><<<dim3(g.KTILES, (rows + BN - 1) / BN), 256, smem, s>>>(g, W, rows, nb0, signs,
                                                                       static_cast<uint8_t *>(blob));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack(const Geom &g, const float *W, int rows, int nb0, const uint32_t *signs, void *blob,
                        cudaStream_t s) {
    if (g.KT == 128) return launch_pack_t<128>(g, W, rows, nb0, signs, blob, s);
    if (g.KT == 256) return launch_pack_t<256>(g, W, rows, nb0, signs, blob, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_unpack(const Geom &g, const void *blob, uint8_t *codes, float *scales, uint8_t *zeros,
                          cudaStream_t s) {
    k_unpack<<<dim3(g.KTILES, g.NB), 256, 0, s>>>(g, static_cast<const uint8_t *>(blob), codes, scales, zeros);
    return cudaGetLastError();
}

}  // namespace hq
