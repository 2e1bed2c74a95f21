// k_act.cu -- rotate + quantize the activations of the verify batch.
//
// Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
// section "How Uzu optimizes bytes and tokens per pass": activations are
// quantized to 8 bits on the fly, after the block-diagonal randomized
// Hadamard transform (32-element blocks, random sign flips before the
// mixing, one overall scale) that the weights went through offline.
//
// One thread block per row.  Thread i holds float4s i, i + T, i + 2T, ...
// of the row, so 8 consecutive lanes hold one 32-element block: butterfly
// strides 1 and 2 are inside a lane's float4, strides 4, 8 and 16 are lane
// exchanges (xor 1, 2, 4).  Every add, subtract and multiply is a separate
// IEEE-rounded fp32 operation in the order 1, 2, 4, 8, 16, so the rotated
// values are bit-identical to a scalar implementation of the same order.
// The codes are written as int8 and/or as the GEMM's operand: fp16 (exact
// for |q| <= 127) or two e4m3 digits (q = 16 h + l), in 128-feature blocks
// laid out as the MMA's B operand, plus, where the GEMM applies a zero point
// through them, the per-group sums of the codes (the Medium identity's
// correction term).
// The grid has one block per operand row: rows past M (padding up to the
// MMA's N) only write zeros.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "hq_internal.cuh"

namespace hq {
namespace {

__device__ __forceinline__ float flip(float x, uint32_t bit) {
    return __int_as_float(__float_as_int(x) ^ (int)(bit << 31));
}

// Stage h in {4, 8, 16}: lane partner = lane ^ (h / 4).  The lane holding the
// lower index keeps a + b, the other keeps a - b (a = lower, b = upper).
__device__ __forceinline__ float bfly_x(float v, int lane_bit, bool upper) {
    float p = __shfl_xor_sync(0xffffffffu, v, lane_bit);
    return upper ? __fsub_rn(p, v) : __fadd_rn(v, p);
}

// e4m3 byte of an integer v in [-8, 8] (exact): 1..8 are 2^e * (1 + m/8).
__device__ __forceinline__ uint32_t e4m3_small(int v) {
    const uint32_t a = (uint32_t)(v < 0 ? -v : v);
    if (a == 0) return 0u;
    const uint32_t e = 31u - __clz(a);          // 0..3
    const uint32_t m = ((a << 3) >> e) & 7u;    // mantissa bits
    return ((e + 7u) << 3) | m | (v < 0 ? 0x80u : 0u);
}
// Low and high e4m3 digits of four codes, one byte each.
__device__ __forceinline__ void digits4(int q0, int q1, int q2, int q3, uint32_t &lo, uint32_t &hi) {
    const int q[4] = {q0, q1, q2, q3};
    lo = hi = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int l = ((q[i] + 8) & 15) - 8;
        const int h = (q[i] - l) / 16;
        lo |= e4m3_small(l) << (8 * i);
        hi |= e4m3_small(h) << (8 * i);
    }
}

template <int V, int T>
__global__ void __launch_bounds__(T) k_rotate_quant_act(const float *__restrict__ X, int M, int K, int G, int rs, int e4, int sums,
                                                        const uint32_t *__restrict__ signs, int8_t *__restrict__ qx,
                                                        int32_t *__restrict__ gsum, uint8_t *__restrict__ qop,
                                                        float *__restrict__ sx) {
    __shared__ float s_red[T / 32];
    __shared__ int s_gs[MAX_K / 16];  // group sums of this row
    pdl_wait();

    const int row = blockIdx.x;
    const int MT = gridDim.x;  // operand rows
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int n4 = K >> 2;  // float4s per row
    const int n4pad = act_blocks(K) * (ACT_BLOCK / 4);
    const int ngk = K / G;
    // operand: K tiles of KT features, each its code blocks then its group sums
    const int bpt = act_kt(G) / ACT_BLOCK;  // code blocks per K tile
    const int gpt = act_kt(G) / G;          // groups per K tile
    const int ngp = act_ktiles(K, G) * gpt; // groups of the operand, padding included
    // bytes per 128-feature block and per K tile: codes, then (where the GEMM
    // reads them) group sums
    const int cb = MT * (rs ? ACT_RS_PITCH : 256);
    const size_t tb = (size_t)bpt * cb + (sums ? (size_t)gpt * MT * 4 : 0);
    // operand position of group sum g of this row
    auto op_s = [&](int g) -> float * {
        return reinterpret_cast<float *>(qop + (size_t)(g / gpt) * tb + (size_t)bpt * cb) + (size_t)(g % gpt) * MT + row;
    };
    // byte offset of the 4 features 4*idx .. 4*idx+3 of this row in the
    // operand: fp16, 8 bytes; digits, 4 bytes of low digits (the high digits
    // are MT rows further)
    auto op_off = [&](int idx) -> size_t {
        const int f = idx * 4;
        const int kb = f / ACT_BLOCK, fb = f % ACT_BLOCK;
        const int kt = bpt == 1 ? kb : kb >> 1, kbi = bpt == 1 ? 0 : kb & 1;  // bpt is 1 or 2
        const size_t blk = (size_t)kt * tb + (size_t)kbi * cb;
        if (rs) return blk + (size_t)row * ACT_RS_PITCH + (size_t)fb * 2;
        if (e4) return blk + ((size_t)(fb / 16) * 2 * MT + row) * 16 + (size_t)(fb % 16);
        return blk + ((size_t)(fb / 8) * MT + row) * 16 + (size_t)(fb % 8) * 2;
    };

    if (row >= M) {
        // padding row of the operand: zero codes, zero group sums
        if (qop) {
            for (int idx = tid; idx < n4pad; idx += T) {
                if (e4) {
                    *reinterpret_cast<uint32_t *>(qop + op_off(idx)) = 0u;
                    *reinterpret_cast<uint32_t *>(qop + op_off(idx) + (size_t)MT * 16) = 0u;
                } else {
                    *reinterpret_cast<uint2 *>(qop + op_off(idx)) = make_uint2(0u, 0u);
                }
            }
            if (sums)
                for (int g = tid; g < ngp; g += T) *op_s(g) = 0.0f;
        }
        pdl_launch_dependents();
        return;
    }
    // group sums: for the caller (gsum) or for the operand (sums)
    const bool need_gs = gsum != nullptr || (qop != nullptr && sums != 0);
    if (need_gs)
        for (int g = tid; g < ngk; g += T) s_gs[g] = 0;

    const float c = __int_as_float((int)HADAMARD_SCALE_BITS);
    const float4 *xr = reinterpret_cast<const float4 *>(X + (size_t)row * K);

    float4 v[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = tid + j * T;
        v[j] = idx < n4 ? __ldg(xr + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = tid + j * T;
        // signs of features 4*idx .. 4*idx+3
        uint32_t sw = 0;
        if (idx < n4) sw = __ldg(signs + (idx >> 3)) >> ((idx & 7) * 4);
        float a0 = flip(v[j].x, sw & 1u), a1 = flip(v[j].y, (sw >> 1) & 1u);
        float a2 = flip(v[j].z, (sw >> 2) & 1u), a3 = flip(v[j].w, (sw >> 3) & 1u);
        // stride 1
        float t0 = __fadd_rn(a0, a1), t1 = __fsub_rn(a0, a1);
        float t2 = __fadd_rn(a2, a3), t3 = __fsub_rn(a2, a3);
        // stride 2
        a0 = __fadd_rn(t0, t2);
        a2 = __fsub_rn(t0, t2);
        a1 = __fadd_rn(t1, t3);
        a3 = __fsub_rn(t1, t3);
        // strides 4, 8, 16 across lanes
#pragma unroll
        for (int lb = 1; lb <= 4; lb <<= 1) {
            const bool up = (lane & lb) != 0;
            a0 = bfly_x(a0, lb, up);
            a1 = bfly_x(a1, lb, up);
            a2 = bfly_x(a2, lb, up);
            a3 = bfly_x(a3, lb, up);
        }
        a0 = __fmul_rn(a0, c);
        a1 = __fmul_rn(a1, c);
        a2 = __fmul_rn(a2, c);
        a3 = __fmul_rn(a3, c);
        v[j] = make_float4(a0, a1, a2, a3);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(a2), fabsf(a3))));
    }

    // The dependent GEMM may launch now that this block's reads of X are in:
    // its blocks' weight prefetch then no longer delays those reads.
    pdl_launch_dependents();

    // row absmax: warp, then every warp reduces the warps' maxima itself
    // (one block barrier; it also orders the zeroing of s_gs before the adds)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_red[tid >> 5] = amax;
    __syncthreads();
    float a = lane < T / 32 ? s_red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float s = a == 0.0f ? 0.0f : __fdiv_rn(a, 127.0f);
    if (tid == 0) sx[row] = s;

    // outputs: int8 codes and/or the GEMM operand (the same codes as fp16,
    // exact), 4 features per thread; the operand's padding past K is zeroed.
    // Group sums: the G/4 consecutive threads of a group (within a warp for
    // G <= 128) reduce by shuffles, one lane adds into shared memory.
    char4 *qr = qx ? reinterpret_cast<char4 *>(qx + (size_t)row * K) : nullptr;
    const int width = G / 4 < 32 ? G / 4 : 32;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int idx = tid + j * T;
        int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
        if (s != 0.0f && idx < n4) {
            q0 = min(127, max(-127, __float2int_rn(__fdiv_rn(v[j].x, s))));
            q1 = min(127, max(-127, __float2int_rn(__fdiv_rn(v[j].y, s))));
            q2 = min(127, max(-127, __float2int_rn(__fdiv_rn(v[j].z, s))));
            q3 = min(127, max(-127, __float2int_rn(__fdiv_rn(v[j].w, s))));
        }
        if (qr && idx < n4) qr[idx] = make_char4((signed char)q0, (signed char)q1, (signed char)q2, (signed char)q3);
        if (qop && idx < n4pad) {
            if (e4) {
                uint32_t lo, hi;
                digits4(q0, q1, q2, q3, lo, hi);
                *reinterpret_cast<uint32_t *>(qop + op_off(idx)) = lo;
                *reinterpret_cast<uint32_t *>(qop + op_off(idx) + (size_t)MT * 16) = hi;
            } else {
                const uint32_t h0 = __half_as_ushort(__int2half_rn(q0)), h1 = __half_as_ushort(__int2half_rn(q1));
                const uint32_t h2 = __half_as_ushort(__int2half_rn(q2)), h3 = __half_as_ushort(__int2half_rn(q3));
                *reinterpret_cast<uint2 *>(qop + op_off(idx)) = make_uint2(h0 | (h1 << 16), h2 | (h3 << 16));
            }
        }
        // every thread of the warp takes part in the shuffles (lanes past the
        // row's end add zeros); a group's G/4 threads are consecutive lanes
        if (need_gs) {
            int gs = q0 + q1 + q2 + q3;
            for (int o = width / 2; o > 0; o >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
            if (idx < n4 && (lane & (width - 1)) == 0) atomicAdd(&s_gs[(idx * 4) / G], gs);
        }
    }
    if (!need_gs) return;
    __syncthreads();
    for (int g = tid; g < ngp; g += T) {
        const int v2 = g < ngk ? s_gs[g] : 0;
        if (gsum && g < ngk) gsum[(size_t)row * ngk + g] = v2;
        if (qop && sums) *op_s(g) = (float)v2;
    }
}

// int8 codes [M][K] -> the GEMM's operand (the same layout and values as
// k_rotate_quant_act writes for these codes): one block per operand row,
// rows past M and features past K zero; group sums formed from the codes.
__global__ void __launch_bounds__(256) k_codes_to_operand(const int8_t *__restrict__ qx, int M, int K, int G, int rs,
                                                          int e4, int sums, uint8_t *__restrict__ qop) {
    constexpr int T = 256;
    pdl_wait();
    // the dependent GEMM may start streaming its weights; its reads of the
    // operand wait for this grid's completion
    pdl_launch_dependents();
    const int row = blockIdx.x, MT = gridDim.x, tid = threadIdx.x;
    const int n4 = K >> 2, n4pad = act_blocks(K) * (ACT_BLOCK / 4);
    const int bpt = act_kt(G) / ACT_BLOCK, gpt = act_kt(G) / G;
    const int cb = MT * (rs ? ACT_RS_PITCH : 256);
    const size_t tb = (size_t)bpt * cb + (sums ? (size_t)gpt * MT * 4 : 0);
    const bool live = row < M;
    for (int idx = tid; idx < n4pad; idx += T) {
        int q[4] = {0, 0, 0, 0};
        if (live && idx < n4) {
            const char4 c = reinterpret_cast<const char4 *>(qx + (size_t)row * K)[idx];
            q[0] = c.x;
            q[1] = c.y;
            q[2] = c.z;
            q[3] = c.w;
        }
        const int f = idx * 4, kb = f / ACT_BLOCK, fb = f % ACT_BLOCK;
        const int kt = bpt == 1 ? kb : kb >> 1, kbi = bpt == 1 ? 0 : kb & 1;
        const size_t blk = (size_t)kt * tb + (size_t)kbi * cb;
        if (e4) {
            uint32_t lo, hi;
            digits4(q[0], q[1], q[2], q[3], lo, hi);
            const size_t o = blk + ((size_t)(fb / 16) * 2 * MT + row) * 16 + (size_t)(fb % 16);
            *reinterpret_cast<uint32_t *>(qop + o) = lo;
            *reinterpret_cast<uint32_t *>(qop + o + (size_t)MT * 16) = hi;
        } else {
            uint32_t h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) h[i] = __half_as_ushort(__int2half_rn(q[i]));
            const size_t o = rs ? blk + (size_t)row * ACT_RS_PITCH + (size_t)fb * 2
                                : blk + ((size_t)(fb / 8) * MT + row) * 16 + (size_t)(fb % 8) * 2;
            *reinterpret_cast<uint2 *>(qop + o) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        }
    }
    if (sums) {
        const int ngp = act_ktiles(K, G) * gpt;
        for (int g = tid; g < ngp; g += T) {
            int acc = 0;
            if (live)
                for (int k = g * G; k < (g + 1) * G && k < K; ++k) acc += qx[(size_t)row * K + k];
            float *d = reinterpret_cast<float *>(qop + (size_t)(g / gpt) * tb + (size_t)bpt * cb) + (size_t)(g % gpt) * MT + row;
            *d = (float)acc;
        }
    }
}

template <int V, int T>
cudaError_t launch_act_t(const float *X, int M, int K, int G, bool rs, bool e4, const uint32_t *signs, int8_t *qx,
                         int32_t *gsum, uint8_t *qop, float *sx, bool pdl, cudaStream_t s, bool sums) {
    cudaLaunchConfig_t cfg = {};
    // one block per operand row (rows past M write the operand's zero padding)
    cfg.gridDim = dim3((unsigned)(qop ? act_rows(M) : M));
    cfg.blockDim = dim3(T);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_rotate_quant_act<V, T>, X, M, K, G, rs ? 1 : 0, e4 ? 1 : 0, sums ? 1 : 0, signs, qx, gsum, qop,
                              sx);
}

}  // namespace

cudaError_t launch_rotate_quant_act(const float *X, int M, int K, int G, bool rs, bool e4, bool sums, const uint32_t *signs,
                                    int8_t *qx, int32_t *gsum, uint8_t *qop, float *sx, bool pdl, cudaStream_t s) {
    // As many threads per row as the row has float4s, up to 1024: the kernel
    // is latency-bound (one block per row), so the shortest chain per thread
    // wins (256 threads x 4 float4s at K = 4096 made the pass 4% slower).
    const int n4 = K / 4;
    if (n4 <= 256 * 1) return launch_act_t<1, 256>(X, M, K, G, rs, e4, signs, qx, gsum, qop, sx, pdl, s, sums);
    if (n4 <= 512 * 1) return launch_act_t<1, 512>(X, M, K, G, rs, e4, signs, qx, gsum, qop, sx, pdl, s, sums);
    if (n4 <= 1024 * 1) return launch_act_t<1, 1024>(X, M, K, G, rs, e4, signs, qx, gsum, qop, sx, pdl, s, sums);
    if (n4 <= 1024 * 2) return launch_act_t<2, 1024>(X, M, K, G, rs, e4, signs, qx, gsum, qop, sx, pdl, s, sums);
    if (n4 <= 1024 * 3) return launch_act_t<3, 1024>(X, M, K, G, rs, e4, signs, qx, gsum, qop, sx, pdl, s, sums);
    if (n4 <= 1024 * 4) return launch_act_t<4, 1024>(X, M, K, G, rs, e4, signs, qx, gsum, qop, sx, pdl, s, sums);
    if (n4 <= 1024 * 8) return launch_act_t<8, 1024>(X, M, K, G, rs, e4, signs, qx, gsum, qop, sx, pdl, s, sums);
    if (n4 <= 1024 * 16) return launch_act_t<16, 1024>(X, M, K, G, rs, e4, signs, qx, gsum, qop, sx, pdl, s, sums);
    return cudaErrorInvalidValue;
}

cudaError_t launch_codes_to_operand(const int8_t *qx, int M, int K, int G, bool rs, bool e4, bool sums, uint8_t *qop,
                                    bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)act_rows(M));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_codes_to_operand, qx, M, K, G, rs ? 1 : 0, e4 ? 1 : 0, sums ? 1 : 0, qop);
}

}  // namespace hq
