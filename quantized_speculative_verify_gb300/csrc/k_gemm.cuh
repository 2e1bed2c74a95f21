// k_gemm.cuh -- the verify GEMM: int8 activations x packed 4-/8-bit weights,
// per-group int32 partial sums, fp32 dequantization epilogue.
//
// Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling":
// section "How Uzu optimizes bytes and tokens per pass" (both operands of the
// verify matmul are integers and run on the int8 matrix path; Medium weights
// are 4-bit asymmetric, Large 8-bit symmetric, grouped along K) and section
// "Why batch-one decoding is memory-bound" (the pass streams every weight
// once, so the kernel is bound by memory bandwidth, not arithmetic).
//
// Work decomposition (stream-K).  The blob is a sequence of T tiles
// (n-block major, K minor).  Thread block c owns tiles [c*T/grid,
// (c+1)*T/grid): one contiguous byte range of the blob.  A block whose range
// covers an n-block from its first to its last K tile writes Y directly; an
// n-block split between blocks is finished by whichever contributor arrives
// last (arrival counter, no waiting), which sums the contributors' fp32
// partial sums in ascending K order.
//
// Inside a block: one producer warp issues one bulk copy per tile into a ring
// of shared-memory stages (mbarrier transaction counts); NCW consumer warps
// each own NW row tiles of 16 channels of the 128-channel n-block and walk the
// tiles in K order.  Per k32 step a lane loads 8 bytes of int8 activations
// per 8-token column tile (the B operand of mma.m16n8k32) and reads its
// 16-byte weight fragment from shared memory (the A operand: 16 channels x
// 32 features; 4-bit codes are widened to bytes with two masks).  After each
// quantization group: P = acc - zero * gsum (int32, exact), then
// y += scale * float(P) with separately rounded fp32 multiply and add, group
// by group in ascending order.
#pragma once

#include <cuda_runtime.h>

#include "hq_internal.cuh"

namespace hq {

struct GemmArgs {
    const uint8_t *blob;
    const int8_t *qx;
    const float *sx;
    const int32_t *gsum;
    float *Y;
    int32_t *partials;
    uint8_t *ws;
    size_t ws_partial_off;  // byte offset of the partial-sum slots in ws
    int M, N, K, NGK, KTILES, T, grid, stages;
    int tile_bytes, code_bytes, scale_bytes;
};

__device__ __forceinline__ int tile_begin(int c, int T, int grid) { return (int)(((long long)c * T) / grid); }
// thread block whose range contains tile t
__device__ __forceinline__ int cta_of_tile(int t, int T, int grid) {
    return (int)((((long long)t + 1) * grid - 1) / T);
}

// End of one quantization group: P = acc - zero * gsum (exact int32), then
// y += scale * float(P), one IEEE-rounded multiply and one add per output.
// gl = group within the tile, gg = group along the whole K.
template <int FMT, int MT, int NW>
__device__ __forceinline__ void group_epilogue(const GemmArgs &a, int (&iacc)[NW][MT][4], float (&facc)[NW][MT][4],
                                               const float *tsc, const uint8_t *tzp, int gl, int gg, int b, int warp,
                                               int g8, int tig) {
    int gs[MT][2];
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) {
        const int tok0 = tt * 8 + tig * 2;
        gs[tt][0] = (FMT == HQ_W4_ASYM && tok0 < a.M) ? __ldg(a.gsum + (size_t)tok0 * a.NGK + gg) : 0;
        gs[tt][1] = (FMT == HQ_W4_ASYM && tok0 + 1 < a.M) ? __ldg(a.gsum + (size_t)(tok0 + 1) * a.NGK + gg) : 0;
    }
#pragma unroll
    for (int j = 0; j < NW; ++j) {
        const int nt = warp * NW + j;
        const float2 sc = *reinterpret_cast<const float2 *>(tsc + ((size_t)gl * NTILES + nt) * 16 + 2 * g8);
        int zl = 0, zh = 0;
        if (FMT == HQ_W4_ASYM) {
            const int zb = tzp[((size_t)gl * NTILES + nt) * 8 + g8];
            zl = zb & 15;
            zh = zb >> 4;
        }
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) {
            int p[4];
            p[0] = iacc[j][tt][0] - zl * gs[tt][0];
            p[1] = iacc[j][tt][1] - zl * gs[tt][1];
            p[2] = iacc[j][tt][2] - zh * gs[tt][0];
            p[3] = iacc[j][tt][3] - zh * gs[tt][1];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float s = (e >> 1) ? sc.y : sc.x;
                facc[j][tt][e] = __fadd_rn(facc[j][tt][e], __fmul_rn(s, __int2float_rn(p[e])));
                iacc[j][tt][e] = 0;
            }
            if (a.partials) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = tt * 8 + tig * 2 + (e & 1);
                    const int n = b * BN + nt * 16 + g8 + 8 * (e >> 1);
                    if (tok < a.M && n < a.N) a.partials[((size_t)tok * a.N + n) * a.NGK + gg] = p[e];
                }
            }
        }
    }
}

template <int FMT, int G, int MT, int NW>
struct GemmCfg {
    static constexpr int KT = G > 128 ? G : 128;
    static constexpr int STEPS = KT / 32;   // k32 steps per tile
    static constexpr int GPT = KT / G;      // groups per tile
    static constexpr int NCW = NTILES / NW; // consumer warps
    static constexpr int THREADS = (NCW + 1) * 32;
};

template <int FMT, int G, int MT, int NW>
__global__ void __launch_bounds__(GemmCfg<FMT, G, MT, NW>::THREADS) k_verify_gemm(const GemmArgs a) {
    using C = GemmCfg<FMT, G, MT, NW>;
    constexpr int KT = C::KT, STEPS = C::STEPS, NCW = C::NCW;
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = a.stages;
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)S * a.tile_bytes);  // full[S], empty[S]
    int *s_flag = reinterpret_cast<int *>(bars + 2 * S);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = tile_begin(blockIdx.x, a.T, a.grid);
    const int t1 = tile_begin(blockIdx.x + 1, a.T, a.grid);
    const int ntl = t1 - t0;
    int *err = reinterpret_cast<int *>(a.ws);

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_addr(&bars[i]), 1);
            mbar_init(smem_addr(&bars[S + i]), NCW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == NCW) {
        // ------------------------------------------------------ producer ---
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int i = 0;
            // The weights never depend on earlier kernels of the stream: the
            // first stages are requested before waiting for them.
            for (; i < ntl && i < S; ++i) {
                const uint32_t fb = smem_addr(&bars[i]);
                mbar_arrive_expect_tx(fb, (uint32_t)a.tile_bytes);
                bulk_copy_g2s(smem_addr(ring + (size_t)i * a.tile_bytes),
                              a.blob + (size_t)(t0 + i) * (size_t)a.tile_bytes, (uint32_t)a.tile_bytes, fb, pol);
            }
            pdl_wait();
            for (; i < ntl; ++i) {
                const int st = i % S;
                const uint32_t ph = (uint32_t)((i / S) & 1);
                if (!mbar_wait_bounded(smem_addr(&bars[S + st]), ph ^ 1u, err)) break;
                const uint32_t fb = smem_addr(&bars[st]);
                mbar_arrive_expect_tx(fb, (uint32_t)a.tile_bytes);
                bulk_copy_g2s(smem_addr(ring + (size_t)st * a.tile_bytes),
                              a.blob + (size_t)(t0 + i) * (size_t)a.tile_bytes, (uint32_t)a.tile_bytes, fb, pol);
            }
            // No copy may still be landing in shared memory when the block exits.
            const int issued = i;
            for (int j = issued > S ? issued - S : 0; j < issued; ++j)
                mbar_wait_bounded(smem_addr(&bars[j % S]), (uint32_t)((j / S) & 1), err);
        }
        return;
    }

    // ---------------------------------------------------------- consumers ---
    pdl_wait();
    const int g8 = lane >> 2, tig = lane & 3;
    const int M = a.M, N = a.N, K = a.K, NGK = a.NGK;
    const int KTILES = a.KTILES;
    float *wsp = reinterpret_cast<float *>(a.ws + a.ws_partial_off);
    int *ctr = reinterpret_cast<int *>(a.ws + ws_counter_offset());

    int iacc[NW][MT][4];
    float facc[NW][MT][4];
    int seg_k0 = 0;
    bool ok = true;

    // A failed (timed-out) wait is sticky: the warp stops waiting but keeps
    // the same control flow, so every consumer warp still reaches each named
    // barrier and every arrival counter is still incremented and reset.
    for (int i = 0; i < ntl; ++i) {
        const int t = t0 + i;
        const int b = t / KTILES, kt = t - b * KTILES;
        if (i == 0 || kt == 0) {
            seg_k0 = kt;
#pragma unroll
            for (int j = 0; j < NW; ++j)
#pragma unroll
                for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) facc[j][tt][e] = 0.0f;
        }
        const int st = i % S;
        if (ok) ok = mbar_wait_bounded(smem_addr(&bars[st]), (uint32_t)((i / S) & 1), err);
        const uint8_t *tile = ring + (size_t)st * a.tile_bytes;
        const float *tsc = reinterpret_cast<const float *>(tile + a.code_bytes);
        const uint8_t *tzp = tile + a.code_bytes + a.scale_bytes;

#pragma unroll
        for (int j = 0; j < NW; ++j)
#pragma unroll
            for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                for (int e = 0; e < 4; ++e) iacc[j][tt][e] = 0;

        uint4 wchunk[NW];
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
            const int kg = kt * KT + s * 32;  // first feature of this k32 step
            if (kg >= K) break;               // padding past the real K
            // A operands (weights) from shared memory
            if (FMT == HQ_W8_SYM || (s & 1) == 0) {
                const int ch = FMT == HQ_W4_ASYM ? s >> 1 : s;
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    const int nt = warp * NW + j;
                    wchunk[j] = *reinterpret_cast<const uint4 *>(tile + (((size_t)ch * NTILES + nt) * 32 + lane) * 16);
                }
            }
            uint32_t A[NW][4];
#pragma unroll
            for (int j = 0; j < NW; ++j) {
                if (FMT == HQ_W4_ASYM) {
                    const uint32_t w0 = (s & 1) ? wchunk[j].z : wchunk[j].x;
                    const uint32_t w1 = (s & 1) ? wchunk[j].w : wchunk[j].y;
                    A[j][0] = w0 & 0x0F0F0F0Fu;
                    A[j][1] = (w0 >> 4) & 0x0F0F0F0Fu;
                    A[j][2] = w1 & 0x0F0F0F0Fu;
                    A[j][3] = (w1 >> 4) & 0x0F0F0F0Fu;
                } else {
                    A[j][0] = wchunk[j].x;
                    A[j][1] = wchunk[j].y;
                    A[j][2] = wchunk[j].z;
                    A[j][3] = wchunk[j].w;
                }
            }
            // B operands (activations): token column tile tt, token tt*8 + g8
            uint32_t B[MT][2];
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) {
                const int tok = tt * 8 + g8;
                if (tok < M) {
                    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(a.qx + (size_t)tok * K + kg + tig * 8));
                    B[tt][0] = v.x;
                    B[tt][1] = v.y;
                } else {
                    B[tt][0] = 0u;
                    B[tt][1] = 0u;
                }
            }
            if (G == 16) {
                // two groups per step: lanes tig 0,1 hold the first 16 features
                int iacc2[NW][MT][4];
#pragma unroll
                for (int j = 0; j < NW; ++j)
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) iacc2[j][tt][e] = 0;
                const bool lowhalf = tig < 2;
#pragma unroll
                for (int j = 0; j < NW; ++j)
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt) {
                        mma_s8_16832(iacc[j][tt], A[j][0], A[j][1], A[j][2], A[j][3], lowhalf ? B[tt][0] : 0u,
                                     lowhalf ? B[tt][1] : 0u);
                        mma_s8_16832(iacc2[j][tt], A[j][0], A[j][1], A[j][2], A[j][3], lowhalf ? 0u : B[tt][0],
                                     lowhalf ? 0u : B[tt][1]);
                    }
                group_epilogue<FMT, MT, NW>(a, iacc, facc, tsc, tzp, 2 * s, kt * C::GPT + 2 * s, b, warp, g8, tig);
                group_epilogue<FMT, MT, NW>(a, iacc2, facc, tsc, tzp, 2 * s + 1, kt * C::GPT + 2 * s + 1, b, warp,
                                            g8, tig);
            } else {
#pragma unroll
                for (int j = 0; j < NW; ++j)
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt)
                        mma_s8_16832(iacc[j][tt], A[j][0], A[j][1], A[j][2], A[j][3], B[tt][0], B[tt][1]);
                if (((s + 1) * 32) % G == 0) {
                    const int gl = ((s + 1) * 32) / G - 1;
                    group_epilogue<FMT, MT, NW>(a, iacc, facc, tsc, tzp, gl, kt * C::GPT + gl, b, warp, g8, tig);
                }
            }
        }
        // release the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bars[S + st]));

        // end of an n-block segment?
        if (kt == KTILES - 1 || i == ntl - 1) {
            const bool whole = seg_k0 == 0 && kt == KTILES - 1;
            if (whole) {
#pragma unroll
                for (int j = 0; j < NW; ++j)
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int row = (warp * NW + j) * 16 + g8 + 8 * (e >> 1);
                            const int tok = tt * 8 + tig * 2 + (e & 1);
                            const int n = b * BN + row;
                            if (tok < M && n < N) a.Y[(size_t)tok * N + n] = __fmul_rn(__ldg(a.sx + tok), facc[j][tt][e]);
                        }
            } else {
                // partial: publish, count arrivals, the last contributor finishes
                const int slot = (b == tile_begin(blockIdx.x, a.T, a.grid) / KTILES) ? 0 : 1;
                float *mys = wsp + ((size_t)blockIdx.x * 2 + slot) * ws_slot_floats(M);
#pragma unroll
                for (int j = 0; j < NW; ++j)
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int row = (warp * NW + j) * 16 + g8 + 8 * (e >> 1);
                            const int tok = tt * 8 + tig * 2 + (e & 1);
                            if (tok < M) __stcg(mys + (size_t)tok * BN + row, facc[j][tt][e]);
                        }
                __threadfence();
                named_barrier(1, NCW * 32);
                const int c_lo = cta_of_tile(b * KTILES, a.T, a.grid);
                const int c_hi = cta_of_tile(b * KTILES + KTILES - 1, a.T, a.grid);
                if (threadIdx.x == 0) {
                    const int prev = atomicAdd(&ctr[b], 1);
                    *s_flag = (prev == c_hi - c_lo) ? 1 : 0;
                }
                named_barrier(1, NCW * 32);
                if (*s_flag) {
                    __threadfence();
                    for (int idx = threadIdx.x; idx < M * BN; idx += NCW * 32) {
                        const int tok = idx / BN, row = idx - tok * BN;
                        float sum = 0.0f;
                        for (int cc = c_lo; cc <= c_hi; ++cc) {
                            const int sl = (b == tile_begin(cc, a.T, a.grid) / KTILES) ? 0 : 1;
                            sum = __fadd_rn(sum, __ldcg(wsp + ((size_t)cc * 2 + sl) * ws_slot_floats(M) +
                                                        (size_t)tok * BN + row));
                        }
                        const int n = b * BN + row;
                        if (n < N) a.Y[(size_t)tok * N + n] = __fmul_rn(__ldg(a.sx + tok), sum);
                    }
                    if (threadIdx.x == 0) atomicExch(&ctr[b], 0);
                }
                named_barrier(1, NCW * 32);
            }
        }
    }
    (void)NGK;
}

// Launch one instance.  Dynamic shared memory: the stage ring, 2*S mbarriers
// and a flag word.
template <int FMT, int G, int MT, int NW>
cudaError_t launch_gemm_instance(const GemmArgs &a, bool pdl, cudaStream_t s) {
    using C = GemmCfg<FMT, G, MT, NW>;
    auto kern = k_verify_gemm<FMT, G, MT, NW>;
    const size_t smem = (size_t)a.stages * (size_t)a.tile_bytes + (size_t)a.stages * 16 + 16;
    static int configured_for = -1;  // device the attribute was last set for
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_for != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        configured_for = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Instances for one format: M buckets {<=8, <=16, <=32, <=64, <=128}.
template <int FMT, int G>
cudaError_t launch_gemm_g(const GemmArgs &a, bool pdl, cudaStream_t s) {
    if (a.M <= 8) return launch_gemm_instance<FMT, G, 1, 2>(a, pdl, s);
    if (a.M <= 16) return launch_gemm_instance<FMT, G, 2, 2>(a, pdl, s);
    if (a.M <= 32) return launch_gemm_instance<FMT, G, 4, 2>(a, pdl, s);
    if (a.M <= 64) return launch_gemm_instance<FMT, G, 8, 1>(a, pdl, s);
    return launch_gemm_instance<FMT, G, 16, 1>(a, pdl, s);
}

template <int FMT>
cudaError_t launch_gemm_fmt(const GemmArgs &a, int G, bool pdl, cudaStream_t s) {
    switch (G) {
        case 16: return launch_gemm_g<FMT, 16>(a, pdl, s);
        case 32: return launch_gemm_g<FMT, 32>(a, pdl, s);
        case 64: return launch_gemm_g<FMT, 64>(a, pdl, s);
        case 128: return launch_gemm_g<FMT, 128>(a, pdl, s);
        case 256: return launch_gemm_g<FMT, 256>(a, pdl, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm_w4(const GemmArgs &a, int G, bool pdl, cudaStream_t s);
cudaError_t launch_gemm_w8(const GemmArgs &a, int G, bool pdl, cudaStream_t s);

}  // namespace hq
