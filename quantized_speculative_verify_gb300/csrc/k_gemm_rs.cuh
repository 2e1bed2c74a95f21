// k_gemm_rs.cuh -- the verify GEMM for up to 32 token rows, with every
// partial sum in registers: warp-level fp16 MMAs on the weights
// widened straight from the packed tile, the per-group dequantization folded
// into the fp32 sums as each group ends.
//
// Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling":
// section "How Uzu optimizes bytes and tokens per pass" (both operands of the
// verify matmul are integers; Medium weights are 4-bit asymmetric, Large
// 8-bit symmetric, grouped along K) and section "Producing several tokens from one model pass" (the
// verify batch: a draft tree of up to 32 tokens shares one weight stream).
//
// Exact integer contraction on fp16 MMAs (mma.sync m16n8k16, fp32
// accumulate): 4-bit weight codes minus the zero point (|q - z| <= 15),
// 8-bit weight codes and activation codes (|q| <= 127) are exact in fp16,
// their products exact in
// fp32, and a group's sum stays below 2^24, so each group's accumulator holds
// the integer partial sum P of the Medium identity exactly (with the zero
// point applied to the weights, no group-sum correction is needed).  With at
// most 32 rows the kernel is bound by instruction issue, not by the tensor
// pipe: the fp16 form issues one instruction per MMA and needs no split of
// the activation codes, where the e4m3 forms on this GPU take several.
//
// Channels are the MMA's M (16 per warp), tokens its N (8 per MMA), so the
// weights are the A operand.  The packed layout gives lane t of a quad one
// 32-bit word per channel and 32 features: the feature pairs (2t, 2t + 1)
// and (2t + 8, 2t + 9) of two 16-feature MMA steps, one pair per nibble
// column.  A mask lifts a pair into the two halves of a register under the
// fp16 exponent bits of 1024, which reads 1024 + q (low nibbles) or
// 1024 + 16 q (high nibbles); one fp16 add of -(1024 + z), or a multiply-add
// by 1/16 and -(64 + z), leaves q - z exactly.  Eight codes cost nine
// instructions (four masks, a shift for the second step, four adds).  8-bit
// codes: lane t's word of a 16-feature run holds the same four features as
// bytes; a bias to unsigned, two byte permutes under the exponent bits of
// 1024 and two fp16 subtractions of 1152 give the two pairs.  The
// activation codes come from the operand's fp16 rows through ldmatrix.
//
// Fold of a group into the running sums, in the oracle's ascending group
// order: y += scale * P.  Exact-order and check modes round the multiply and
// the add separately (the oracle's arithmetic; the partial sums P written in
// check mode); otherwise one fused multiply-add, within the fp32 tolerance of
// the oracle.
//
// Thread block: one lane of warp 0 streams the weight tiles and the
// activation K tiles (gemm_common.cuh), warps 1..4 compute, three blocks per
// SM.  Consumer warp w owns channels 32 w .. 32 w + 31 of every tile (two MMA
// row tiles) and every token; it needs no other warp between a stage's
// arrival and its release.
#pragma once

#include <cuda_runtime.h>

#include "gemm_common.cuh"
#include "hq_internal.cuh"
#include "hq_tc.cuh"

namespace hq {


constexpr int RS_CONSUMERS = 8 / RS_RT;              // consumer warps: the tile's 128 channels
constexpr int RS_THREADS = (1 + RS_CONSUMERS) * 32;  // + the producer

// D (+)= A (16 x 16 fp16, row-major) x B (16 x 8 fp16, column-major).  A
// function of its registers alone (not volatile): the compiler may move the
// next step's loads ahead of it.
__device__ __forceinline__ void mma_f16_acc(float (&d)[4], const uint32_t (&A)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(A[0]), "r"(A[1]), "r"(A[2]), "r"(A[3]), "r"(b0), "r"(b1));
}
// same with a zero accumulator input (a group's first K step)
__device__ __forceinline__ void mma_f16_zero(float (&d)[4], const uint32_t (&A)[4], uint32_t b0, uint32_t b1) {
    const float z = 0.0f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(A[0]), "r"(A[1]), "r"(A[2]), "r"(A[3]), "r"(b0), "r"(b1), "f"(z));
}
// The pair in nibbles (0, 4) of each half-word (bits 0..3, 16..19) ->
// fp16x2 (q - z), zlo = fp16x2(-(1024 + z)).
__device__ __forceinline__ uint32_t widen_lo(uint32_t w, uint32_t zlo) {
    const uint32_t x = (w & 0x000F000Fu) | 0x64006400u;
    uint32_t r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(zlo));
    return r;
}
// The pair at bits 4..7, 20..23 -> fp16x2 (q - z), zhi = fp16x2(-(64 + z)).
__device__ __forceinline__ uint32_t widen_hi(uint32_t w, uint32_t zhi) {
    const uint32_t x = (w & 0x00F000F0u) | 0x64006400u;
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0x2C002C00u), "r"(zhi));  // x / 16 - (64 + z)
    return r;
}
// Four int8 codes (bytes 0..3 of w) -> the fp16x2 q of bytes (0, 1) in lo
// and (2, 3) in hi: biased to unsigned under the fp16 exponent bits 0x64
// (1024 + 128 + q), then 1152 subtracted, exactly.
__device__ __forceinline__ void widen_i8_pairs(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t l, h;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(l) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(h) : "r"(u), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(0x64806480u));
}
// four 8 x 16-byte row blocks of shared memory, one row address per lane
// (a memory read: it stays after the wait for the stage)
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(addr)
        : "memory");
}

// FMT: weight format; MT: token rows (16 or 32); G: quantization group
// (16 .. 256), fixed at compile time so that a tile's K steps and groups
// unroll completely.
template <int FMT, int MT, int G, bool EXACT>
__global__ void __launch_bounds__(RS_THREADS, rs_bps(MT)) k_verify_gemm_rs(const GemmArgs a) {
    constexpr int NT = MT / 8;             // MMA column tiles of tokens
    constexpr int KT = G > 128 ? G : 128;  // features per tile
    constexpr int GPT = KT / G;            // groups per tile
    constexpr int KS = G / 16;             // K steps of 16 features per group
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw);
    uint64_t *empty = full + MAX_STAGES;
    // accumulating mode: two segment flags; then the initial fill's counter
    int *sflag = reinterpret_cast<int *>(empty + MAX_STAGES);
    uint8_t *ring = smem_raw + 1024;
    const int S = a.stages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const GemmBlock blk = make_gemm_block(a, ring, full, empty, sflag);
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_addr(&full[i]), 2);             // the two producers' arrivals
            mbar_init(smem_addr(&empty[i]), RS_CONSUMERS);  // one per consumer warp
        }
        sflag[0] = sflag[1] = sflag[2] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == 0) {
        // two stages of weights before the dependency wait
        if (lane == 0) gemm_producer(a, blk, 2);
        return;
    }

    // ------------------------------------------------------------ consumers ---
    pdl_wait();
    const int cw = warp - 1;                  // consumer warp: channels 16 RT cw .. 16 RT (cw + 1) - 1
    const int ctid = threadIdx.x - 32;        // consumer thread 0 .. RS_CONSUMERS * 32 - 1
    const int g = lane >> 2, tig = lane & 3;  // MMA lane coordinates
    const int M = a.M, KTILES = a.KTILES;
    float *wsp = reinterpret_cast<float *>(a.ws + ws_partial_offset());
    bool ok = true;
    int pend0 = -1, pend1 = -1, nsplit = 0;
    const int first_b = blk.t0 / KTILES;
    const int mark_old = gemm_zero_outputs(a, blk, ctid, RS_CONSUMERS * 32, 1);

    constexpr int RT = RS_RT;
    // y[r][n][e]: channel 16 (RT cw + r) + g + 8 (e >> 1), token 8 n + 2 tig + (e & 1)
    float y[RT][NT][4];
    int eb = blk.t0 / KTILES, ekt = blk.t0 - eb * KTILES, seg_k0 = ekt;
    const int chw = 16 * RT * cw + g;  // the lane's channels: chw + 16 r, + 8

    // lane's ldmatrix row within a 4-matrix load: matrix (lane >> 3) holds
    // features +0..7 / +8..15 (bit 0) of tokens +0..7 / +8..15 (bit 1); the
    // operand's blocks are [MT rows][272 bytes]
    const int lm = lane >> 3, lr = lane & 7;
    const uint32_t lrow_off = (uint32_t)(((lm >> 1) * 8 + lr) * ACT_RS_PITCH + (lm & 1) * 16);

    RingPos ps{0, 0u};
    for (int u = 0; u < blk.nunits; ++u) {
        const int nt = blk.unit_tiles(u);
        const int st = ps.slot;
        if (ok) ok = mbar_wait_bounded(smem_addr(&full[st]), ps.phase, blk.err);
        const uint8_t *stage = ring + (size_t)st * a.stage_bytes;
#pragma unroll
        for (int j = 0; j < RS_UNIT; ++j) {
            if (j >= nt) break;
            const int i = u * blk.U + j;
            if (i == 0 || ekt == 0) {
                seg_k0 = ekt;
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e) y[r][n][e] = 0.0f;
            }
            const uint8_t *tile = stage + (size_t)j * a.tile_bytes;
            const float *tsc = reinterpret_cast<const float *>(tile + a.code_bytes);  // scales [channel][GPT]
            const uint8_t *tzp = tile + a.code_bytes + a.scale_bytes;                // zero nibbles [channel * GPT + g]
            const uint32_t act_s = smem_addr(stage + a.act_off + (size_t)j * a.act_tile_bytes);
            // the lane's word of its channels' runs: [KT / 32 (4-bit) or KT / 16
            // (8-bit) runs][BN][4 words]
            const uint32_t *wc0 = reinterpret_cast<const uint32_t *>(tile) + 4 * chw + tig;
            // the current run's word of each channel (two 16-feature steps,
            // which may belong to two groups)
            uint32_t wq[RT][2];
#pragma unroll
            for (int gl = 0; gl < GPT; ++gl) {
                // zero points -> the widening's additive constants (fp16 bits of
                // -(1024 + z) = 0xE400 + z, of -(64 + z) = 0xD400 + 16 z); scales
                uint32_t zlo[RT][2], zhi[RT][2];
                float sc[RT][2];
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int zi = (chw + 16 * r + 8 * h) * GPT + gl;
                        if (FMT == HQ_W4_ASYM) {
                            const uint32_t z = (tzp[zi >> 1] >> ((zi & 1) * 4)) & 15u;
                            zlo[r][h] = z * 0x00010001u + 0xE400E400u;
                            zhi[r][h] = z * 0x00100010u + 0xD400D400u;
                        }
                        sc[r][h] = tsc[zi];
                    }
                float acc[RT][NT][4];
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int s = gl * KS + ks;  // 16-feature step of the tile
                    // B: tokens' fp16 codes, features 16 s ..: block s / 8, chunks 2 (s % 8), + 1
                    const uint32_t b_s = act_s + (uint32_t)((s >> 3) * (MT * ACT_RS_PITCH) + (s & 7) * 32);
                    uint32_t bq[NT / 2][4];
#pragma unroll
                    for (int n2 = 0; n2 < NT; n2 += 2)
                        ldmatrix_x4(bq[n2 / 2], b_s + lrow_off + (uint32_t)(n2 * 8 * ACT_RS_PITCH));
#pragma unroll
                    for (int r = 0; r < RT; ++r) {
                        // A: rows g, g + 8 (channels chw + 16 r, + 8), features
                        // 2 tig, + 1 and 2 tig + 8, + 9 of the step
                        uint32_t A[4];
                        if (FMT == HQ_W4_ASYM) {
                            if ((s & 1) == 0) {
                                wq[r][0] = wc0[4 * ((s >> 1) * BN + 16 * r)];
                                wq[r][1] = wc0[4 * ((s >> 1) * BN + 16 * r + 8)];
                            }
                            // nibbles 0, 4 and 1, 5 of the step's half-words;
                            // the odd step's pairs sit 8 bits higher
                            const uint32_t v0 = (s & 1) ? wq[r][0] >> 8 : wq[r][0];
                            const uint32_t v1 = (s & 1) ? wq[r][1] >> 8 : wq[r][1];
                            A[0] = widen_lo(v0, zlo[r][0]);
                            A[1] = widen_lo(v1, zlo[r][1]);
                            A[2] = widen_hi(v0, zhi[r][0]);
                            A[3] = widen_hi(v1, zhi[r][1]);
                        } else {
                            // one word per channel and step: bytes (0, 1), (2, 3)
                            widen_i8_pairs(wc0[4 * (s * BN + 16 * r)], A[0], A[2]);
                            widen_i8_pairs(wc0[4 * (s * BN + 16 * r + 8)], A[1], A[3]);
                        }
#pragma unroll
                        for (int n2 = 0; n2 < NT; n2 += 2) {
                            if (ks == 0) {
                                mma_f16_zero(acc[r][n2], A, bq[n2 / 2][0], bq[n2 / 2][1]);
                                mma_f16_zero(acc[r][n2 + 1], A, bq[n2 / 2][2], bq[n2 / 2][3]);
                            } else {
                                mma_f16_acc(acc[r][n2], A, bq[n2 / 2][0], bq[n2 / 2][1]);
                                mma_f16_acc(acc[r][n2 + 1], A, bq[n2 / 2][2], bq[n2 / 2][3]);
                            }
                        }
                    }
                }
                // fold the group: y += scale * P (P exact in acc)
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float s_ch = sc[r][e >> 1];
                            if constexpr (EXACT) {
                                if (a.partials) {
                                    const int tok = 8 * n + 2 * tig + (e & 1);
                                    const int nn = eb * BN + chw + 16 * r + 8 * (e >> 1);
                                    const int gq = ekt * GPT + gl;
                                    if (tok < M && nn < a.N && gq < a.NGK)
                                        a.partials[((size_t)tok * a.N + nn) * a.NGK + gq] = __float2int_rn(acc[r][n][e]);
                                }
                                // y += scale * P: product rounded, then sum rounded
                                y[r][n][e] = __fadd_rn(y[r][n][e], __fmul_rn(s_ch, acc[r][n][e]));
                            } else {
                                y[r][n][e] = fmaf(s_ch, acc[r][n][e], y[r][n][e]);
                            }
                        }
            }
            // end of an n-block segment?
            if (ekt == KTILES - 1 || i == blk.ntl - 1) {
                int kind;
                float *slot_base = nullptr;
                if (seg_k0 == 0 && ekt == KTILES - 1) {
                    kind = SEG_FULL;  // the whole K range of the n-block
                } else if (blk.det) {
                    kind = SEG_PUBLISH;
                    const int slot = eb == first_b ? 0 : 1;
                    slot_base = wsp + ((size_t)blockIdx.x * 2 + slot) * ws_slot_floats();
                    if (slot == 0)
                        pend0 = eb;
                    else
                        pend1 = eb;
                } else {
                    kind = SEG_ADD;  // once the zeroing is visible (the segment's flag)
                    if (ok) ok = wait_flag_bounded(smem_addr(&sflag[nsplit]), blk.err);
                    ++nsplit;
                }
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int nl = chw + 16 * r + 8 * (e >> 1);
                            gemm_segment_out(a, kind, slot_base, 8 * n + 2 * tig + (e & 1), nl, eb * BN + nl,
                                             y[r][n][e]);
                        }
            }
            if (++ekt == KTILES) {
                ekt = 0;
                ++eb;
            }
        }
        // this warp no longer reads the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
        ps.next(S);
    }

    gemm_finish(a, blk, ok, pend0, pend1, mark_old, ctid, RS_CONSUMERS * 32, 1);
}

template <int FMT, int MT, int G, bool EXACT>
cudaError_t launch_gemm_rs_instance(const GemmArgs &a, bool pdl, cudaStream_t s) {
    auto kern = k_verify_gemm_rs<FMT, MT, G, EXACT>;
    const size_t smem = 1024 + (size_t)a.stages * (size_t)a.stage_bytes;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<int> configured[CACHE_DEVICES];
    int done = 0;
    e = cached_per_device(configured, dev, &done, [&](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_LIMIT);
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.grid);
    cfg.blockDim = dim3(RS_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int FMT, int MT, bool EXACT>
cudaError_t launch_gemm_rs_g(const GemmArgs &a, bool pdl, cudaStream_t s) {
    switch (a.G) {
        case 16: return launch_gemm_rs_instance<FMT, MT, 16, EXACT>(a, pdl, s);
        case 32: return launch_gemm_rs_instance<FMT, MT, 32, EXACT>(a, pdl, s);
        case 64: return launch_gemm_rs_instance<FMT, MT, 64, EXACT>(a, pdl, s);
        case 128: return launch_gemm_rs_instance<FMT, MT, 128, EXACT>(a, pdl, s);
        case 256: return launch_gemm_rs_instance<FMT, MT, 256, EXACT>(a, pdl, s);
        default: return cudaErrorInvalidValue;
    }
}

// Weights of format FMT, the fp16 row operand, up to 32 rows.
template <int FMT>
cudaError_t launch_gemm_rs(const GemmArgs &a, bool pdl, cudaStream_t s) {
    const bool exact = a.partials != nullptr || a.nb_align != 0;
    if (act_rows(a.M) <= 16)
        return exact ? launch_gemm_rs_g<FMT, 16, true>(a, pdl, s) : launch_gemm_rs_g<FMT, 16, false>(a, pdl, s);
    return exact ? launch_gemm_rs_g<FMT, 32, true>(a, pdl, s) : launch_gemm_rs_g<FMT, 32, false>(a, pdl, s);
}

}  // namespace hq
