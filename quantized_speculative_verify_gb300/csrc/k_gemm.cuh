// k_gemm.cuh -- the verify GEMM: activation codes x packed 4-/8-bit weights,
// per-group exact integer partial sums, fp32 dequantization epilogue.
//
// Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling":
// section "How Uzu optimizes bytes and tokens per pass" (both operands of the
// verify matmul are integers; Medium weights are 4-bit asymmetric, Large 8-bit
// symmetric, grouped along K) and section "Why batch-one decoding is
// memory-bound" (the pass streams every weight once, so the kernel is bound by
// memory bandwidth, not arithmetic).
//
// Integer arithmetic on fp16 tensor cores.  The int8 MMA rate of this GPU is
// far below its fp16 rate, so the integer contraction runs as an exact fp16
// MMA with fp32 accumulation: activation codes (|q| <= 127), weight codes
// minus zero point (|q - z| <= 15) and 8-bit weight codes (|q| <= 127) are
// exact in fp16, their products are exact in fp32, and a group's sum stays
// below 127 * 127 * 256 < 2^24, so the fp32 accumulator holds the integer
// partial sum P exactly.  The zero point is applied while widening the 4-bit
// codes: (1024 + q) - (1024 + z) = q - z in fp16.
//
// Work decomposition (stream-K).  The blob is a sequence of T tiles
// (n-block major, K minor).  Thread block c owns tiles [c*T/grid,
// (c+1)*T/grid): one contiguous byte range of the blob.  A block whose range
// covers an n-block from its first to its last K tile writes Y directly.  An
// n-block split between blocks is combined in one of two ways:
//  - accumulating (default): the block holding the n-block's first K tile
//    zeroes its outputs when it starts and marks the n-block's counter; each
//    contributor adds sx * (its partial sum) into Y with fp32 atomic adds as
//    soon as its segment ends and the mark is visible.  No block waits for
//    another's tiles; the order of the adds, and so the last bits of a split
//    output, may differ from run to run.
//  - deterministic (HQ_LAUNCH_DETERMINISTIC): each contributor stores its
//    partial sum; when all have arrived they share the work of summing them
//    in ascending K order, so results repeat bit for bit.
//
// Inside a block: one producer thread issues, per tile, a bulk copy of the
// weight tile and one of the activation block for the tile's features into a
// ring of shared-memory stages (mbarrier transaction counts).  The weight
// copies of the first stages are issued before waiting for the previous
// kernel of the stream (weights never depend on it); the activation copies
// after.  Four consumer warps each own two row tiles of 16 channels of the
// 128-channel n-block and walk the tiles in K order: per 32 features a lane
// reads 16 bytes of fp16 activation codes per 8-token column tile (the B
// operands of two mma.m16n8k16) and widens its 16-byte weight chunk into the
// A operands.  After each quantization group: y += scale * P with separately
// rounded fp32 multiply and add, group by group in ascending order.
#pragma once

#include <cuda_runtime.h>

#include "hq_internal.cuh"

namespace hq {

struct GemmArgs {
    const uint8_t *blob;
    const uint8_t *qop;  // activation operand: [K/128][M_total][128 fp16], odd rows swizzled
    const float *sx;     // [M_total]
    float *Y;            // [M_total][N]
    int32_t *partials;   // check mode: [M_total][N][K/G] or NULL
    uint8_t *ws;
    int det;                // 1: split outputs summed in fixed order after a wait; 0: accumulated atomically
    int M_total, m0, M;     // rows of the call, first row of this launch, rows of this launch (<= 32)
    int N, K, NGK, NB, KTILES, T, grid, stages;
    int tile_bytes, code_bytes, scale_bytes, act_bytes;
};

// Accumulating mode: added (with the zeroing block's own arrival, + 1) to a
// split n-block's counter once its outputs are zero; above any count of
// arrivals (at most MAX_CTAS blocks).
constexpr int ZERO_MARK = 1 << 24;

// Weight stages a block copies in before waiting for the previous kernel.
constexpr int PREFETCH_STAGES = 2;

__device__ __forceinline__ int tile_begin(int c, int T, int grid) { return (int)(((long long)c * T) / grid); }
// thread block whose range contains tile t
__device__ __forceinline__ int cta_of_tile(int t, int T, int grid) {
    return (int)((((long long)t + 1) * grid - 1) / T);
}

// 4-bit codes -> fp16 (q - z).  Word layout (nibble i at bits 4i):
// (n0, n4) row g features b, b+1; (n1, n5) row g+8 features b, b+1;
// (n2, n6) row g features b+2, b+3; (n3, n7) row g+8 features b+2, b+3.
// Low nibbles of a half become 1024 + q via the fp16 exponent bits 0x6400;
// nibbles at bits 4..7 of a half become 1024 + 16 q and are scaled by 1/16.
// kA = fp16x2(1024 + z_g), kB = fp16x2(-(64 + z_{g+8})).
__device__ __forceinline__ void widen_w4(uint32_t w, uint32_t kA, uint32_t kB, uint32_t (&A)[4]) {
    const uint32_t w8 = w >> 8;
    const uint32_t x0 = (w & 0x000F000Fu) | 0x64006400u;
    const uint32_t x1 = (w & 0x00F000F0u) | 0x64006400u;
    const uint32_t x2 = (w8 & 0x000F000Fu) | 0x64006400u;
    const uint32_t x3 = (w8 & 0x00F000F0u) | 0x64006400u;
    const uint32_t sixteenth = 0x2C002C00u;  // fp16x2(1/16)
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(A[0]) : "r"(x0), "r"(kA));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(A[1]) : "r"(x1), "r"(sixteenth), "r"(kB));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(A[2]) : "r"(x2), "r"(kA));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(A[3]) : "r"(x3), "r"(sixteenth), "r"(kB));
}

// Four int8 codes -> two fp16x2: bias to unsigned, place under the fp16
// exponent bits 0x64 (1024 + 128 + q), subtract 1152.
__device__ __forceinline__ void widen_i8(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t l, h;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(l) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(h) : "r"(u), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(0x64806480u));
}

// D = A(16x16, fp16) * B(16x8, fp16) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&A)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(A[0]), "r"(A[1]), "r"(A[2]), "r"(A[3]), "r"(b0), "r"(b1));
}
// Same with a zero accumulator input (first step of a group).
__device__ __forceinline__ void mma_f16_16816_z(float (&d)[4], const uint32_t (&A)[4], uint32_t b0, uint32_t b1) {
    const float z = 0.0f;
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(A[0]), "r"(A[1]), "r"(A[2]), "r"(A[3]), "r"(b0), "r"(b1), "f"(z));
}

// (f0, f1) += s * (a0, a1): product rounded, then sum rounded (not fused).
__device__ __forceinline__ void scale_add2(float &f0, float &f1, float a0, float a1, float s) {
    f0 = __fadd_rn(f0, __fmul_rn(s, a0));
    f1 = __fadd_rn(f1, __fmul_rn(s, a1));
}

template <int FMT, int G, int MT>
struct GemmCfg {
    static constexpr int MROWS = 8 * MT;          // activation rows staged per block (zero past M)
    static constexpr int NW = 2;                  // row tiles per consumer warp
    static constexpr int KT = G > 128 ? G : 128;  // features per tile
    static constexpr int STEPS = KT / 32;         // 32-feature steps per tile
    static constexpr int GPT = KT / G;            // groups per tile
    static constexpr int NCW = NTILES / NW;       // consumer warps
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int BLOCKS_PER_SM = 3;  // the launch puts three blocks on each SM
};

// CHECK: also write the exact integer partial sums (check mode).
template <int FMT, int G, int MT, bool CHECK>
__global__ void __launch_bounds__(GemmCfg<FMT, G, MT>::THREADS, GemmCfg<FMT, G, MT>::BLOCKS_PER_SM)
    k_verify_gemm(const GemmArgs a) {
    using C = GemmCfg<FMT, G, MT>;
    constexpr int KT = C::KT, NCW = C::NCW, NW = C::NW;
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = a.stages;
    const int stage_bytes = a.tile_bytes + a.act_bytes;  // shared-memory footprint of a stage
    // bytes that land in a stage: the weight tile and M rows of each 128-feature activation block
    const uint32_t tx_bytes = (uint32_t)a.tile_bytes + (uint32_t)a.M * 256u * (uint32_t)(C::KT / 128);
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)S * stage_bytes);  // full[S], empty[S]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = tile_begin(blockIdx.x, a.T, a.grid);
    const int t1 = tile_begin(blockIdx.x + 1, a.T, a.grid);
    const int ntl = t1 - t0;
    int *err = reinterpret_cast<int *>(a.ws);

    // after the ring barriers, accumulating mode: one flag per split segment
    // of the block, raised by the producer once the n-block's zeroing is
    // visible
    int *sflag = reinterpret_cast<int *>(bars + 2 * S);
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_addr(&bars[i]), 1);
            mbar_init(smem_addr(&bars[S + i]), NCW);
        }
        sflag[0] = sflag[1] = 0;
        fence_mbar_init();
    }
    if (a.M < C::MROWS) {
        // activation rows past M are never copied: keep them zero so the B
        // operand loads need no bounds check
        const int pad = (C::MROWS - a.M) * 256 / 16;
        for (int st = 0; st < S; ++st)
            for (int kk = 0; kk < KT / 128; ++kk) {
                uint4 *dst = reinterpret_cast<uint4 *>(ring + (size_t)st * stage_bytes + a.tile_bytes +
                                                       (size_t)kk * C::MROWS * 256 + (size_t)a.M * 256);
                for (int q = threadIdx.x; q < pad; q += blockDim.x) dst[q] = make_uint4(0u, 0u, 0u, 0u);
            }
    }
    __syncthreads();
    pdl_launch_dependents();

    const bool det = a.det != 0;
    // Accumulating mode: this block holds K tile 0 of n-block zb and another
    // block holds its last K tile -> this block zeroes zb's outputs.
    const int zb = (t1 - 1) / a.KTILES;
    const bool zeroer = !det && ntl > 0 && zb * a.KTILES >= t0 && (zb + 1) * a.KTILES > t1;
    int *ctr = reinterpret_cast<int *>(a.ws + ws_counter_offset());

    if (warp == NCW) {
        // ------------------------------------------------------ producer ---
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            const int KTILES = a.KTILES;
            const int blocks = KT / 128;
            const uint32_t row_bytes = (uint32_t)a.M * 256;  // one 128-feature activation block of this launch
            const uint32_t region_bytes = (uint32_t)C::MROWS * 256;
            // activation blocks of the i-th tile of this thread block -> its stage
            auto copy_acts = [&](int i, int st) {
                const int kb = ((t0 + i) % KTILES) * blocks;
                const uint8_t *src = a.qop + ((size_t)kb * a.M_total + a.m0) * 256;
                const uint32_t dst = smem_addr(ring + (size_t)st * stage_bytes + a.tile_bytes);
                const uint32_t fb = smem_addr(&bars[st]);
                for (int kk = 0; kk < blocks; ++kk)
                    bulk_copy_g2s(dst + kk * region_bytes, src + (size_t)kk * a.M_total * 256, row_bytes, fb, pol_a);
            };
            // Accumulating mode: after the copies of a tile that ends a split
            // segment, count this block into the n-block's counter (acquire),
            // wait until the zeroing mark is in (or the counter was reset,
            // which happens only after the mark), reset the counter if this
            // count completes it, and raise the segment's flag for the
            // consumers (release, CTA scope).  The round trips fall on this
            // thread, which runs stages ahead of the consumers.  The zeroing
            // block's own n-block needs neither: its mark carries its count,
            // and its consumers zeroed before a block barrier.  Every access
            // to a counter is a read-modify-write, so the reset continues the
            // mark's release sequence and a wait that reads it acquires the
            // zeroing.
            int nsplit = 0;
            auto check = [&](int j) {
                const int t = t0 + j, bb = t / KTILES, kb = t - bb * KTILES;
                if (!((kb == KTILES - 1 || j == ntl - 1) && !(bb * KTILES >= t0 && kb == KTILES - 1))) return;
                if (!(zeroer && bb == zb)) {
                    const int nc = cta_of_tile(bb * KTILES + KTILES - 1, a.T, a.grid) -
                                   cta_of_tile(bb * KTILES, a.T, a.grid) + 1;
                    const int v = atom_add_acquire_gpu(&ctr[bb], 1);
                    if (v < ZERO_MARK) wait_mark_bounded(&ctr[bb], ZERO_MARK, v + 1, err);
                    if (v == ZERO_MARK + nc - 1) atomicExch(&ctr[bb], 0);
                }
                st_release_cta_shared(smem_addr(&sflag[nsplit]), 1);
                ++nsplit;
            };
            int i = 0;
            // Weights never depend on earlier kernels of the stream: the first
            // PREFETCH_STAGES stages' weight copies go out before waiting for
            // them.  Not the whole ring: the burst of every block's prefetch
            // delays the previous kernel's memory accesses (an activation
            // kernel reading its input); two stages (8.5 MB over the grid on the
            // W4 G64 decoder layers) made the verify pass 2.9% faster than
            // four, with the same GEMM-only time.
            for (; i < ntl && i < S && i < PREFETCH_STAGES; ++i) {
                const uint32_t fb = smem_addr(&bars[i]);
                mbar_arrive_expect_tx(fb, tx_bytes);
                bulk_copy_g2s(smem_addr(ring + (size_t)i * stage_bytes),
                              a.blob + (size_t)(t0 + i) * (size_t)a.tile_bytes, (uint32_t)a.tile_bytes, fb, pol_w);
            }
            pdl_wait();
            for (int j = 0; j < i; ++j) copy_acts(j, j);
            if (!det)
                for (int j = 0; j < i; ++j) check(j);
            for (; i < ntl; ++i) {
                const int st = i % S;
                const uint32_t ph = (uint32_t)((i / S) & 1);
                if (!mbar_wait_bounded(smem_addr(&bars[S + st]), ph ^ 1u, err)) break;
                const uint32_t fb = smem_addr(&bars[st]);
                mbar_arrive_expect_tx(fb, tx_bytes);
                bulk_copy_g2s(smem_addr(ring + (size_t)st * stage_bytes),
                              a.blob + (size_t)(t0 + i) * (size_t)a.tile_bytes, (uint32_t)a.tile_bytes, fb, pol_w);
                copy_acts(i, st);
                if (!det) check(i);
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
    const int M = a.M, N = a.N, KTILES = a.KTILES;
    float *wsp = reinterpret_cast<float *>(a.ws + ws_partial_offset());
    const float *sxm = a.sx + a.m0;
    float *Ym = a.Y + (size_t)a.m0 * N;
    // byte offsets of this lane's B operand rows (token tt*8 + g8) in a stage
    uint32_t boff[MT];
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) boff[tt] = (uint32_t)(tt * 8 + g8) * 256u;

    float acc[NW][MT][4], acc2[NW][MT][4];
    float facc[NW][MT][4];
    bool ok = true;
    // n-blocks whose partial sums this block published: its first n-block
    // (slot 0) and its last one (slot 1)
    int pend0 = -1, pend1 = -1;
    const int first_b = t0 / KTILES;
    // Accumulating mode: nsplit counts the split segments met so far (the
    // producer raises their flags in the same order).  The zeroing block
    // zeroes zb's outputs, then adds the mark and its own arrival (release);
    // mark_old, the count before it, is read after the last tile.
    int nsplit = 0, mark_old = 0;
    if (zeroer) {
        for (int q = threadIdx.x; q < M * BN; q += NCW * 32) {
            const int tok = q / BN, n = zb * BN + (q - tok * BN);
            if (n < N) Ym[(size_t)tok * N + n] = 0.0f;
        }
        named_barrier(1, NCW * 32);
        if (threadIdx.x == 0) mark_old = atom_add_release_gpu(&ctr[zb], ZERO_MARK + 1);
    }

    // running position: tile t0 + i is n-block b, K tile kt, in stage st of phase ph
    int b = t0 / KTILES, kt = t0 - b * KTILES, st = 0;
    uint32_t ph = 0;
    int seg_k0 = kt;

    // A failed (timed-out) wait is sticky: the warp stops waiting but keeps
    // the same control flow, so every consumer warp still reaches each named
    // barrier and every arrival counter is still incremented and reset.
    for (int i = 0; i < ntl; ++i) {
        if (i == 0 || kt == 0) {
            seg_k0 = kt;
#pragma unroll
            for (int j = 0; j < NW; ++j)
#pragma unroll
                for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) facc[j][tt][e] = 0.0f;
        }
        if (ok) ok = mbar_wait_bounded(smem_addr(&bars[st]), ph, err);
        const uint8_t *tile = ring + (size_t)st * stage_bytes;
        const uint8_t *acts = tile + a.tile_bytes;
        const float *tsc = reinterpret_cast<const float *>(tile + a.code_bytes);
        const uint8_t *tzp = tile + a.code_bytes + a.scale_bytes;

        uint4 wchunk[NW];
        uint32_t kA[NW], kB[NW];  // zero-point constants of the lane's current group (4-bit format)
#pragma unroll
        for (int c = 0; c < C::STEPS; ++c) {
            // B operands: 8 fp16 activation codes of token tt*8 + g8, features c*32 + tig*8 .. +7
            uint4 bq[MT];
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) {
                const uint32_t q = (uint32_t)(((c & 3) * 4 + tig) ^ (((tt * 8 + g8) & 1) << 2));  // swizzled chunk
                bq[tt] = *reinterpret_cast<const uint4 *>(acts + (size_t)(c >> 2) * C::MROWS * 256 + boff[tt] + q * 16);
            }
            // A operands: the lane's 16-byte weight chunk (64 features for 4-bit, 32 for 8-bit)
            if (FMT == HQ_W8_SYM || (c & 1) == 0) {
                const int ch = FMT == HQ_W4_ASYM ? c >> 1 : c;
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    const int nt = warp * NW + j;
                    wchunk[j] = *reinterpret_cast<const uint4 *>(tile + (((size_t)ch * NTILES + nt) * 32 + lane) * 16);
                }
            }
            const bool group_start = G <= 32 || (c * 32) % G == 0;
            if (FMT == HQ_W4_ASYM && group_start) {
                const int gl = G == 16 ? 2 * c + (tig >> 1) : (c * 32) / G;  // group of the lane's features
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    const int nt = warp * NW + j;
                    const uint32_t zb = tzp[((size_t)gl * NTILES + nt) * 8 + g8];
                    kA[j] = (0x6400u | (zb & 15u)) * 0x10001u;
                    kB[j] = (0xD400u | ((zb >> 4) << 4)) * 0x10001u;
                }
            }
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {  // the two 16-feature MMA steps
                uint32_t A[NW][4];
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    if (FMT == HQ_W4_ASYM) {
                        const uint32_t w = (c & 1) ? (s2 ? wchunk[j].w : wchunk[j].z) : (s2 ? wchunk[j].y : wchunk[j].x);
                        widen_w4(w, kA[j], kB[j], A[j]);
                    } else {
                        widen_i8(s2 ? wchunk[j].z : wchunk[j].x, A[j][0], A[j][2]);
                        widen_i8(s2 ? wchunk[j].w : wchunk[j].y, A[j][1], A[j][3]);
                    }
                }
                const bool first = group_start && s2 == 0;
#pragma unroll
                for (int tt = 0; tt < MT; ++tt) {
                    const uint32_t b0 = s2 ? bq[tt].z : bq[tt].x;
                    const uint32_t b1 = s2 ? bq[tt].w : bq[tt].y;
                    if (G == 16) {
                        // two groups per step: lanes tig 0,1 hold the first 16 features
                        const bool lowhalf = tig < 2;
                        const uint32_t l0 = lowhalf ? b0 : 0u, l1 = lowhalf ? b1 : 0u;
                        const uint32_t h0 = lowhalf ? 0u : b0, h1 = lowhalf ? 0u : b1;
#pragma unroll
                        for (int j = 0; j < NW; ++j) {
                            if (first) {
                                mma_f16_16816_z(acc[j][tt], A[j], l0, l1);
                                mma_f16_16816_z(acc2[j][tt], A[j], h0, h1);
                            } else {
                                mma_f16_16816(acc[j][tt], A[j], l0, l1);
                                mma_f16_16816(acc2[j][tt], A[j], h0, h1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < NW; ++j) {
                            if (first)
                                mma_f16_16816_z(acc[j][tt], A[j], b0, b1);
                            else
                                mma_f16_16816(acc[j][tt], A[j], b0, b1);
                        }
                    }
                }
            }
            // end of a group: fold it into the fp32 sums
            auto epilogue = [&](float(&ac)[NW][MT][4], int gl) {
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    const int nt = warp * NW + j;
                    const float2 sc = *reinterpret_cast<const float2 *>(tsc + ((size_t)gl * NTILES + nt) * 16 + 2 * g8);
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt) {
                        scale_add2(facc[j][tt][0], facc[j][tt][1], ac[j][tt][0], ac[j][tt][1], sc.x);
                        scale_add2(facc[j][tt][2], facc[j][tt][3], ac[j][tt][2], ac[j][tt][3], sc.y);
                        if (CHECK) {
                            const int gg = kt * C::GPT + gl;
                            if (gg < a.NGK) {
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int tok = tt * 8 + tig * 2 + (e & 1);
                                    const int n = b * BN + nt * 16 + g8 + 8 * (e >> 1);
                                    if (tok < M && n < N)
                                        a.partials[((size_t)(a.m0 + tok) * N + n) * a.NGK + gg] =
                                            __float2int_rn(ac[j][tt][e]);
                                }
                            }
                        }
                    }
                }
            };
            if (G == 16) {
                epilogue(acc, 2 * c);
                epilogue(acc2, 2 * c + 1);
            } else if (((c + 1) * 32) % G == 0) {
                epilogue(acc, ((c + 1) * 32) / G - 1);
            }
        }
        // release the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bars[S + st]));

        // end of an n-block segment?
        if (kt == KTILES - 1 || i == ntl - 1) {
            if (seg_k0 == 0 && kt == KTILES - 1) {
                // the whole K range of the n-block: write Y
#pragma unroll
                for (int j = 0; j < NW; ++j)
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int row = (warp * NW + j) * 16 + g8 + 8 * (e >> 1);
                            const int tok = tt * 8 + tig * 2 + (e & 1);
                            const int n = b * BN + row;
                            if (tok < M && n < N)
                                Ym[(size_t)tok * N + n] = __fmul_rn(__ldg(sxm + tok), facc[j][tt][e]);
                        }
            } else if (det) {
                // part of the K range: publish the partial sums now, count the
                // arrival once this block's tiles are all done
                const int slot = b == first_b ? 0 : 1;
                float *mys = wsp + ((size_t)blockIdx.x * 2 + slot) * ws_slot_floats();
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
                if (slot == 0)
                    pend0 = b;
                else
                    pend1 = b;
            } else {
                // part of the K range, accumulating mode: once the zeroing is
                // visible (the segment's flag), add sx * (this block's sum) into Y
                if (ok) ok = wait_flag_bounded(smem_addr(&sflag[nsplit]), err);
                ++nsplit;
#pragma unroll
                for (int j = 0; j < NW; ++j)
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int row = (warp * NW + j) * 16 + g8 + 8 * (e >> 1);
                            const int tok = tt * 8 + tig * 2 + (e & 1);
                            const int n = b * BN + row;
                            if (tok < M && n < N)
                                atomicAdd(Ym + (size_t)tok * N + n, __fmul_rn(__ldg(sxm + tok), facc[j][tt][e]));
                        }
            }
        }
        // advance the running position
        if (++st == S) {
            st = 0;
            ph ^= 1u;
        }
        if (++kt == KTILES) {
            kt = 0;
            ++b;
        }
    }

    // Accumulating mode: if every other contributor of zb counted before the
    // mark, the mark completed the count and this block resets the counter.
    if (zeroer && threadIdx.x == 0) {
        const int nc = cta_of_tile(zb * KTILES + KTILES - 1, a.T, a.grid) - cta_of_tile(zb * KTILES, a.T, a.grid) + 1;
        if (mark_old == nc - 1) atomicExch(&ctr[zb], 0);
    }

    // Split n-blocks: every contributor arrives, waits until all contributors
    // of the n-block have arrived, then sums its 1/nc share of the n-block's
    // outputs over all contributors' partial sums in ascending K order (slot 0
    // of a contributor is its first segment, slot 1 its last), multiplies by
    // the row scale and writes Y.  The wait is safe because every thread
    // block of the launch is resident: the grid never exceeds the blocks that
    // fit on the device at once, and dependent kernels are launched only
    // after every block of this one has started.  The last contributor to
    // finish resets the n-block's two counters for the next call.  Threads 0
    // and 1 serve the two pending n-blocks at the same time.
    if (pend0 >= 0 || pend1 >= 0) {
        int *done = ctr + a.NB;
        // every consumer thread's partial-sum stores precede the arrivals
        named_barrier(1, NCW * 32);
        int my_bb = -1, my_nc = 0, done_before = 0;
        if (threadIdx.x < 2) {
            my_bb = threadIdx.x == 0 ? pend0 : pend1;
            if (my_bb >= 0) {
                my_nc = cta_of_tile(my_bb * KTILES + KTILES - 1, a.T, a.grid) -
                        cta_of_tile(my_bb * KTILES, a.T, a.grid) + 1;
                red_add_release_gpu(&ctr[my_bb], 1);
                if (ok) ok = wait_count_bounded(&ctr[my_bb], my_nc, err);
                // passed the wait: count it now, the answer arrives during the sums
                done_before = atomicAdd(&done[my_bb], 1);
            }
        }
        // the acquires of threads 0 and 1 are ordered before every thread's loads below
        named_barrier(1, NCW * 32);
        // Shares of both pending n-blocks as one list of 4-channel output
        // groups (n0 from the first, then the second); two groups per
        // iteration, with all their loads in flight together.
        const int total = M * (BN / 4);
        int e_lo[2], e_cnt[2], e_clo[2], e_chi[2], e_slot[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int bb = p == 0 ? pend0 : pend1;
            e_cnt[p] = 0;
            e_lo[p] = e_clo[p] = e_chi[p] = e_slot[p] = 0;
            if (bb < 0) continue;
            const int c_lo = cta_of_tile(bb * KTILES, a.T, a.grid);
            const int c_hi = cta_of_tile(bb * KTILES + KTILES - 1, a.T, a.grid);
            const int nc = c_hi - c_lo + 1;
            const int per = (total + nc - 1) / nc;
            const int lo = (blockIdx.x - c_lo) * per;
            const int hi = lo + per < total ? lo + per : total;
            e_lo[p] = lo;
            e_cnt[p] = hi > lo ? hi - lo : 0;
            e_clo[p] = c_lo;
            e_chi[p] = c_hi;
            // Every contributor after the first starts inside this n-block, so
            // it is their first n-block (slot 0); the first contributor used
            // slot 1 if it started in an earlier n-block.
            e_slot[p] = tile_begin(c_lo, a.T, a.grid) < bb * KTILES ? 1 : 0;
        }
        const int n_all = e_cnt[0] + e_cnt[1];
        for (int base = 0; base < n_all; base += 2 * NCW * 32) {
            float4 sum[2];
            int gis[2], ps[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int idx = base + h * NCW * 32 + (int)threadIdx.x;
                ps[h] = idx < e_cnt[0] ? 0 : (idx < n_all ? 1 : -1);
                gis[h] = ps[h] == 0 ? e_lo[0] + idx : (ps[h] == 1 ? e_lo[1] + idx - e_cnt[0] : 0);
                sum[h] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            const int span = (ps[0] >= 0 ? e_chi[ps[0]] - e_clo[ps[0]] + 1 : 0) >
                                     (ps[1] >= 0 ? e_chi[ps[1]] - e_clo[ps[1]] + 1 : 0)
                                 ? (ps[0] >= 0 ? e_chi[ps[0]] - e_clo[ps[0]] + 1 : 0)
                                 : (ps[1] >= 0 ? e_chi[ps[1]] - e_clo[ps[1]] + 1 : 0);
            // up to 8 contributors of each group in flight, added in contributor order
            for (int cc = 0; cc < span; cc += 8) {
                float4 x[2][8];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int p = ps[h];
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        if (p < 0) continue;
                        const int c2 = e_clo[p] + cc + v;
                        const int sl = cc + v == 0 ? e_slot[p] : 0;
                        if (c2 <= e_chi[p])
                            x[h][v] = __ldcg(reinterpret_cast<const float4 *>(
                                wsp + ((size_t)c2 * 2 + sl) * ws_slot_floats() + (size_t)gis[h] * 4));
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int p = ps[h];
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        if (p < 0 || e_clo[p] + cc + v > e_chi[p]) continue;
                        sum[h].x = __fadd_rn(sum[h].x, x[h][v].x);
                        sum[h].y = __fadd_rn(sum[h].y, x[h][v].y);
                        sum[h].z = __fadd_rn(sum[h].z, x[h][v].z);
                        sum[h].w = __fadd_rn(sum[h].w, x[h][v].w);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (ps[h] < 0) continue;
                const int bb = ps[h] == 0 ? pend0 : pend1;
                const int gi = gis[h];
                const int tok = gi / (BN / 4), r4 = (gi - tok * (BN / 4)) * 4;
                const float sxt = __ldg(sxm + tok);
                const int n = bb * BN + r4;
                float *yr = Ym + (size_t)tok * N;
                if (n + 0 < N) yr[n + 0] = __fmul_rn(sxt, sum[h].x);
                if (n + 1 < N) yr[n + 1] = __fmul_rn(sxt, sum[h].y);
                if (n + 2 < N) yr[n + 2] = __fmul_rn(sxt, sum[h].z);
                if (n + 3 < N) yr[n + 3] = __fmul_rn(sxt, sum[h].w);
            }
        }
        // every contributor has passed its wait once all have counted
        if (my_bb >= 0 && done_before == my_nc - 1) {
            atomicExch(&ctr[my_bb], 0);
            atomicExch(&done[my_bb], 0);
        }
    }
}

// Launch one instance.  Dynamic shared memory: the stage ring, 2*S mbarriers
// and the accumulating mode's two segment flags.
template <int FMT, int G, int MT, bool CHECK>
cudaError_t launch_gemm_instance(const GemmArgs &a, bool pdl, cudaStream_t s) {
    using C = GemmCfg<FMT, G, MT>;
    auto kern = k_verify_gemm<FMT, G, MT, CHECK>;
    const size_t smem = (size_t)a.stages * (size_t)(a.tile_bytes + a.act_bytes) + (size_t)a.stages * 16 + 16;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<int> configured[CACHE_DEVICES];
    int done = 0;
    e = cached_per_device(configured, dev, &done, [&](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    });
    if (e != cudaSuccess) return e;
    // The split-K reduction makes blocks wait for one another: the grid must
    // never exceed the blocks that are resident at once.
    static std::atomic<int> resident[CACHE_DEVICES];
    int resident_blocks = 0;
    e = cached_per_device(resident, dev, &resident_blocks, [&](int *v) {
        int per_sm = 0;
        const cudaError_t r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::THREADS, smem);
        *v = per_sm * device_sm_count();
        return r;
    });
    if (e != cudaSuccess) return e;
    if (resident_blocks < 1) return cudaErrorLaunchOutOfResources;
    GemmArgs la = a;
    if (la.grid > resident_blocks) la.grid = resident_blocks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)la.grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, la);
}

// Instances for one format: token buckets {<=8, <=16, <=32} per launch.
template <int FMT, int G>
cudaError_t launch_gemm_g(const GemmArgs &a, bool pdl, cudaStream_t s) {
    if (a.partials) {
        if (a.M <= 8) return launch_gemm_instance<FMT, G, 1, true>(a, pdl, s);
        if (a.M <= 16) return launch_gemm_instance<FMT, G, 2, true>(a, pdl, s);
        return launch_gemm_instance<FMT, G, 4, true>(a, pdl, s);
    }
    if (a.M <= 8) return launch_gemm_instance<FMT, G, 1, false>(a, pdl, s);
    if (a.M <= 16) return launch_gemm_instance<FMT, G, 2, false>(a, pdl, s);
    return launch_gemm_instance<FMT, G, 4, false>(a, pdl, s);
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
