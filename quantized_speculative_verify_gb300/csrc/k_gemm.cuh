// k_gemm.cuh -- the verify GEMM on fifth-generation tensor cores: activation
// codes x packed 4-/8-bit weights, exact per-group integer partial sums in
// tensor memory, fp32 dequantization epilogue in the oracle's group order.
//
// Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling":
// section "How Uzu optimizes bytes and tokens per pass" (both operands of the
// verify matmul are integers; Medium weights are 4-bit asymmetric, Large 8-bit
// symmetric, grouped along K) and section "Why batch-one decoding is
// memory-bound" (the pass streams every weight once, so the kernel is bound by
// memory bandwidth, not arithmetic).
//
// Integer arithmetic on fp16 tensor cores.  The integer MMA of this GPU is
// far slower than its fp16 MMA, so the contraction runs as an exact fp16
// tcgen05.mma with fp32 accumulation in tensor memory (TMEM):
//  - 8-bit codes q (|q| <= 127) are widened to fp16 q exactly (magic-number
//    conversion: (1152 + q) - 1152);
//  - 4-bit codes q are widened to fp16 64 + q (the nibble placed under the
//    exponent of 64, whose ulp is 1/16: two bitwise operations for two codes),
//    and the zero point z is applied after the MMA through the group sums of
//    the activation codes, S = sum_{k in g} qx[k]:
//        P = sum qx (q - z) = sum qx (64 + q) - (64 + z) S
//    (the Medium identity of the method); |sum qx (64 + q)| <= 127 * 79 * 256
//    < 2^24, so every partial sum is an exact fp32 integer and one fused
//    multiply-add gives P exactly.
// Activation codes (fp16, exact) are the B operand in shared memory, the
// widened weights the A operand in TMEM (128 channels = 128 TMEM lanes), and
// each quantization group's P lands in its own TMEM accumulator slot.
//
// Epilogue: y += scale * P with separately rounded fp32 multiply and add, in
// ascending group order, so an output whose whole K range is handled by one
// thread block is bit-identical to the oracle's sequential sum.  (The packed
// f32x2 multiply and add are not used there: the compiler contracts the pair
// into a fused multiply-add, which rounds once.)
//
// Thread block (one per SM, 14 warps, each role running tiles ahead of the
// next through rings of shared-memory stages, A buffers and accumulator
// slots):
//  - warp 0, one lane: producer.  Per tile, one bulk copy of the weight tile,
//    one of the activation blocks and one of their group sums into a stage
//    (mbarrier transaction counts).  The weight copies of the first stages go
//    out before waiting for the previous kernel of the stream; the activation
//    copies after.
//  - warp 1: tensor-memory owner and MMA issuer (one elected lane).  Per
//    group: wait for a free accumulator slot, issue group/16 MMAs (K = 16
//    each) from one unrolled sequence, commit to the slot's "full" barrier.
//  - warps 2..5: widening.  Warp w owns TMEM lanes 32 (w % 4) .. + 31 (= the
//    tile's channels); each thread widens its channel's codes of the whole
//    tile into the tile's A buffer (tcgen05.st).
//  - warps 6..13: epilogue.  Same lanes, and half h = (w - 6) / 4 of the
//    tokens: fold each group out of its accumulator slot (tcgen05.ld) into the
//    running fp32 sums, and write, add or publish them at the end of a
//    128-channel block's segment.
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
#pragma once

#include <cuda_runtime.h>

#include "hq_internal.cuh"
#include "hq_tc.cuh"

namespace hq {

struct GemmArgs {
    const uint8_t *blob;
    const uint8_t *qop;  // activation operand (layout in hq_internal.cuh)
    const float *sx;     // [M]
    float *Y;            // [M][N]
    int32_t *partials;   // check mode: [M][N][K/G] or NULL
    uint8_t *ws;
    int det;  // 1: split outputs summed in fixed order after a wait; 0: accumulated atomically
    int nb_align;  // 1: block ranges start at n-block boundaries (no output is split between blocks)
    int wait_extra;  // self-test only: the deterministic wait asks for this many arrivals more than exist
    long long wait_ns;  // bound of the waits between thread blocks
    int M;    // token rows (the operand is padded to MT rows)
    int N, K, G, KT, GPT, NGK, NB, KTILES, T, grid, stages, na, nd;
    int tile_bytes, code_bytes, scale_bytes;
    int act_off;     // offset of the activation blocks within a stage
    int act_bytes;   // activation blocks per stage: (KT/128) * MT * 256
    int s_bytes;     // group sums per stage: GPT * MT * 4
    int stage_bytes;
    long long op_s_offset;  // byte offset of the group sums in the operand
};

// Accumulating mode: added (with the zeroing block's own arrival, + 1) to a
// split n-block's counter once its outputs are zero; above any count of
// arrivals (at most MAX_CTAS blocks).
constexpr int ZERO_MARK = 1 << 24;

// Weight stages a block copies in before waiting for the previous kernel.
constexpr int PREFETCH_STAGES = 2;

// Back-off of the waits of the roles that are not on the MMA warp's critical
// path (producer, widening, epilogue): their polling would otherwise take
// issue slots from the MMA warp on the same scheduler.
#ifndef HQ_WAIT_SLEEP_NS
#define HQ_WAIT_SLEEP_NS 64
#endif
constexpr uint32_t WAIT_SLEEP_NS = HQ_WAIT_SLEEP_NS;

constexpr int NWID = 4;                       // widening warps
constexpr int NEPI = 8;                       // epilogue warps
constexpr int WID0 = 2, EPI0 = WID0 + NWID;   // first warp of each role
constexpr int GEMM_THREADS = (EPI0 + NEPI) * 32;
constexpr int TMEM_COLS = 512;                // one block per SM owns all of TMEM
constexpr int MAX_NA = 4;                     // A buffers (widened weight tiles) in TMEM
constexpr int MAX_ND = 16;                    // accumulator slots in TMEM
constexpr int MAX_STAGES = 32;
// Every block asks for at least this much shared memory, so that no two
// blocks of the kernel share an SM (each takes all of its TMEM).
constexpr int MIN_GEMM_SMEM = 120 * 1024;
constexpr int GEMM_SMEM_LIMIT = 227 * 1024;   // opt-in maximum of dynamic shared memory per block

__device__ __forceinline__ int tile_begin(int c, int T, int grid) { return (int)(((long long)c * T) / grid); }
// first tile of thread block c (c = grid: one past the last tile)
__device__ __forceinline__ int range_begin(const GemmArgs &a, int c) {
    return a.nb_align ? (int)(((long long)c * a.NB) / a.grid) * a.KTILES : tile_begin(c, a.T, a.grid);
}
// thread block whose range contains tile t
__device__ __forceinline__ int cta_of_tile(int t, int T, int grid) {
    return (int)((((long long)t + 1) * grid - 1) / T);
}

// Eight 4-bit codes -> four fp16x2 (64 + q).  Nibble i of w holds feature
// 2 * (i & 3) + (i >> 2) of an 8-feature run, so that the four results are
// the features (0,1) (2,3) (4,5) (6,7): a code at bits 4..7 of a 16-bit half
// under the exponent bits 0x5400 (fp16 64, ulp 1/16) reads 64 + q.
__device__ __forceinline__ void widen_w4(uint32_t w, uint32_t *o) {
    constexpr uint32_t M4 = 0x00F000F0u, E64 = 0x54005400u;
    o[0] = ((w << 4) & M4) | E64;
    o[1] = (w & M4) | E64;
    o[2] = ((w >> 4) & M4) | E64;
    o[3] = ((w >> 8) & M4) | E64;
}

// Four int8 codes -> two fp16x2 q: bias to unsigned, place under the fp16
// exponent bits 0x64 (1024 + 128 + q), subtract 1152.
__device__ __forceinline__ void widen_i8(uint32_t w, uint32_t *o) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t l, h;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(l) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(h) : "r"(u), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[0]) : "r"(l), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[1]) : "r"(h), "r"(0x64806480u));
}

// Position in a ring of n slots: slot index and the parity of its current
// phase, advanced without divisions.
struct RingPos {
    int slot;
    uint32_t phase;
    __device__ __forceinline__ void next(int n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// The KS MMAs (K = 16 each) of one quantization group, from one unrolled
// sequence: A advances 8 TMEM columns per step, B 32 * MT bytes (two core
// matrices of 8 features x MT rows).
template <int KS, int MT>
__device__ __forceinline__ void issue_group(uint32_t d_tm, uint32_t a_tm, uint64_t bdesc, uint32_t idesc) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
        tc_mma_f16_ts(d_tm, a_tm + (uint32_t)(ks * 8), bdesc + (uint64_t)((ks * 32 * MT) >> 4), idesc, ks > 0 ? 1u : 0u);
}

template <int MH>
__device__ __forceinline__ void tmem_ld_tokens(uint32_t taddr, float *v) {
    if constexpr (MH == 8) {
        tmem_ld8(taddr, v);
    } else if constexpr (MH == 16) {
        tmem_ld16(taddr, v);
    } else if constexpr (MH == 32) {
        tmem_ld32(taddr, v);
    } else {
        tmem_ld32(taddr, v);
        tmem_ld32(taddr + 32, v + 32);
    }
}

// CHECK: also write the exact integer partial sums (check mode).
template <int FMT, int MT, bool CHECK>
__global__ void __launch_bounds__(GEMM_THREADS, 1) k_verify_gemm(const GemmArgs a) {
    constexpr int MH = MT / 2;          // tokens per epilogue thread
    constexpr int CH = MH < 32 ? MH : 32;  // tokens per tensor-memory load
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int S = a.stages, NA = a.na, ND = a.nd;
    const int KT = a.KT, GPT = a.GPT, G = a.G;
    const int KSTEPS_G = G / 16;  // MMAs per group
    // barriers and flags first, the stage ring after
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw);
    uint64_t *empty = full + MAX_STAGES;
    uint64_t *a_full = empty + MAX_STAGES;
    uint64_t *a_empty = a_full + MAX_NA;
    uint64_t *d_full = a_empty + MAX_NA;
    uint64_t *d_empty = d_full + MAX_ND;
    uint64_t *done_bar = d_empty + MAX_ND;
    int *sflag = reinterpret_cast<int *>(done_bar + 1);  // accumulating mode: two segment flags
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sflag + 2);
    uint8_t *ring = smem_raw + 2048;

    // warp index made visibly warp-uniform (tensor-memory addresses derive from it)
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    const int t0 = range_begin(a, blockIdx.x);
    const int t1 = range_begin(a, blockIdx.x + 1);
    const int ntl = t1 - t0;
    int *err = reinterpret_cast<int *>(a.ws);
    const uint32_t tx_bytes = (uint32_t)(a.tile_bytes + a.act_bytes + a.s_bytes);

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            // widening warps + epilogue warps + the MMAs' commit
            mbar_init(smem_addr(&empty[i]), NWID + NEPI + 1);
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(smem_addr(&a_full[i]), NWID);
            mbar_init(smem_addr(&a_empty[i]), 1);
        }
        for (int i = 0; i < ND; ++i) {
            mbar_init(smem_addr(&d_full[i]), 1);
            mbar_init(smem_addr(&d_empty[i]), NEPI);
        }
        mbar_init(smem_addr(done_bar), 1);
        sflag[0] = sflag[1] = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    pdl_launch_dependents();

    const bool det = a.det != 0;
    const int KTILES = a.KTILES;
    // Accumulating mode: this block holds K tile 0 of n-block zb and another
    // block holds its last K tile -> this block zeroes zb's outputs.
    const int zb = (t1 - 1) / KTILES;
    const bool zeroer = !det && ntl > 0 && zb * KTILES >= t0 && (zb + 1) * KTILES > t1;
    int *ctr = reinterpret_cast<int *>(a.ws + ws_counter_offset());
    const int acols = KT / 2;          // TMEM columns of one A buffer
    const int dcol0 = NA * acols;      // first accumulator column
    const int quarter = warp & 3;      // TMEM lanes 32 * quarter .. (widening and epilogue warps)
    const int n = quarter * 32 + lane; // channel within the tile
    const uint32_t lane_field = (uint32_t)(quarter * 32) << 16;

    if (warp == 0) {
        // ------------------------------------------------------ producer ---
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            auto copy_acts = [&](int i, int st) {
                const int kt = (t0 + i) % KTILES;
                uint8_t *stage = ring + (size_t)st * a.stage_bytes;
                const uint32_t fb = smem_addr(&full[st]);
                bulk_copy_g2s(smem_addr(stage + a.act_off), a.qop + (size_t)kt * a.act_bytes, (uint32_t)a.act_bytes,
                              fb, pol_a);
                bulk_copy_g2s(smem_addr(stage + a.act_off + a.act_bytes),
                              a.qop + a.op_s_offset + (size_t)kt * a.s_bytes, (uint32_t)a.s_bytes, fb, pol_a);
            };
            // Accumulating mode: after the copies of a tile that ends a split
            // segment, count this block into the n-block's counter (acquire),
            // wait until the zeroing mark is in (or the counter was reset,
            // which happens only after the mark), reset the counter if this
            // count completes it, and raise the segment's flag for the
            // epilogue warps (release, CTA scope).  The zeroing block's own
            // n-block needs neither: its mark carries its count, and its
            // epilogue warps zeroed before a barrier.  Every access to a
            // counter is a read-modify-write, so the reset continues the
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
                    if (v < ZERO_MARK) wait_mark_bounded(&ctr[bb], ZERO_MARK, v + 1, err, a.wait_ns);
                    if (v == ZERO_MARK + nc - 1) atomicExch(&ctr[bb], 0);
                }
                st_release_cta_shared(smem_addr(&sflag[nsplit]), 1);
                ++nsplit;
            };
            int i = 0;
            for (; i < ntl && i < S && i < PREFETCH_STAGES; ++i) {
                const uint32_t fb = smem_addr(&full[i]);
                mbar_arrive_expect_tx(fb, tx_bytes);
                bulk_copy_g2s(smem_addr(ring + (size_t)i * a.stage_bytes),
                              a.blob + (size_t)(t0 + i) * (size_t)a.tile_bytes, (uint32_t)a.tile_bytes, fb, pol_w);
            }
            pdl_wait();
            for (int j = 0; j < i; ++j) copy_acts(j, j);
            if (!det)
                for (int j = 0; j < i; ++j) check(j);
            RingPos ps{i % S, (uint32_t)((i / S) & 1)};
            for (; i < ntl; ++i) {
                const int st = ps.slot;
                if (!mbar_wait_sleep(smem_addr(&empty[st]), ps.phase ^ 1u, err, WAIT_SLEEP_NS)) break;
                const uint32_t fb = smem_addr(&full[st]);
                mbar_arrive_expect_tx(fb, tx_bytes);
                bulk_copy_g2s(smem_addr(ring + (size_t)st * a.stage_bytes),
                              a.blob + (size_t)(t0 + i) * (size_t)a.tile_bytes, (uint32_t)a.tile_bytes, fb, pol_w);
                copy_acts(i, st);
                if (!det) check(i);
                ps.next(S);
            }
            // No copy may still be landing in shared memory when the block exits.
            const int issued = i;
            for (int j = issued > S ? issued - S : 0; j < issued; ++j)
                mbar_wait_bounded(smem_addr(&full[j % S]), (uint32_t)((j / S) & 1), err);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer ---
        const uint32_t idesc = tc_idesc_f16(128, MT);
        // descriptor of the first stage's activation blocks; stage st adds
        // st * stage_bytes (the start address field counts 16-byte units)
        const uint64_t bdesc_ring = tc_smem_desc(smem_addr(ring + a.act_off), 16u * MT, 128u);
        const uint32_t stage_units = (uint32_t)(a.stage_bytes >> 4);
        // One elected lane waits and issues; the other lanes only keep the
        // warp's ring positions in step.
        bool ok = true;
        RingPos ps{0, 0u}, pa{0, 0u}, pd{0, 0u};
        for (int i = 0; i < ntl; ++i) {
            const uint32_t a_tm = tbase + (uint32_t)(pa.slot * acols);
            const uint64_t bdesc = bdesc_ring + (uint64_t)(ps.slot * stage_units);
            __syncwarp();
            if (elect_one()) {
                if (ok) ok = mbar_wait_bounded(smem_addr(&full[ps.slot]), ps.phase, err);
                if (ok) ok = mbar_wait_bounded(smem_addr(&a_full[pa.slot]), pa.phase, err);
                RingPos pg = pd;
                for (int gl = 0; gl < GPT; ++gl) {
                    if (ok) ok = mbar_wait_bounded(smem_addr(&d_empty[pg.slot]), pg.phase ^ 1u, err);
                    tc_fence_after();
                    const uint32_t d_tm = tbase + (uint32_t)(dcol0 + pg.slot * MT);
                    const uint32_t a_g = a_tm + (uint32_t)(gl * KSTEPS_G * 8);
                    const uint64_t b_g = bdesc + (uint64_t)((gl * KSTEPS_G * 32 * MT) >> 4);
                    switch (KSTEPS_G) {
                        case 1: issue_group<1, MT>(d_tm, a_g, b_g, idesc); break;
                        case 2: issue_group<2, MT>(d_tm, a_g, b_g, idesc); break;
                        case 4: issue_group<4, MT>(d_tm, a_g, b_g, idesc); break;
                        case 8: issue_group<8, MT>(d_tm, a_g, b_g, idesc); break;
                        default: issue_group<16, MT>(d_tm, a_g, b_g, idesc); break;
                    }
                    tc_commit(smem_addr(&d_full[pg.slot]));
                    pg.next(ND);
                }
                tc_commit(smem_addr(&a_empty[pa.slot]));
                tc_commit(smem_addr(&empty[ps.slot]));
            }
            __syncwarp();
            for (int gl = 0; gl < GPT; ++gl) pd.next(ND);
            ps.next(S);
            pa.next(NA);
        }
        // every MMA has completed before the block frees TMEM
        __syncwarp();
        if (elect_one()) tc_commit(smem_addr(done_bar));
        __syncwarp();
        mbar_wait_bounded(smem_addr(done_bar), 0u, err);
    } else if (warp < EPI0) {
        // ----------------------------------------------------- widening ---
        const int KC = KT / 64;  // 64-feature chunks per tile
        bool ok = true;
        RingPos ps{0, 0u}, pa{0, 0u};
        for (int i = 0; i < ntl; ++i) {
            const int st = ps.slot, ab = pa.slot;
            if (ok) ok = mbar_wait_sleep(smem_addr(&full[st]), ps.phase, err, WAIT_SLEEP_NS);
            if (ok) ok = mbar_wait_sleep(smem_addr(&a_empty[ab]), pa.phase ^ 1u, err, WAIT_SLEEP_NS);
            __syncwarp();
            tc_fence_after();
            const uint8_t *tile = ring + (size_t)st * a.stage_bytes;
            for (int c = 0; c < KC; ++c) {
                uint32_t v[32];
                if (FMT == HQ_W4_ASYM) {
                    uint4 u[2];
#pragma unroll
                    for (int p = 0; p < 2; ++p)
                        u[p] = *reinterpret_cast<const uint4 *>(tile + ((size_t)(c * 2 + p) * BN + n) * 16);
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        widen_w4(u[p].x, v + 16 * p + 0);
                        widen_w4(u[p].y, v + 16 * p + 4);
                        widen_w4(u[p].z, v + 16 * p + 8);
                        widen_w4(u[p].w, v + 16 * p + 12);
                    }
                } else {
                    uint4 u[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        u[p] = *reinterpret_cast<const uint4 *>(tile + ((size_t)(c * 4 + p) * BN + n) * 16);
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        widen_i8(u[p].x, v + 8 * p + 0);
                        widen_i8(u[p].y, v + 8 * p + 2);
                        widen_i8(u[p].z, v + 8 * p + 4);
                        widen_i8(u[p].w, v + 8 * p + 6);
                    }
                }
                tmem_st32(tbase + lane_field + (uint32_t)(ab * acols + c * 32), v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_addr(&a_full[ab]));
                mbar_arrive(smem_addr(&empty[st]));  // this warp no longer reads the stage
            }
            ps.next(S);
            pa.next(NA);
        }
    } else {
        // ----------------------------------------------------- epilogue ---
        pdl_wait();
        const int mt = threadIdx.x - EPI0 * 32;  // epilogue thread 0..255
        const int h = (warp - EPI0) >> 2;        // token half
        const int M = a.M, N = a.N;
        float *wsp = reinterpret_cast<float *>(a.ws + ws_partial_offset());

        float y[MH];
        bool ok = true;
        int pend0 = -1, pend1 = -1;
        const int first_b = t0 / KTILES;
        int nsplit = 0, mark_old = 0;
        if (zeroer) {
            for (int q = mt; q < M * BN; q += NEPI * 32) {
                const int tok = q / BN, nn = zb * BN + (q - tok * BN);
                if (nn < N) a.Y[(size_t)tok * N + nn] = 0.0f;
            }
            named_barrier(1, NEPI * 32);
            if (mt == 0) mark_old = atom_add_release_gpu(&ctr[zb], ZERO_MARK + 1);
        }

        RingPos ps{0, 0u}, pd{0, 0u};
        // position of the tile being folded: n-block eb, K tile ekt
        int eb = t0 / KTILES, ekt = t0 - eb * KTILES, seg_k0 = ekt;
        for (int i = 0; i < ntl; ++i) {
            const int st = ps.slot;
            if (i == 0 || ekt == 0) {
                seg_k0 = ekt;
#pragma unroll
                for (int t = 0; t < MH; ++t) y[t] = 0.0f;
            }
            // the stage's scales, zero points and group sums are read below
            if (ok) ok = mbar_wait_sleep(smem_addr(&full[st]), ps.phase, err, WAIT_SLEEP_NS);
            const uint8_t *tile = ring + (size_t)st * a.stage_bytes;
            const float *tsc = reinterpret_cast<const float *>(tile + a.code_bytes) + (size_t)n * GPT;
            const uint8_t *tzp = tile + a.code_bytes + a.scale_bytes;
            const float *tS = reinterpret_cast<const float *>(tile + a.act_off + a.act_bytes);
            for (int gl = 0; gl < GPT; ++gl) {
                const int slot = pd.slot;
                if (ok) ok = mbar_wait_sleep(smem_addr(&d_full[slot]), pd.phase, err, WAIT_SLEEP_NS);
                __syncwarp();
                tc_fence_after();
                const float sc = tsc[gl];
                float nz = 0.0f;
                if (FMT == HQ_W4_ASYM) {
                    const int zi = n * GPT + gl;
                    const uint32_t zb8 = tzp[zi >> 1];
                    nz = -(float)(64u + ((zi & 1) ? (zb8 >> 4) : (zb8 & 15u)));
                }
                const f2 nz2 = f2_make(nz, nz);
                const float *Sg = tS + gl * MT + h * MH;
#pragma unroll
                for (int c0 = 0; c0 < MH; c0 += CH) {
                    float acc[CH];
                    const uint32_t taddr = tbase + lane_field + (uint32_t)(dcol0 + slot * MT + h * MH + c0);
                    if constexpr (CH == 8)
                        tmem_ld8(taddr, acc);
                    else if constexpr (CH == 16)
                        tmem_ld16(taddr, acc);
                    else
                        tmem_ld32(taddr, acc);
                    tmem_wait_ld();
#pragma unroll
                    for (int p = 0; p < CH / 2; ++p) {
                        float p0 = acc[2 * p], p1 = acc[2 * p + 1];
                        if (FMT == HQ_W4_ASYM) {
                            // exact: P = sum qx (64 + q) - (64 + z) S, integers below 2^24
                            const float2 sv = *reinterpret_cast<const float2 *>(Sg + c0 + 2 * p);
                            f2_split(f2_fma(nz2, f2_make(sv.x, sv.y), f2_make(p0, p1)), p0, p1);
                        }
                        const int tok = h * MH + c0 + 2 * p;
                        if (CHECK) {
                            const int gg = ekt * GPT + gl;
                            const int nn = eb * BN + n;
                            if (gg < a.NGK && nn < N) {
                                if (tok < M) a.partials[((size_t)tok * N + nn) * a.NGK + gg] = __float2int_rn(p0);
                                if (tok + 1 < M) a.partials[((size_t)(tok + 1) * N + nn) * a.NGK + gg] = __float2int_rn(p1);
                            }
                        }
                        // y += scale * P: product rounded, then sum rounded
                        y[c0 + 2 * p] = __fadd_rn(y[c0 + 2 * p], __fmul_rn(sc, p0));
                        y[c0 + 2 * p + 1] = __fadd_rn(y[c0 + 2 * p + 1], __fmul_rn(sc, p1));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&d_empty[slot]));
                pd.next(ND);
            }
            // this warp no longer reads the stage
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty[st]));

            // end of an n-block segment?
            if (ekt == KTILES - 1 || i == ntl - 1) {
                const int nn = eb * BN + n;
                if (seg_k0 == 0 && ekt == KTILES - 1) {
                    // the whole K range of the n-block: write Y
#pragma unroll
                    for (int t = 0; t < MH; ++t) {
                        const int tok = h * MH + t;
                        if (tok < M && nn < N) a.Y[(size_t)tok * N + nn] = __fmul_rn(__ldg(a.sx + tok), y[t]);
                    }
                } else if (det) {
                    // part of the K range: publish the partial sums now, count
                    // the arrival once this block's tiles are all done
                    const int slot = eb == first_b ? 0 : 1;
                    float *mys = wsp + ((size_t)blockIdx.x * 2 + slot) * ws_slot_floats();
#pragma unroll
                    for (int t = 0; t < MH; ++t) {
                        const int tok = h * MH + t;
                        if (tok < M) __stcg(mys + (size_t)tok * BN + n, y[t]);
                    }
                    if (slot == 0)
                        pend0 = eb;
                    else
                        pend1 = eb;
                } else {
                    // part of the K range, accumulating mode: once the zeroing
                    // is visible (the segment's flag), add sx * (this block's
                    // sum) into Y
                    if (ok) ok = wait_flag_bounded(smem_addr(&sflag[nsplit]), err);
                    ++nsplit;
#pragma unroll
                    for (int t = 0; t < MH; ++t) {
                        const int tok = h * MH + t;
                        if (tok < M && nn < N) atomicAdd(a.Y + (size_t)tok * N + nn, __fmul_rn(__ldg(a.sx + tok), y[t]));
                    }
                }
            }
            if (++ekt == KTILES) {
                ekt = 0;
                ++eb;
            }
            ps.next(S);
        }

        // Accumulating mode: if every other contributor of zb counted before
        // the mark, the mark completed the count and this block resets the
        // counter.
        if (zeroer && mt == 0) {
            const int nc = cta_of_tile(zb * KTILES + KTILES - 1, a.T, a.grid) - cta_of_tile(zb * KTILES, a.T, a.grid) + 1;
            if (mark_old == nc - 1) atomicExch(&ctr[zb], 0);
        }
        // Split n-blocks, deterministic mode: every contributor arrives,
        // waits until all contributors of the n-block have arrived, then sums
        // its 1/nc share of the n-block's outputs over all contributors'
        // partial sums in ascending K order (slot 0 of a contributor is its
        // first segment, slot 1 its last), multiplies by the row scale and
        // writes Y.  The wait is safe because every thread block of the launch
        // is resident: the grid never exceeds the SMs (one block per SM), and
        // dependent kernels are launched only after every block of this one
        // has started.  The last contributor to finish resets the n-block's
        // two counters for the next call.  Threads 0 and 1 of the epilogue warps
        // serve the two pending n-blocks at the same time.
        if (pend0 >= 0 || pend1 >= 0) {
            int *done = ctr + a.NB;
            // every epilogue thread's partial-sum stores precede the arrivals
            named_barrier(1, NEPI * 32);
            int my_bb = -1, my_nc = 0, done_before = 0;
            if (mt < 2) {
                my_bb = mt == 0 ? pend0 : pend1;
                if (my_bb >= 0) {
                    my_nc = cta_of_tile(my_bb * KTILES + KTILES - 1, a.T, a.grid) -
                            cta_of_tile(my_bb * KTILES, a.T, a.grid) + 1;
                    red_add_release_gpu(&ctr[my_bb], 1);
                    if (ok) ok = wait_count_bounded(&ctr[my_bb], my_nc + a.wait_extra, err, a.wait_ns);
                    // passed the wait: count it now, the answer arrives during the sums
                    done_before = atomicAdd(&done[my_bb], 1);
                }
            }
            // the acquires of threads 0 and 1 are ordered before every thread's loads below
            named_barrier(1, NEPI * 32);
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
                // Every contributor after the first starts inside this n-block,
                // so it is their first n-block (slot 0); the first contributor
                // used slot 1 if it started in an earlier n-block.
                e_slot[p] = tile_begin(c_lo, a.T, a.grid) < bb * KTILES ? 1 : 0;
            }
            const int n_all = e_cnt[0] + e_cnt[1];
            for (int base = 0; base < n_all; base += 2 * NEPI * 32) {
                float4 sum[2];
                int gis[2], ps[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int idx = base + hh * NEPI * 32 + mt;
                    ps[hh] = idx < e_cnt[0] ? 0 : (idx < n_all ? 1 : -1);
                    gis[hh] = ps[hh] == 0 ? e_lo[0] + idx : (ps[hh] == 1 ? e_lo[1] + idx - e_cnt[0] : 0);
                    sum[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                const int sp0 = ps[0] >= 0 ? e_chi[ps[0]] - e_clo[ps[0]] + 1 : 0;
                const int sp1 = ps[1] >= 0 ? e_chi[ps[1]] - e_clo[ps[1]] + 1 : 0;
                const int span = sp0 > sp1 ? sp0 : sp1;
                // up to 8 contributors of each group in flight, added in contributor order
                for (int cc = 0; cc < span; cc += 8) {
                    float4 x[2][8];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int p = ps[hh];
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            if (p < 0) continue;
                            const int c2 = e_clo[p] + cc + v;
                            const int sl = cc + v == 0 ? e_slot[p] : 0;
                            if (c2 <= e_chi[p])
                                x[hh][v] = __ldcg(reinterpret_cast<const float4 *>(
                                    wsp + ((size_t)c2 * 2 + sl) * ws_slot_floats() + (size_t)gis[hh] * 4));
                        }
                    }
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int p = ps[hh];
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            if (p < 0 || e_clo[p] + cc + v > e_chi[p]) continue;
                            sum[hh].x = __fadd_rn(sum[hh].x, x[hh][v].x);
                            sum[hh].y = __fadd_rn(sum[hh].y, x[hh][v].y);
                            sum[hh].z = __fadd_rn(sum[hh].z, x[hh][v].z);
                            sum[hh].w = __fadd_rn(sum[hh].w, x[hh][v].w);
                        }
                    }
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (ps[hh] < 0) continue;
                    const int bb = ps[hh] == 0 ? pend0 : pend1;
                    const int gi = gis[hh];
                    const int tok = gi / (BN / 4), r4 = (gi - tok * (BN / 4)) * 4;
                    const float sxt = __ldg(a.sx + tok);
                    const int nn = bb * BN + r4;
                    float *yr = a.Y + (size_t)tok * N;
                    if (nn + 0 < N) yr[nn + 0] = __fmul_rn(sxt, sum[hh].x);
                    if (nn + 1 < N) yr[nn + 1] = __fmul_rn(sxt, sum[hh].y);
                    if (nn + 2 < N) yr[nn + 2] = __fmul_rn(sxt, sum[hh].z);
                    if (nn + 3 < N) yr[nn + 3] = __fmul_rn(sxt, sum[hh].w);
                }
            }
            // every contributor has passed its wait once all have counted
            if (my_bb >= 0 && done_before == my_nc - 1) {
                atomicExch(&ctr[my_bb], 0);
                atomicExch(&done[my_bb], 0);
            }
        }
    }

    // every role is done with TMEM (the MMA issuer waited for its last
    // commit; the epilogue warps waited for every slot they read)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, TMEM_COLS);
}

// Launch one instance.
template <int FMT, int MT, bool CHECK>
cudaError_t launch_gemm_instance(const GemmArgs &a, bool pdl, cudaStream_t s) {
    auto kern = k_verify_gemm<FMT, MT, CHECK>;
    size_t smem = 2048 + (size_t)a.stages * (size_t)a.stage_bytes;
    if (smem < (size_t)MIN_GEMM_SMEM) smem = MIN_GEMM_SMEM;
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
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int FMT>
cudaError_t launch_gemm_fmt(const GemmArgs &a, bool pdl, cudaStream_t s) {
    const int mt = act_rows(a.M);
    if (a.partials) {
        switch (mt) {
            case 16: return launch_gemm_instance<FMT, 16, true>(a, pdl, s);
            case 32: return launch_gemm_instance<FMT, 32, true>(a, pdl, s);
            case 64: return launch_gemm_instance<FMT, 64, true>(a, pdl, s);
            default: return launch_gemm_instance<FMT, 128, true>(a, pdl, s);
        }
    }
    switch (mt) {
        case 16: return launch_gemm_instance<FMT, 16, false>(a, pdl, s);
        case 32: return launch_gemm_instance<FMT, 32, false>(a, pdl, s);
        case 64: return launch_gemm_instance<FMT, 64, false>(a, pdl, s);
        default: return launch_gemm_instance<FMT, 128, false>(a, pdl, s);
    }
}

cudaError_t launch_gemm_w4(const GemmArgs &a, bool pdl, cudaStream_t s);
cudaError_t launch_gemm_w8(const GemmArgs &a, bool pdl, cudaStream_t s);

}  // namespace hq
