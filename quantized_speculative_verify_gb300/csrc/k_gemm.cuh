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
// Integer arithmetic on floating-point tensor cores.  The integer MMA of this
// GPU is far slower than its floating-point MMAs, so the contraction runs as
// exact tcgen05.mma with fp32 accumulation in tensor memory (TMEM), the
// widened weights as the A operand in TMEM (128 channels = 128 TMEM lanes),
// the activation codes as the B operand in shared memory, each quantization
// group's integer sum in its own TMEM accumulator slot:
//  - 4-bit weights, up to 64 rows, groups of 32 or more: kind::f8f6f4.  A
//    4-bit code q in a byte is the e4m3 number q * 2^-9 (subnormal up to 7,
//    then exponent 1), so the codes need only be spread to bytes; an
//    activation code is split into two exact e4m3 digits, q = 16 h + l, which
//    the MMA's N covers side by side (N = 2 * rows).  D = 2^-9 sum q l and
//    2^-9 sum q h, exact; P = 2^9 (D_l + 16 D_h) - z S with the group sum S
//    (the Medium identity: sum qx (q - z) = sum qx q - z sum qx).
//  - otherwise kind::f16 with A in fp16: 8-bit codes widened exactly
//    ((1152 + q) - 1152); 4-bit codes widened to 64 + q (the nibble under the
//    exponent of 64, whose ulp is 1/16), and P = sum qx (64 + q) - (64 + z) S.
// Every partial sum is an exact fp32 value (integers, or multiples of 2^-9,
// below 2^24 units), so the integer P is exact.
//
// Epilogue: y += scale * P with separately rounded fp32 multiply and add, in
// ascending group order, so an output whose whole K range is handled by one
// thread block is bit-identical to the oracle's sequential sum.  (The packed
// f32x2 multiply and add are not used there: the compiler contracts the pair
// into a fused multiply-add, which rounds once.)
//
// Thread block (one per SM, 14 warps, each role running ahead of the next
// through rings of shared-memory stages, A buffers and accumulator slots).
// The unit of the rings is U consecutive tiles of the block's range (U = 2
// where tensor memory allows): every barrier wait, which costs about a
// hundred cycles beside running MMAs, serves U tiles.
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
    int U;           // tiles per pipeline unit (stage, A buffer)
    int V;           // groups per accumulator unit (one wait / commit each)
    int tile_bytes, code_bytes, scale_bytes;
    int act_off;     // offset of the activation blocks within a stage (after U weight tiles)
    int s_off;       // offset of the group sums within a stage (after U activation blocks)
    int act_bytes;   // activation blocks of one tile: (KT/128) * MT * 256
    int s_bytes;     // group sums of one tile: GPT * MT * 4
    int stage_bytes; // one unit: U weight tiles, their activation blocks and group sums
    long long op_s_offset;  // byte offset of the group sums in the operand
};

// Accumulating mode: added (with the zeroing block's own arrival, + 1) to a
// split n-block's counter once its outputs are zero; above any count of
// arrivals (at most MAX_CTAS blocks).
constexpr int ZERO_MARK = 1 << 24;

// Weight stages a block copies in before waiting for the previous kernel.
constexpr int PREFETCH_STAGES = 2;

constexpr int NWID = 4;                       // widening warps
constexpr int WID0 = 2, EPI0 = WID0 + NWID;   // first warp of each role
// epilogue warps: one per TMEM lane quarter up to 32 rows, two above (token
// halves)
__host__ __device__ constexpr int gemm_nepi(int MT) { return MT <= 32 ? 4 : 8; }
__host__ __device__ constexpr int gemm_threads(int MT) { return (EPI0 + gemm_nepi(MT)) * 32; }
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

// Eight 4-bit codes (byte b: features b and b + 4) -> the e4m3 bytes of
// features 0..3 and 4..7.
__device__ __forceinline__ void widen_w4_e4(uint32_t w, uint32_t *o) {
    o[0] = w & 0x0F0F0F0Fu;
    o[1] = (w >> 4) & 0x0F0F0F0Fu;
}

// Eight 4-bit codes (byte b: features b and b + 4) -> four fp16x2 (64 + q),
// features (0,1) (2,3) (4,5) (6,7): a code at bits 4..7 of a 16-bit half
// under the exponent bits 0x5400 (fp16 64, ulp 1/16) reads 64 + q.
__device__ __forceinline__ void widen_w4_f16(uint32_t w, uint32_t *o) {
    constexpr uint32_t M4 = 0x00F000F0u, E64 = 0x54005400u;
    uint32_t y01, y23;  // bytes (0, -, 1, -) and (2, -, 3, -)
    asm("prmt.b32 %0, %1, 0, 0x4140;" : "=r"(y01) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0x4342;" : "=r"(y23) : "r"(w));
    o[0] = ((y01 << 4) & M4) | E64;  // features 0, 1
    o[1] = ((y23 << 4) & M4) | E64;  // 2, 3
    o[2] = (y01 & M4) | E64;         // 4, 5
    o[3] = (y23 & M4) | E64;         // 6, 7
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

// E4: the kind::f8f6f4 path (4-bit weights, digit-encoded operand); CHECK:
// also write the exact integer partial sums (check mode).
template <int FMT, int MT, bool E4, bool CHECK>
__global__ void __launch_bounds__(gemm_threads(MT), 1) k_verify_gemm(const GemmArgs a) {
    constexpr int NEPI = gemm_nepi(MT);
    constexpr int MH = NEPI == 4 ? MT : MT / 2;  // tokens per epilogue thread
    constexpr int CH = MH < 32 ? MH : 32;        // tokens per tensor-memory load
    constexpr int BROWS = E4 ? 2 * MT : MT;      // rows of the B operand (the MMA's N)
    constexpr int DC = BROWS;                    // TMEM columns of one group's accumulator
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int S = a.stages, NA = a.na, ND = a.nd, U = a.U, V = a.V;
    const int vmask = V - 1;  // V is a power of two
    const int KT = a.KT, GPT = a.GPT, G = a.G;
    const int KSTEPS_G = E4 ? G / 32 : G / 16;  // MMAs per group
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
    const int nunits = (ntl + U - 1) / U;
    const int ngroups = ntl * GPT;  // groups of the block, in the order they are computed
    int *err = reinterpret_cast<int *>(a.ws);

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
    const int acols = E4 ? KT / 4 : KT / 2;  // TMEM columns of one tile's A operand
    const int dcol0 = NA * U * acols;         // first accumulator column
    const int quarter = warp & 3;             // TMEM lanes 32 * quarter .. (widening and epilogue warps)
    const int n = quarter * 32 + lane;        // channel within the tile
    const uint32_t lane_field = (uint32_t)(quarter * 32) << 16;

    if (warp == 0) {
        // ------------------------------------------------------ producer ---
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            auto unit_tiles = [&](int u) { return ntl - u * U < U ? ntl - u * U : U; };
            auto copy_weights = [&](int u, int st) {
                const uint32_t fb = smem_addr(&full[st]);
                const int nt = unit_tiles(u);
                mbar_arrive_expect_tx(fb, (uint32_t)(nt * (a.tile_bytes + a.act_bytes + a.s_bytes)));
                // the unit's tiles are consecutive in the blob
                bulk_copy_g2s(smem_addr(ring + (size_t)st * a.stage_bytes),
                              a.blob + (size_t)(t0 + u * U) * (size_t)a.tile_bytes, (uint32_t)(nt * a.tile_bytes), fb,
                              pol_w);
            };
            auto copy_acts = [&](int u, int st) {
                uint8_t *stage = ring + (size_t)st * a.stage_bytes;
                const uint32_t fb = smem_addr(&full[st]);
                for (int j = 0; j < unit_tiles(u); ++j) {
                    const int kt = (t0 + u * U + j) % KTILES;
                    bulk_copy_g2s(smem_addr(stage + a.act_off + j * a.act_bytes), a.qop + (size_t)kt * a.act_bytes,
                                  (uint32_t)a.act_bytes, fb, pol_a);
                    bulk_copy_g2s(smem_addr(stage + a.s_off + j * a.s_bytes),
                                  a.qop + a.op_s_offset + (size_t)kt * a.s_bytes, (uint32_t)a.s_bytes, fb, pol_a);
                }
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
            auto check_unit = [&](int u) {
                for (int j = 0; j < unit_tiles(u); ++j) check(u * U + j);
            };
            int u = 0;
            for (; u < nunits && u < S && u < PREFETCH_STAGES; ++u) copy_weights(u, u);
            pdl_wait();
            for (int j = 0; j < u; ++j) copy_acts(j, j);
            if (!det)
                for (int j = 0; j < u; ++j) check_unit(j);
            RingPos ps{u % S, (uint32_t)((u / S) & 1)};
            for (; u < nunits; ++u) {
                const int st = ps.slot;
                if (!mbar_wait_bounded(smem_addr(&empty[st]), ps.phase ^ 1u, err)) break;
                copy_weights(u, st);
                copy_acts(u, st);
                if (!det) check_unit(u);
                ps.next(S);
            }
            // No copy may still be landing in shared memory when the block exits.
            const int issued = u;
            for (int j = issued > S ? issued - S : 0; j < issued; ++j)
                mbar_wait_bounded(smem_addr(&full[j % S]), (uint32_t)((j / S) & 1), err);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer ---
        const uint32_t idesc = tc_idesc_f16(128, BROWS);
        // descriptor of the first stage's activation blocks; stage st adds
        // st * stage_bytes (the start address field counts 16-byte units)
        const uint64_t bdesc_ring = tc_smem_desc(smem_addr(ring + a.act_off), 16u * BROWS, 128u);
        const uint32_t stage_units = (uint32_t)(a.stage_bytes >> 4);
        const uint32_t tile_act_units = (uint32_t)(a.act_bytes >> 4);
        const uint32_t group_b_units = (uint32_t)((KSTEPS_G * 32 * BROWS) >> 4);
        // The whole warp runs the loop (all values warp-uniform) and waits;
        // one elected lane issues each MMA and commit through a predicate.
        // The unit's stage needs no wait of its own: its A buffer is widened
        // only after the stage has landed.
        __syncwarp();
        const uint32_t leader = elect_one() ? 1u : 0u;
        bool ok = true;
        RingPos ps{0, 0u}, pa{0, 0u}, pd{0, 0u};
        int g = 0;  // groups issued so far
        for (int u = 0; u < nunits; ++u) {
            const int nt = ntl - u * U < U ? ntl - u * U : U;
            const uint32_t a_tm = tbase + (uint32_t)(pa.slot * U * acols);
            const uint64_t bdesc = bdesc_ring + (uint64_t)(ps.slot * stage_units);
            if (ok) ok = mbar_wait_bounded(smem_addr(&a_full[pa.slot]), pa.phase, err);
            tc_fence_after();
            for (int j = 0; j < nt; ++j) {
                for (int gl = 0; gl < GPT; ++gl, ++g) {
                    const int r = g & vmask;
                    if (r == 0) {
                        if (ok) ok = mbar_wait_bounded(smem_addr(&d_empty[pd.slot]), pd.phase ^ 1u, err);
                        tc_fence_after();
                    }
                    const uint32_t d_tm = tbase + (uint32_t)(dcol0 + (pd.slot * V + r) * DC);
                    const uint32_t a_g = a_tm + (uint32_t)(j * acols + gl * KSTEPS_G * 8);
                    uint64_t b_g = bdesc + (uint64_t)(j * tile_act_units + gl * group_b_units);
                    for (int ks = 0; ks < KSTEPS_G; ++ks) {
                        if (E4)
                            tc_mma_e4m3_ts_if(leader, d_tm, a_g + (uint32_t)(ks * 8), b_g, idesc, ks > 0 ? 1u : 0u);
                        else
                            tc_mma_f16_ts_if(leader, d_tm, a_g + (uint32_t)(ks * 8), b_g, idesc, ks > 0 ? 1u : 0u);
                        b_g += (uint64_t)((32 * BROWS) >> 4);
                    }
                    if (r == vmask || g == ngroups - 1) {
                        tc_commit_if(leader, smem_addr(&d_full[pd.slot]));
                        pd.next(ND);
                    }
                }
            }
            tc_commit_if(leader, smem_addr(&a_empty[pa.slot]));
            tc_commit_if(leader, smem_addr(&empty[ps.slot]));
            ps.next(S);
            pa.next(NA);
        }
        // every MMA has completed before the block frees TMEM
        tc_commit_if(leader, smem_addr(done_bar));
        mbar_wait_bounded(smem_addr(done_bar), 0u, err);
    } else if (warp < EPI0) {
        // ----------------------------------------------------- widening ---
        const int KC = KT / 64;  // 64-feature chunks per tile
        bool ok = true;
        RingPos ps{0, 0u}, pa{0, 0u};
        for (int u = 0; u < nunits; ++u) {
            const int nt = ntl - u * U < U ? ntl - u * U : U;
            const int st = ps.slot, ab = pa.slot;
            if (ok) ok = mbar_wait_bounded(smem_addr(&full[st]), ps.phase, err);
            if (ok) ok = mbar_wait_bounded(smem_addr(&a_empty[ab]), pa.phase ^ 1u, err);
            __syncwarp();
            tc_fence_after();
            for (int j = 0; j < nt; ++j) {
                const uint8_t *tile = ring + (size_t)st * a.stage_bytes + (size_t)j * a.tile_bytes;
                const uint32_t a_col = (uint32_t)((ab * U + j) * acols);
                if (E4) {
                    // 64 features -> 16 columns of e4m3 bytes; one store per 128 features
                    for (int c = 0; c < KC; c += 2) {
                        uint32_t v[32];
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            uint4 uu[2];
#pragma unroll
                            for (int p = 0; p < 2; ++p)
                                uu[p] = *reinterpret_cast<const uint4 *>(tile + ((size_t)((c + cc) * 2 + p) * BN + n) * 16);
#pragma unroll
                            for (int p = 0; p < 2; ++p) {
                                uint32_t *o = v + 16 * cc + 8 * p;
                                widen_w4_e4(uu[p].x, o + 0);
                                widen_w4_e4(uu[p].y, o + 2);
                                widen_w4_e4(uu[p].z, o + 4);
                                widen_w4_e4(uu[p].w, o + 6);
                            }
                        }
                        tmem_st32(tbase + lane_field + a_col + (uint32_t)(c * 16), v);
                    }
                } else {
                    for (int c = 0; c < KC; ++c) {
                        uint32_t v[32];
                        if (FMT == HQ_W4_ASYM) {
                            uint4 uu[2];
#pragma unroll
                            for (int p = 0; p < 2; ++p)
                                uu[p] = *reinterpret_cast<const uint4 *>(tile + ((size_t)(c * 2 + p) * BN + n) * 16);
#pragma unroll
                            for (int p = 0; p < 2; ++p) {
                                widen_w4_f16(uu[p].x, v + 16 * p + 0);
                                widen_w4_f16(uu[p].y, v + 16 * p + 4);
                                widen_w4_f16(uu[p].z, v + 16 * p + 8);
                                widen_w4_f16(uu[p].w, v + 16 * p + 12);
                            }
                        } else {
                            uint4 uu[4];
#pragma unroll
                            for (int p = 0; p < 4; ++p)
                                uu[p] = *reinterpret_cast<const uint4 *>(tile + ((size_t)(c * 4 + p) * BN + n) * 16);
#pragma unroll
                            for (int p = 0; p < 4; ++p) {
                                widen_i8(uu[p].x, v + 8 * p + 0);
                                widen_i8(uu[p].y, v + 8 * p + 2);
                                widen_i8(uu[p].z, v + 8 * p + 4);
                                widen_i8(uu[p].w, v + 8 * p + 6);
                            }
                        }
                        tmem_st32(tbase + lane_field + a_col + (uint32_t)(c * 32), v);
                    }
                }
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
        const int mt = threadIdx.x - EPI0 * 32;  // epilogue thread 0..NEPI*32-1
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
        int g = 0;  // groups folded so far
        // position of the tile being folded: n-block eb, K tile ekt
        int eb = t0 / KTILES, ekt = t0 - eb * KTILES, seg_k0 = ekt;
        for (int u = 0; u < nunits; ++u) {
            const int nt = ntl - u * U < U ? ntl - u * U : U;
            const int st = ps.slot;
            // the stage's scales, zero points and group sums are read below
            if (ok) ok = mbar_wait_bounded(smem_addr(&full[st]), ps.phase, err);
            for (int j = 0; j < nt; ++j) {
                const int i = u * U + j;
                if (i == 0 || ekt == 0) {
                    seg_k0 = ekt;
#pragma unroll
                    for (int t = 0; t < MH; ++t) y[t] = 0.0f;
                }
                const uint8_t *tile = ring + (size_t)st * a.stage_bytes + (size_t)j * a.tile_bytes;
                const float *tsc = reinterpret_cast<const float *>(tile + a.code_bytes) + (size_t)n * GPT;
                const uint8_t *tzp = tile + a.code_bytes + a.scale_bytes;
                const float *tS = reinterpret_cast<const float *>(ring + (size_t)st * a.stage_bytes + a.s_off +
                                                                  (size_t)j * a.s_bytes);
                for (int gl = 0; gl < GPT; ++gl, ++g) {
                    const int r = g & vmask;
                    if (r == 0) {
                        if (ok) ok = mbar_wait_bounded(smem_addr(&d_full[pd.slot]), pd.phase, err);
                        __syncwarp();
                        tc_fence_after();
                    }
                    const float sc = tsc[gl];
                    float nz = 0.0f;
                    if (FMT == HQ_W4_ASYM) {
                        const int zi = n * GPT + gl;
                        const uint32_t zb8 = tzp[zi >> 1];
                        const float z = (float)((zi & 1) ? (zb8 >> 4) : (zb8 & 15u));
                        // E4: in units of 2^-9 (the accumulators hold 2^-9 sum q d)
                        nz = E4 ? -z * (1.0f / 512.0f) : -(64.0f + z);
                    }
                    const f2 nz2 = f2_make(nz, nz);
                    const float scale = E4 ? sc * 512.0f : sc;  // exact: a power-of-two multiple
                    const float *Sg = tS + gl * MT + h * MH;
#pragma unroll
                    for (int c0 = 0; c0 < MH; c0 += CH) {
                        float acc[CH], acc_h[E4 ? CH : 1];
                        const uint32_t taddr =
                            tbase + lane_field + (uint32_t)(dcol0 + (pd.slot * V + r) * DC + h * MH + c0);
                        if constexpr (CH == 8) {
                            tmem_ld8(taddr, acc);
                            if constexpr (E4) tmem_ld8(taddr + MT, acc_h);
                        } else if constexpr (CH == 16) {
                            tmem_ld16(taddr, acc);
                            if constexpr (E4) tmem_ld16(taddr + MT, acc_h);
                        } else {
                            tmem_ld32(taddr, acc);
                            if constexpr (E4) tmem_ld32(taddr + MT, acc_h);
                        }
                        tmem_wait_ld();
#pragma unroll
                        for (int p = 0; p < CH / 2; ++p) {
                            f2 P2 = f2_make(acc[2 * p], acc[2 * p + 1]);
                            if constexpr (E4)  // low digit + 16 x high digit (exact)
                                P2 = f2_fma(f2_make(16.0f, 16.0f), f2_make(acc_h[2 * p], acc_h[2 * p + 1]), P2);
                            if (FMT == HQ_W4_ASYM) {
                                // exact: P = sum qx q' - (z or 64 + z) S, below 2^24 units
                                const float2 sv = *reinterpret_cast<const float2 *>(Sg + c0 + 2 * p);
                                P2 = f2_fma(nz2, f2_make(sv.x, sv.y), P2);
                            }
                            float p0, p1;
                            f2_split(P2, p0, p1);
                            const int tok = h * MH + c0 + 2 * p;
                            if (CHECK) {
                                const int gq = ekt * GPT + gl;
                                const int nn = eb * BN + n;
                                const float uu = E4 ? 512.0f : 1.0f;
                                if (gq < a.NGK && nn < N) {
                                    if (tok < M) a.partials[((size_t)tok * N + nn) * a.NGK + gq] = __float2int_rn(p0 * uu);
                                    if (tok + 1 < M)
                                        a.partials[((size_t)(tok + 1) * N + nn) * a.NGK + gq] = __float2int_rn(p1 * uu);
                                }
                            }
                            // y += scale * P: product rounded, then sum rounded
                            y[c0 + 2 * p] = __fadd_rn(y[c0 + 2 * p], __fmul_rn(scale, p0));
                            y[c0 + 2 * p + 1] = __fadd_rn(y[c0 + 2 * p + 1], __fmul_rn(scale, p1));
                        }
                    }
                    if (r == vmask || g == ngroups - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_addr(&d_empty[pd.slot]));
                        pd.next(ND);
                    }
                }

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
                        // part of the K range: publish the partial sums now,
                        // count the arrival once this block's tiles are all done
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
                        // part of the K range, accumulating mode: once the
                        // zeroing is visible (the segment's flag), add sx *
                        // (this block's sum) into Y
                        if (ok) ok = wait_flag_bounded(smem_addr(&sflag[nsplit]), err);
                        ++nsplit;
#pragma unroll
                        for (int t = 0; t < MH; ++t) {
                            const int tok = h * MH + t;
                            if (tok < M && nn < N)
                                atomicAdd(a.Y + (size_t)tok * N + nn, __fmul_rn(__ldg(a.sx + tok), y[t]));
                        }
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
template <int FMT, int MT, bool E4, bool CHECK>
cudaError_t launch_gemm_instance(const GemmArgs &a, bool pdl, cudaStream_t s) {
    auto kern = k_verify_gemm<FMT, MT, E4, CHECK>;
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
    cfg.blockDim = dim3(gemm_threads(MT));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int FMT, bool CHECK>
cudaError_t launch_gemm_check(const GemmArgs &a, bool pdl, cudaStream_t s) {
    const int mt = act_rows(a.M);
    if constexpr (FMT == HQ_W4_ASYM) {
        if (act_e4(FMT, a.M, a.G)) {
            switch (mt) {
                case 16: return launch_gemm_instance<FMT, 16, true, CHECK>(a, pdl, s);
                case 32: return launch_gemm_instance<FMT, 32, true, CHECK>(a, pdl, s);
                default: return launch_gemm_instance<FMT, 64, true, CHECK>(a, pdl, s);
            }
        }
    }
    switch (mt) {
        case 16: return launch_gemm_instance<FMT, 16, false, CHECK>(a, pdl, s);
        case 32: return launch_gemm_instance<FMT, 32, false, CHECK>(a, pdl, s);
        case 64: return launch_gemm_instance<FMT, 64, false, CHECK>(a, pdl, s);
        default: return launch_gemm_instance<FMT, 128, false, CHECK>(a, pdl, s);
    }
}

template <int FMT>
cudaError_t launch_gemm_fmt(const GemmArgs &a, bool pdl, cudaStream_t s) {
    return a.partials ? launch_gemm_check<FMT, true>(a, pdl, s) : launch_gemm_check<FMT, false>(a, pdl, s);
}

cudaError_t launch_gemm_w4(const GemmArgs &a, bool pdl, cudaStream_t s);
cudaError_t launch_gemm_w8(const GemmArgs &a, bool pdl, cudaStream_t s);

}  // namespace hq
