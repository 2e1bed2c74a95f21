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
//  - 4-bit weights, 33 to 64 rows (fewer rows run on the register-resident
//    kernel, k_gemm_rs.cuh), groups of 32 or more: kind::f8f6f4.  A
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
// Epilogue: y += scale * P in ascending group order.  In exact-order and
// check modes the multiply and the add round separately (scalar fp32
// operations), so an output whose whole K range is handled by one thread
// block is bit-identical to the oracle's sequential sum; the packed f32x2
// multiply and add are not used there because the compiler contracts the pair
// into a fused multiply-add, which rounds once.  Otherwise each group is one
// packed fused multiply-add (two tokens per instruction): one rounding per
// group instead of two, within the fp32 tolerance of the oracle.
//
// Thread block (one per SM, 11 or 15 warps, each role running ahead of the next
// through rings of shared-memory stages, A buffers and accumulator slots).
// The unit of the rings is U consecutive tiles of the block's range (up to 32
// rows U = 4 where tensor memory allows, else 2 or 1; above 32 rows U = 1):
// every barrier wait, which costs about a hundred cycles beside running MMAs,
// serves U tiles.
//  - warp 0, one lane: weight producer, and the last warp, one lane:
//    activation producer (gemm_common.cuh).  Per unit, one bulk copy of its
//    weight tiles and one per run of activation K tiles (codes and group
//    sums) into a stage (mbarrier transaction counts).  The weight copies of
//    the first stage go out before waiting for the previous kernel of the
//    stream; the activation copies after.
//  - warp 1: tensor-memory owner and MMA issuer (one elected lane).  Per
//    group: wait for a free accumulator slot, issue group/16 MMAs (K = 16
//    each) from one unrolled sequence, commit to the slot's "full" barrier.
//  - warps 2..5: widening.  Warp w owns TMEM lanes 32 (w % 4) .. + 31 (= the
//    tile's channels); each thread widens its channel's codes of the whole
//    tile into the tile's A buffer (tcgen05.st).
//  - warps 6..9 (up to 32 rows) or 6..13: epilogue.  Same lanes, and half h = (w - 6) / 4 of the
//    tokens: fold each group out of its accumulator slot (tcgen05.ld) into the
//    running fp32 sums, and write, add or publish them at the end of a
//    128-channel block's segment.
#pragma once

#include <cuda_runtime.h>

#include "gemm_common.cuh"
#include "hq_internal.cuh"
#include "hq_tc.cuh"

namespace hq {

constexpr int NWID = 4;                       // widening warps
constexpr int WID0 = 2, EPI0 = WID0 + NWID;   // first warp of each role
// epilogue warps: one per TMEM lane quarter up to 32 rows, two above (token
// halves); the activation producer comes after them
__host__ __device__ constexpr int gemm_nepi(int MT) { return MT <= 32 ? 4 : 8; }
__host__ __device__ constexpr int gemm_threads(int MT) { return (EPI0 + gemm_nepi(MT) + 1) * 32; }
constexpr int TMEM_COLS = 512;                // one block per SM owns all of TMEM
constexpr int MAX_NA = 4;                     // A buffers (widened weight tiles) in TMEM
constexpr int MAX_ND = 16;                    // accumulator slots in TMEM
// Every block asks for at least this much shared memory, so that no two
// blocks of the kernel share an SM (each takes all of its TMEM).
constexpr int MIN_GEMM_SMEM = 120 * 1024;

// Words t and t + 1 (t even) of a 32-feature run (nibble i of word t: feature
// 2t + 8i, nibble i + 4: feature 2t + 8i + 1) -> the e4m3 bytes of features
// 2t + 8i .. 2t + 8i + 3 in o[t / 2 + 2i], i = 0..3.  A byte permute gathers
// the four bytes holding each feature quad's low (then high) nibbles.
__device__ __forceinline__ void widen_w4_e4(uint32_t w0, uint32_t w1, int t, uint32_t *o) {
    uint32_t p, q;
    asm("prmt.b32 %0, %1, %2, 0x6420;" : "=r"(p) : "r"(w0), "r"(w1));  // bytes 0, 2 of each
    asm("prmt.b32 %0, %1, %2, 0x7531;" : "=r"(q) : "r"(w0), "r"(w1));  // bytes 1, 3 of each
    o[t / 2 + 0] = p & 0x0F0F0F0Fu;
    o[t / 2 + 2] = (p >> 4) & 0x0F0F0F0Fu;
    o[t / 2 + 4] = q & 0x0F0F0F0Fu;
    o[t / 2 + 6] = (q >> 4) & 0x0F0F0F0Fu;
}

// Word t of a 32-feature run -> four fp16x2 (64 + q) of the feature pairs
// (2t + 8i, 2t + 8i + 1) in o[t + 4i]: a code at bits 4..7 of a 16-bit half
// under the exponent bits 0x5400 (fp16 64, ulp 1/16) reads 64 + q.
__device__ __forceinline__ void widen_w4_f16(uint32_t w, int t, uint32_t *o) {
    constexpr uint32_t M4 = 0x00F000F0u, E64 = 0x54005400u;
    o[t + 0] = ((w << 4) & M4) | E64;
    o[t + 4] = (w & M4) | E64;
    o[t + 8] = ((w >> 4) & M4) | E64;
    o[t + 12] = ((w >> 8) & M4) | E64;
}

// Four int8 codes (word t of a 16-feature run: features 2t, 2t+1, 2t+8,
// 2t+9) -> the fp16x2 q of the pairs (2t, 2t+1) in lo and (2t+8, 2t+9) in
// hi: bias to unsigned, place under the fp16 exponent bits 0x64
// (1024 + 128 + q), subtract 1152.
__device__ __forceinline__ void widen_i8(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t l, h;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(l) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(h) : "r"(u), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(0x64806480u));
}

// E4: the kind::f8f6f4 path (4-bit weights, digit-encoded operand).  EXACT:
// y += scale * P with separately rounded multiply and add (the oracle's
// arithmetic), and the exact integer partial sums written where the caller
// asks for them (check mode); otherwise one fused multiply-add per group.
template <int FMT, int MT, bool E4, bool EXACT>
__global__ void __launch_bounds__(gemm_threads(MT), 1) k_verify_gemm(const GemmArgs a) {
    constexpr int NEPI = gemm_nepi(MT);
    constexpr int MH = NEPI == 4 ? MT : MT / 2;  // tokens per epilogue thread
    constexpr int CH = MH < 32 ? MH : 32;        // tokens per tensor-memory load
    constexpr int NCH = MH / CH;                 // loads per group (per digit)
    constexpr int BUF = (E4 ? 2 : 1) * CH;       // accumulator values of one load (both digits)
    // The loads of the next group overlap the arithmetic of this one where
    // the registers allow a second buffer.
    constexpr bool PIPE = NCH == 1 && NEPI == 4 && 2 * BUF + MH <= 96;
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
    // accumulating mode: two segment flags; then the initial fill's counter
    int *sflag = reinterpret_cast<int *>(done_bar + 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sflag + 4);
    uint8_t *ring = smem_raw + 2048;

    // warp index made visibly warp-uniform (tensor-memory addresses derive from it)
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    const GemmBlock blk = make_gemm_block(a, ring, full, empty, sflag);
    const int t0 = blk.t0, ntl = blk.ntl, nunits = blk.nunits;
    int *err = blk.err;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            // the two producers' arrivals (each with its transaction bytes)
            mbar_init(smem_addr(&full[i]), 2);
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
        sflag[0] = sflag[1] = sflag[2] = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    pdl_launch_dependents();

    const bool det = blk.det;
    const int KTILES = a.KTILES;
    const int acols = E4 ? KT / 4 : KT / 2;  // TMEM columns of one tile's A operand
    const int dcol0 = NA * U * acols;         // first accumulator column
    const int quarter = warp & 3;             // TMEM lanes 32 * quarter .. (widening and epilogue warps)
    const int n = quarter * 32 + lane;        // channel within the tile
    const uint32_t lane_field = (uint32_t)(quarter * 32) << 16;

    if (warp == 0) {
        // ----------------------------------------------- weight producer ---
        if (lane == 0) gemm_weight_producer(a, blk);
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer ---
        // A unit's MMAs form one sequence: MMA m (K = 32 e4m3 bytes or 16
        // fp16 features) of tile j = m / MPT reads A columns 8 m of the
        // unit's A buffer (the unit's tiles are adjacent there) and K slice
        // m % MPT of tile j's activation codes.  The accumulator slot and the
        // accumulate flag depend on the group layout: MMA k of an accumulator
        // unit adds into group k / KSTEPS_G's slot, starting it when
        // k % KSTEPS_G == 0.
        const uint32_t idesc = tc_idesc_f16(128, BROWS);
        // descriptor of the first stage's activation blocks; the start
        // address field (bits 0..13, 16-byte units) never carries into the
        // next field, so offsets are added to the low word alone
        const uint64_t bdesc_ring = tc_smem_desc(smem_addr(ring + a.act_off), 16u * BROWS, 128u);
        const uint32_t bd_lo = (uint32_t)bdesc_ring, bd_hi = (uint32_t)(bdesc_ring >> 32);
        const uint32_t stage_units = (uint32_t)(a.stage_bytes >> 4);
        constexpr uint32_t BSTEP = (32u * BROWS) >> 4;  // one MMA's K slice of the B operand
        const int MPT = E4 ? KT / 32 : KT / 16;         // MMAs per tile (a power of two)
        const int lmpt = __ffs(MPT) - 1;
        const uint32_t tile_units = (uint32_t)(a.act_tile_bytes >> 4);
        const int ksm = KSTEPS_G - 1;                    // KSTEPS_G is a power of two
        const int lks = __ffs(KSTEPS_G) - 1;
        const int vmm = V * KSTEPS_G;                    // MMAs per accumulator unit
        // The whole warp runs the loop (all values warp-uniform) and waits;
        // one elected lane issues each MMA and commit through a predicate.
        // The unit's stage needs no wait of its own: its A buffer is widened
        // only after the stage has landed.
        __syncwarp();
        const uint32_t leader = elect_one() ? 1u : 0u;
        bool ok = true;
        RingPos ps{0, 0u}, pa{0, 0u}, pd{0, 0u};
        for (int u = 0; u < nunits; ++u) {
            const int nt = ntl - u * U < U ? ntl - u * U : U;
            const int nm = nt * MPT;
            const uint32_t a_unit = tbase + (uint32_t)(pa.slot * U * acols);
            const uint32_t b_unit = bd_lo + (uint32_t)ps.slot * stage_units;
            if (ok) ok = mbar_wait_bounded(smem_addr(&a_full[pa.slot]), pa.phase, err);
            tc_fence_after();
            for (int m0 = 0; m0 < nm; m0 += vmm) {
                if (ok) ok = mbar_wait_bounded(smem_addr(&d_empty[pd.slot]), pd.phase ^ 1u, err);
                tc_fence_after();
                const uint32_t d_unit = tbase + (uint32_t)(dcol0 + pd.slot * V * DC);
                const int m1 = nm - m0 < vmm ? nm : m0 + vmm;
                // the accumulator unit's MMAs, tile by tile
                for (int m = m0; m < m1;) {
                    const int j = m >> lmpt;
                    const int mj = m1 < (j + 1) * MPT ? m1 : (j + 1) * MPT;
                    const uint32_t b_tile = b_unit + (uint32_t)j * tile_units - (uint32_t)(j * MPT) * BSTEP;
#pragma unroll 4
                    for (; m < mj; ++m) {
                        const int k = m - m0;
                        const uint32_t d = d_unit + (uint32_t)((k >> lks) * DC);
                        const uint64_t bd = ((uint64_t)bd_hi << 32) | (uint64_t)(b_tile + (uint32_t)m * BSTEP);
                        const uint32_t acc = (uint32_t)(k & ksm);
                        if (E4)
                            tc_mma_e4m3_ts_if(leader, d, a_unit + (uint32_t)(m * 8), bd, idesc, acc);
                        else
                            tc_mma_f16_ts_if(leader, d, a_unit + (uint32_t)(m * 8), bd, idesc, acc);
                    }
                }
                tc_commit_if(leader, smem_addr(&d_full[pd.slot]));
                pd.next(ND);
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
                                widen_w4_e4(uu[p].x, uu[p].y, 0, o);
                                widen_w4_e4(uu[p].z, uu[p].w, 2, o);
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
                                widen_w4_f16(uu[p].x, 0, v + 16 * p);
                                widen_w4_f16(uu[p].y, 1, v + 16 * p);
                                widen_w4_f16(uu[p].z, 2, v + 16 * p);
                                widen_w4_f16(uu[p].w, 3, v + 16 * p);
                            }
                        } else {
                            uint4 uu[4];
#pragma unroll
                            for (int p = 0; p < 4; ++p)
                                uu[p] = *reinterpret_cast<const uint4 *>(tile + ((size_t)(c * 4 + p) * BN + n) * 16);
#pragma unroll
                            for (int p = 0; p < 4; ++p) {
                                widen_i8(uu[p].x, v[8 * p + 0], v[8 * p + 4]);
                                widen_i8(uu[p].y, v[8 * p + 1], v[8 * p + 5]);
                                widen_i8(uu[p].z, v[8 * p + 2], v[8 * p + 6]);
                                widen_i8(uu[p].w, v[8 * p + 3], v[8 * p + 7]);
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
    } else if (warp < EPI0 + NEPI) {
        // ----------------------------------------------------- epilogue ---
        pdl_wait();
        const int mt = threadIdx.x - EPI0 * 32;  // epilogue thread 0..NEPI*32-1
        const int h = (warp - EPI0) >> 2;        // token half
        const int M = a.M, N = a.N;
        float *wsp = reinterpret_cast<float *>(a.ws + ws_partial_offset());

        // y[p]: the running sums of tokens h*MH + 2p, + 2p + 1
        f2 y[MH / 2];
        bool ok = true;
        int pend0 = -1, pend1 = -1;
        const int first_b = t0 / KTILES;
        int nsplit = 0, mark_old = 0;
        mark_old = gemm_zero_outputs(a, blk, mt, NEPI * 32, 1);

        RingPos ps{0, 0u}, pd{0, 0u};
        // position of the tile being folded: n-block eb, K tile ekt
        int eb = t0 / KTILES, ekt = t0 - eb * KTILES, seg_k0 = ekt;
        // the tile being folded: its scales (this channel's row), zero points, group sums
        const float *tsc = nullptr;
        const uint8_t *tzp = nullptr;
        const float *tS = nullptr;
        const f2 c16 = f2_make(16.0f, 16.0f);

        // End of tile i of the block's range: the end of an n-block segment?
        auto tile_end = [&](int i) {
            if (ekt == KTILES - 1 || i == ntl - 1) {
                const int nn = eb * BN + n;
                if (seg_k0 == 0 && ekt == KTILES - 1) {
                    // the whole K range of the n-block: write Y
#pragma unroll
                    for (int p = 0; p < MH / 2; ++p) {
                        float v0, v1;
                        f2_split(y[p], v0, v1);
                        const int tok = h * MH + 2 * p;
                        if (tok < M && nn < N) a.Y[(size_t)tok * N + nn] = __fmul_rn(__ldg(a.sx + tok), v0);
                        if (tok + 1 < M && nn < N) a.Y[(size_t)(tok + 1) * N + nn] = __fmul_rn(__ldg(a.sx + tok + 1), v1);
                    }
                } else if (det) {
                    // part of the K range: publish the partial sums now,
                    // count the arrival once this block's tiles are all done
                    const int slot = eb == first_b ? 0 : 1;
                    float *mys = wsp + ((size_t)blockIdx.x * 2 + slot) * ws_slot_floats();
#pragma unroll
                    for (int p = 0; p < MH / 2; ++p) {
                        float v0, v1;
                        f2_split(y[p], v0, v1);
                        const int tok = h * MH + 2 * p;
                        if (tok < M) __stcg(mys + (size_t)tok * BN + n, v0);
                        if (tok + 1 < M) __stcg(mys + (size_t)(tok + 1) * BN + n, v1);
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
                    for (int p = 0; p < MH / 2; ++p) {
                        float v0, v1;
                        f2_split(y[p], v0, v1);
                        const int tok = h * MH + 2 * p;
                        if (tok < M && nn < N) atomicAdd(a.Y + (size_t)tok * N + nn, __fmul_rn(__ldg(a.sx + tok), v0));
                        if (tok + 1 < M && nn < N)
                            atomicAdd(a.Y + (size_t)(tok + 1) * N + nn, __fmul_rn(__ldg(a.sx + tok + 1), v1));
                    }
                }
            }
            if (++ekt == KTILES) {
                ekt = 0;
                ++eb;
            }
        };

        // Per group gl of the current tile: the scale as applied to the
        // accumulators (x 2^9 on the e4m3 path, exact) and the zero-point
        // factor of the group sums (-z 2^-9 there, -(64 + z) on the fp16 path).
        auto group_params = [&](int gl, float &scale, float &nz) {
            const float sc = tsc[gl];
            scale = E4 ? sc * 512.0f : sc;
            nz = 0.0f;
            if (FMT == HQ_W4_ASYM) {
                const int zi = n * GPT + gl;
                const uint32_t zb8 = tzp[zi >> 1];
                const float z = (float)((zi & 1) ? (zb8 >> 4) : (zb8 & 15u));
                nz = E4 ? -z * (1.0f / 512.0f) : -(64.0f + z);
            }
        };
        // group sums of tokens h*MH + c*CH .. + CH - 1 (4-bit weights only;
        // read ahead of the fold where the loads are pipelined, else read by
        // the fold itself)
        auto load_S = [&](int gl, int c, float (&sv)[CH]) {
            if (FMT == HQ_W4_ASYM && PIPE) {
                const float4 *src = reinterpret_cast<const float4 *>(tS + gl * MT + c * CH);
#pragma unroll
                for (int q = 0; q < CH / 4; ++q) {
                    const float4 v = src[q];
                    sv[4 * q] = v.x;
                    sv[4 * q + 1] = v.y;
                    sv[4 * q + 2] = v.z;
                    sv[4 * q + 3] = v.w;
                }
            }
        };
        // Fold chunk c of group gl (accumulators in b: CH low-digit values,
        // then CH high-digit values on the e4m3 path) into y.
        auto fold = [&](int gl, int c, const float (&b)[BUF], const float (&sv)[CH], float scale, float nz) {
            const f2 nz2 = f2_make(nz, nz), sc2 = f2_make(scale, scale);
#pragma unroll
            for (int p = 0; p < CH / 2; ++p) {
                f2 P2 = f2_make(b[2 * p], b[2 * p + 1]);
                if constexpr (E4)  // low digit + 16 x high digit (exact)
                    P2 = f2_fma(c16, f2_make(b[CH + 2 * p], b[CH + 2 * p + 1]), P2);
                if (FMT == HQ_W4_ASYM) {  // exact: P = sum qx q' - (z or 64 + z) S, below 2^24 units
                    if constexpr (PIPE) {
                        P2 = f2_fma(nz2, f2_make(sv[2 * p], sv[2 * p + 1]), P2);
                    } else {
                        const float2 s = *reinterpret_cast<const float2 *>(tS + gl * MT + c * CH + 2 * p);
                        P2 = f2_fma(nz2, f2_make(s.x, s.y), P2);
                    }
                }
                const int yp = c * (CH / 2) + p;
                if constexpr (EXACT) {
                    float p0, p1, y0, y1;
                    f2_split(P2, p0, p1);
                    if (a.partials) {
                        const int gq = ekt * GPT + gl;
                        const int nn = eb * BN + n;
                        const int tok = h * MH + c * CH + 2 * p;
                        const float uu = E4 ? 512.0f : 1.0f;
                        if (gq < a.NGK && nn < N) {
                            if (tok < M) a.partials[((size_t)tok * N + nn) * a.NGK + gq] = __float2int_rn(p0 * uu);
                            if (tok + 1 < M)
                                a.partials[((size_t)(tok + 1) * N + nn) * a.NGK + gq] = __float2int_rn(p1 * uu);
                        }
                    }
                    // y += scale * P: product rounded, then sum rounded
                    f2_split(y[yp], y0, y1);
                    y0 = __fadd_rn(y0, __fmul_rn(scale, p0));
                    y1 = __fadd_rn(y1, __fmul_rn(scale, p1));
                    y[yp] = f2_make(y0, y1);
                } else {
                    // y += scale * P, one rounding
                    y[yp] = f2_fma(sc2, P2, y[yp]);
                }
            }
        };
        // tensor-memory loads of chunk c of unit group q into b
        auto load_acc = [&](int q, int c, float (&b)[BUF]) {
            const uint32_t ta =
                tbase + lane_field + (uint32_t)(dcol0 + (pd.slot * V + (q & vmask)) * DC + h * MH + c * CH);
            if constexpr (CH == 8) {
                tmem_ld8(ta, b);
                if constexpr (E4) tmem_ld8(ta + MT, b + CH);
            } else if constexpr (CH == 16) {
                tmem_ld16(ta, b);
                if constexpr (E4) tmem_ld16(ta + MT, b + CH);
            } else {
                tmem_ld32(ta, b);
                if constexpr (E4) tmem_ld32(ta + MT, b + CH);
            }
        };
        auto acc_wait = [&]() {
            if (ok) ok = mbar_wait_bounded(smem_addr(&d_full[pd.slot]), pd.phase, err);
            __syncwarp();
            tc_fence_after();
        };
        auto acc_free = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&d_empty[pd.slot]));
            pd.next(ND);
        };

        for (int u = 0; u < nunits; ++u) {
            const int nt = ntl - u * U < U ? ntl - u * U : U;
            const int nq = nt * GPT;  // groups of the unit; accumulator units start at multiples of V
            const int st = ps.slot;
            const uint8_t *stage = ring + (size_t)st * a.stage_bytes;
            // the stage's scales, zero points and group sums are read below
            if (ok) ok = mbar_wait_bounded(smem_addr(&full[st]), ps.phase, err);
            int j = 0, gl = 0;  // tile and group being folded
            auto tile_begin = [&]() {
                const int i = u * U + j;
                if (i == 0 || ekt == 0) {
                    seg_k0 = ekt;
#pragma unroll
                    for (int p = 0; p < MH / 2; ++p) y[p] = f2_make(0.0f, 0.0f);
                }
                const uint8_t *tile = stage + (size_t)j * a.tile_bytes;
                tsc = reinterpret_cast<const float *>(tile + a.code_bytes) + (size_t)n * GPT;
                tzp = tile + a.code_bytes + a.scale_bytes;
                tS = reinterpret_cast<const float *>(stage + a.act_off + (size_t)j * a.act_tile_bytes + a.act_bytes) +
                     h * MH;
            };
            auto next_group = [&]() {
                if (++gl == GPT) {
                    tile_end(u * U + j);
                    gl = 0;
                    if (++j < nt) tile_begin();
                }
            };
            tile_begin();
            if constexpr (PIPE) {
                // The loads of group q + 1 go out before group q is folded.
                float bA[BUF], bB[BUF];
                acc_wait();  // a unit starts an accumulator unit
                load_acc(0, 0, bA);
                auto step = [&](int q, float (&cur)[BUF], float (&nxt)[BUF]) {
                    float scale, nz, sv[CH];
                    group_params(gl, scale, nz);
                    load_S(gl, 0, sv);
                    tmem_wait_ld();
                    if ((q & vmask) == vmask || q == nq - 1) acc_free();
                    if (q + 1 < nq) {
                        if (((q + 1) & vmask) == 0) acc_wait();
                        load_acc(q + 1, 0, nxt);
                    }
                    fold(gl, 0, cur, sv, scale, nz);
                    next_group();
                };
                for (int q = 0; q < nq; q += 2) {
                    step(q, bA, bB);
                    if (q + 1 < nq) step(q + 1, bB, bA);
                }
            } else {
                for (int q = 0; q < nq; ++q) {
                    if ((q & vmask) == 0) acc_wait();
                    float scale, nz;
                    group_params(gl, scale, nz);
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        float b[BUF], sv[CH];
                        load_S(gl, c, sv);
                        load_acc(q, c, b);
                        tmem_wait_ld();
                        fold(gl, c, b, sv, scale, nz);
                    }
                    if ((q & vmask) == vmask || q == nq - 1) acc_free();
                    next_group();
                }
            }
            // this warp no longer reads the stage
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
            ps.next(S);
        }

        gemm_finish(a, blk, ok, pend0, pend1, mark_old, mt, NEPI * 32, 1);
    } else {
        // ------------------------------------------- activation producer ---
        if (lane == 0) gemm_act_producer(a, blk);
    }

    // every role is done with TMEM (the MMA issuer waited for its last
    // commit; the epilogue warps waited for every slot they read)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, TMEM_COLS);
}

// Launch one instance.
template <int FMT, int MT, bool E4, bool EXACT>
cudaError_t launch_gemm_instance(const GemmArgs &a, bool pdl, cudaStream_t s) {
    auto kern = k_verify_gemm<FMT, MT, E4, EXACT>;
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

template <int FMT, bool EXACT>
cudaError_t launch_gemm_mode(const GemmArgs &a, bool pdl, cudaStream_t s) {
    const int mt = act_rows(a.M);
    if constexpr (FMT == HQ_W4_ASYM) {
        // the digit-encoded operand up to 32 rows goes to the register-resident kernel
        if (act_e4(FMT, a.M, a.G)) return launch_gemm_instance<FMT, 64, true, EXACT>(a, pdl, s);
    }
    switch (mt) {
        case 16: return launch_gemm_instance<FMT, 16, false, EXACT>(a, pdl, s);
        case 32: return launch_gemm_instance<FMT, 32, false, EXACT>(a, pdl, s);
        case 64: return launch_gemm_instance<FMT, 64, false, EXACT>(a, pdl, s);
        default: return launch_gemm_instance<FMT, 128, false, EXACT>(a, pdl, s);
    }
}

template <int FMT>
cudaError_t launch_gemm_fmt(const GemmArgs &a, bool pdl, cudaStream_t s) {
    // check mode and exact-order mode: the oracle's rounding of every step
    return a.partials || a.nb_align ? launch_gemm_mode<FMT, true>(a, pdl, s) : launch_gemm_mode<FMT, false>(a, pdl, s);
}

cudaError_t launch_gemm_w4(const GemmArgs &a, bool pdl, cudaStream_t s);
cudaError_t launch_gemm_w8(const GemmArgs &a, bool pdl, cudaStream_t s);
// register-resident kernel: 4-bit weights, fp16-encoded operand, up to 32 rows
cudaError_t launch_gemm_w4_rs(const GemmArgs &a, bool pdl, cudaStream_t s);
cudaError_t launch_gemm_w8_rs(const GemmArgs &a, bool pdl, cudaStream_t s);

}  // namespace hq
