// gemm_common.cuh -- what the verify GEMM's kernels share: the launch
// arguments, the stream-K work split, the two producers that stream weight
// tiles and activation K tiles into a ring of shared-memory stages, and the
// combination of outputs whose K range is split between thread blocks.
//
// Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
// section "Why batch-one decoding is memory-bound": the verify pass streams
// every weight once, so the kernels are organised around that stream.
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
// Pipeline unit: U consecutive tiles of the block's range.  A stage holds a
// unit's U weight tiles, then its U activation K tiles (codes and group
// sums), each copied by its own producer warp with one bulk copy per run:
// a bulk copy holds up the warp that issues it, and the weight stream must
// not wait behind the activation copies.  A stage's `full` barrier completes
// once both producers' bytes have landed.  An SM serves its bulk copies in the
// order they are issued, so while the ring first fills, unit u's weights go
// out only after unit u - 1's activations: the first units land first
// instead of behind the whole ring's weights.
#pragma once

#include <cuda_runtime.h>

#include "hq_internal.cuh"

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
    int act_off;     // offset of the activation K tiles within a stage (after U weight tiles)
    int act_bytes;   // codes of one activation K tile: (KT/128) * MT * 256
    int s_bytes;     // group sums of one activation K tile: GPT * MT * 4
    int act_tile_bytes;  // one activation K tile: codes, then group sums
    int stage_bytes; // one unit: U weight tiles, then their U activation K tiles
};

// Accumulating mode: added (with the zeroing block's own arrival, + 1) to a
// split n-block's counter once its outputs are zero; above any count of
// arrivals (at most MAX_CTAS blocks).
constexpr int ZERO_MARK = 1 << 24;

constexpr int MAX_STAGES = 32;
// register-resident GEMM: tiles per pipeline unit, MMA row tiles (16
// channels) per consumer warp, thread blocks per SM for MT token rows.
// Units of one tile: a block's consumers start on its first tile as soon as
// that tile is in, and the ring holds more, smaller stages (verify pass 2.204
// -> 2.145 ms against units of two).
// Three blocks of one producer and four 32-channel consumer warps at 16 rows:
// twelve consumer warps per SM hide the MMA and shared-memory latencies, and
// an SM frees a third of its room for the next kernel of the stream as soon
// as one of its blocks ends.  At 32 rows the sums of a warp need more than
// the 128 registers a thread has at three blocks: two blocks.
constexpr int RS_UNIT = 1;
constexpr int RS_RT = 2;
__host__ __device__ constexpr int rs_bps(int MT) { return MT <= 16 ? 3 : 2; }
constexpr int GEMM_SMEM_LIMIT = 227 * 1024;   // opt-in maximum of dynamic shared memory per block

// floor(x * y / z) for 0 <= x <= MAX_CTAS (or a tile index), y, z > 0: in
// 32-bit arithmetic while the product fits (every layer below 2^23 tiles),
// the 64-bit division (a long instruction sequence) otherwise.
__device__ __forceinline__ int muldiv(int x, int y, int z) {
    const long long p = (long long)x * y;
    return p < (1LL << 31) ? (int)((unsigned)p / (unsigned)z) : (int)(p / z);
}
__device__ __forceinline__ int tile_begin(int c, int T, int grid) { return muldiv(c, T, grid); }
// first tile of thread block c (c = grid: one past the last tile)
__device__ __forceinline__ int range_begin(const GemmArgs &a, int c) {
    return a.nb_align ? muldiv(c, a.NB, a.grid) * a.KTILES : tile_begin(c, a.T, a.grid);
}
// thread block whose range contains tile t
__device__ __forceinline__ int cta_of_tile(int t, int T, int grid) {
    const long long p = ((long long)t + 1) * grid - 1;
    return p < (1LL << 31) ? (int)((unsigned)p / (unsigned)T) : (int)(p / T);
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

// What a thread block knows about its share of the work and its stage ring.
struct GemmBlock {
    int t0, t1, ntl, nunits, U, S, KTILES;
    bool det;     // deterministic combination of split n-blocks
    bool zeroer;  // accumulating mode: this block zeroes n-block zb's outputs
    int zb;
    int *err;     // workspace error word
    int *ctr;     // n-block counters
    uint8_t *ring;
    uint64_t *full, *empty;
    int *sflag;   // accumulating mode: the block's two segment flags
    int *acts_issued;  // units whose activation copies have been issued (initial fill)
    __device__ __forceinline__ int unit_tiles(int u) const { return ntl - u * U < U ? ntl - u * U : U; }
};

__device__ __forceinline__ GemmBlock make_gemm_block(const GemmArgs &a, uint8_t *ring, uint64_t *full, uint64_t *empty,
                                                     int *sflag) {
    GemmBlock b;
    b.t0 = range_begin(a, blockIdx.x);
    b.t1 = range_begin(a, blockIdx.x + 1);
    b.ntl = b.t1 - b.t0;
    b.U = a.U;
    b.S = a.stages;
    b.nunits = (b.ntl + b.U - 1) / b.U;
    b.KTILES = a.KTILES;
    b.det = a.det != 0;
    // Accumulating mode: this block holds K tile 0 of n-block zb and another
    // block holds its last K tile -> this block zeroes zb's outputs.
    b.zb = (b.t1 - 1) / b.KTILES;
    b.zeroer = !b.det && b.ntl > 0 && b.zb * b.KTILES >= b.t0 && (b.zb + 1) * b.KTILES > b.t1;
    b.err = reinterpret_cast<int *>(a.ws);
    b.ctr = reinterpret_cast<int *>(a.ws + ws_counter_offset());
    b.ring = ring;
    b.full = full;
    b.empty = empty;
    b.sflag = sflag;
    b.acts_issued = sflag + 2;
    return b;
}

// Weight producer (one lane).  One bulk copy per unit: its tiles are
// consecutive in the blob.  The copies that fill the ring go out before
// waiting for the previous kernel of the stream (the blob is not its output).
__device__ __forceinline__ void gemm_weight_producer(const GemmArgs &a, const GemmBlock &b) {
    const uint64_t pol_w = policy_evict_first();
    const int S = b.S;
    auto copy_weights = [&](int u, int st) {
        const uint32_t fb = smem_addr(&b.full[st]);
        const int nt = b.unit_tiles(u);
        mbar_arrive_expect_tx(fb, (uint32_t)(nt * a.tile_bytes));
        bulk_copy_g2s(smem_addr(b.ring + (size_t)st * a.stage_bytes),
                      a.blob + (size_t)(b.t0 + u * b.U) * (size_t)a.tile_bytes, (uint32_t)(nt * a.tile_bytes), fb, pol_w);
    };
    int u = 0;
    if (b.nunits > 0) copy_weights(u++, 0);
    pdl_wait();
    // the rest of the initial fill: unit u's weights after unit u - 1's activations
    for (; u < b.nunits && u < S; ++u) {
        if (!wait_count_shared_bounded(smem_addr(b.acts_issued), u, b.err)) break;
        copy_weights(u, u);
    }
    RingPos ps{u % S, (uint32_t)((u / S) & 1)};
    for (; u < b.nunits; ++u) {
        const int st = ps.slot;
        if (!mbar_wait_bounded(smem_addr(&b.empty[st]), ps.phase ^ 1u, b.err)) break;
        copy_weights(u, st);
        ps.next(S);
    }
    // No copy may still be landing in shared memory when the block exits (a
    // stage's phase completes once both producers' copies have landed).
    const int issued = u;
    for (int j = issued > S ? issued - S : 0; j < issued; ++j)
        mbar_wait_bounded(smem_addr(&b.full[j % S]), (uint32_t)((j / S) & 1), b.err);
}

// Activation producer (one lane).  One bulk copy per run of consecutive K
// tiles (one per unit unless the unit crosses the end of an n-block's K
// range).
//
// Accumulating mode: after the copies of a tile that ends a split segment,
// count this block into the n-block's counter (acquire), wait until the
// zeroing mark is in (or the counter was reset, which happens only after the
// mark), reset the counter if this count completes it, and raise the
// segment's flag for the consumers (release, CTA scope).  The zeroing block's
// own n-block needs neither: its mark carries its count, and its consumers
// zeroed before a barrier.  Every access to a counter is a read-modify-write,
// so the reset continues the mark's release sequence and a wait that reads it
// acquires the zeroing.
__device__ __forceinline__ void gemm_act_producer(const GemmArgs &a, const GemmBlock &b) {
    pdl_wait();
    const uint64_t pol_a = policy_evict_last();
    const int KTILES = b.KTILES;
    auto copy_acts = [&](int u, int st) {
        uint8_t *dst = b.ring + (size_t)st * a.stage_bytes + a.act_off;
        const uint32_t fb = smem_addr(&b.full[st]);
        const int nt = b.unit_tiles(u);
        mbar_arrive_expect_tx(fb, (uint32_t)(nt * a.act_tile_bytes));
        for (int j = 0; j < nt;) {
            const int kt = (b.t0 + u * b.U + j) % KTILES;
            const int run = nt - j < KTILES - kt ? nt - j : KTILES - kt;
            bulk_copy_g2s(smem_addr(dst + (size_t)j * a.act_tile_bytes), a.qop + (size_t)kt * a.act_tile_bytes,
                          (uint32_t)(run * a.act_tile_bytes), fb, pol_a);
            j += run;
        }
    };
    int nsplit = 0;
    auto check = [&](int j) {
        const int t = b.t0 + j, bb = t / KTILES, kb = t - bb * KTILES;
        if (!((kb == KTILES - 1 || j == b.ntl - 1) && !(bb * KTILES >= b.t0 && kb == KTILES - 1))) return;
        if (!(b.zeroer && bb == b.zb)) {
            const int nc = cta_of_tile(bb * KTILES + KTILES - 1, a.T, a.grid) - cta_of_tile(bb * KTILES, a.T, a.grid) + 1;
            const int v = atom_add_acquire_gpu(&b.ctr[bb], 1);
            if (v < ZERO_MARK) wait_mark_bounded(&b.ctr[bb], ZERO_MARK, v + 1, b.err, a.wait_ns);
            if (v == ZERO_MARK + nc - 1) atomicExch(&b.ctr[bb], 0);
        }
        st_release_cta_shared(smem_addr(&b.sflag[nsplit]), 1);
        ++nsplit;
    };
    RingPos ps{0, 0u};
    for (int u = 0; u < b.nunits; ++u) {
        const int st = ps.slot;
        if (!mbar_wait_bounded(smem_addr(&b.empty[st]), ps.phase ^ 1u, b.err)) break;
        copy_acts(u, st);
        if (u < b.S) st_release_cta_shared(smem_addr(b.acts_issued), u + 1);
        if (!b.det)
            for (int j = 0; j < b.unit_tiles(u); ++j) check(u * b.U + j);
        ps.next(b.S);
    }
}

// Both streams from one lane: the weight copies of the first `prefetch` units
// before waiting for the previous kernel of the stream, their activation
// copies after it, then unit by unit as stages free up: the unit's weights,
// then its activations (one copy per run of consecutive K tiles).  Split
// segments are counted as in gemm_act_producer.
__device__ __forceinline__ void gemm_producer(const GemmArgs &a, const GemmBlock &b, int prefetch) {
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    const int S = b.S, KTILES = b.KTILES;
    auto copy_weights = [&](int u, int st) {
        const uint32_t fb = smem_addr(&b.full[st]);
        const int nt = b.unit_tiles(u);
        mbar_arrive_expect_tx(fb, (uint32_t)(nt * a.tile_bytes));
        bulk_copy_g2s(smem_addr(b.ring + (size_t)st * a.stage_bytes),
                      a.blob + (size_t)(b.t0 + u * b.U) * (size_t)a.tile_bytes, (uint32_t)(nt * a.tile_bytes), fb, pol_w);
    };
    auto copy_acts = [&](int u, int st) {
        uint8_t *dst = b.ring + (size_t)st * a.stage_bytes + a.act_off;
        const uint32_t fb = smem_addr(&b.full[st]);
        const int nt = b.unit_tiles(u);
        mbar_arrive_expect_tx(fb, (uint32_t)(nt * a.act_tile_bytes));
        for (int j = 0; j < nt;) {
            const int kt = (b.t0 + u * b.U + j) % KTILES;
            const int run = nt - j < KTILES - kt ? nt - j : KTILES - kt;
            bulk_copy_g2s(smem_addr(dst + (size_t)j * a.act_tile_bytes), a.qop + (size_t)kt * a.act_tile_bytes,
                          (uint32_t)(run * a.act_tile_bytes), fb, pol_a);
            j += run;
        }
    };
    int nsplit = 0;
    auto check = [&](int j) {
        const int t = b.t0 + j, bb = t / KTILES, kb = t - bb * KTILES;
        if (!((kb == KTILES - 1 || j == b.ntl - 1) && !(bb * KTILES >= b.t0 && kb == KTILES - 1))) return;
        if (!(b.zeroer && bb == b.zb)) {
            const int nc = cta_of_tile(bb * KTILES + KTILES - 1, a.T, a.grid) - cta_of_tile(bb * KTILES, a.T, a.grid) + 1;
            const int v = atom_add_acquire_gpu(&b.ctr[bb], 1);
            if (v < ZERO_MARK) wait_mark_bounded(&b.ctr[bb], ZERO_MARK, v + 1, b.err, a.wait_ns);
            if (v == ZERO_MARK + nc - 1) atomicExch(&b.ctr[bb], 0);
        }
        st_release_cta_shared(smem_addr(&b.sflag[nsplit]), 1);
        ++nsplit;
    };
    int u = 0;
    for (; u < b.nunits && u < S && u < prefetch; ++u) copy_weights(u, u);
    pdl_wait();
    for (int v = 0; v < u; ++v) {
        copy_acts(v, v);
        if (!b.det)
            for (int j = 0; j < b.unit_tiles(v); ++j) check(v * b.U + j);
    }
    RingPos ps{u % S, (uint32_t)((u / S) & 1)};
    for (; u < b.nunits; ++u) {
        const int st = ps.slot;
        if (!mbar_wait_bounded(smem_addr(&b.empty[st]), ps.phase ^ 1u, b.err)) break;
        copy_weights(u, st);
        copy_acts(u, st);
        if (!b.det)
            for (int j = 0; j < b.unit_tiles(u); ++j) check(u * b.U + j);
        ps.next(S);
    }
    // no copy may still be landing in shared memory when the block exits
    const int issued = u;
    for (int j = issued > S ? issued - S : 0; j < issued; ++j)
        mbar_wait_bounded(smem_addr(&b.full[j % S]), (uint32_t)((j / S) & 1), b.err);
}

// Accumulating mode, zeroing block: its consumer threads (tid of nthr, named
// barrier bar) zero n-block zb's outputs, then thread 0 adds the mark and the
// block's own arrival (release).  Returns the counter before the mark
// (thread 0; read after the last tile by gemm_finish).
__device__ __forceinline__ int gemm_zero_outputs(const GemmArgs &a, const GemmBlock &b, int tid, int nthr, int bar) {
    int mark_old = 0;
    if (b.zeroer) {
        for (int q = tid; q < a.M * BN; q += nthr) {
            const int tok = q / BN, nn = b.zb * BN + (q - tok * BN);
            if (nn < a.N) a.Y[(size_t)tok * a.N + nn] = 0.0f;
        }
        named_barrier(bar, nthr);
        if (tid == 0) mark_old = atom_add_release_gpu(&b.ctr[b.zb], ZERO_MARK + 1);
    }
    return mark_old;
}

// After the block's last tile, on its consumer threads (tid of nthr, named
// barrier bar).  Accumulating mode: if every other contributor of zb counted
// before the mark, the mark completed the count and this block resets the
// counter.  Deterministic mode, split n-blocks (pend0: the block's first
// n-block, published in slot 0; pend1: its last, slot 1; -1 if none):
// every contributor arrives, waits until all contributors of the n-block have
// arrived, then sums its 1/nc share of the n-block's outputs over all
// contributors' partial sums in ascending K order (slot 0 of a contributor is
// its first segment, slot 1 its last), multiplies by the row scale and writes
// Y.  The wait is safe because every thread block of the launch is resident:
// the grid never exceeds the SMs (one block per SM), and dependent kernels are
// launched only after every block of this one has started.  The last
// contributor to finish resets the n-block's two counters for the next call.
// Threads 0 and 1 serve the two pending n-blocks at the same time.
__device__ __forceinline__ void gemm_finish(const GemmArgs &a, const GemmBlock &b, bool ok, int pend0, int pend1,
                                            int mark_old, int tid, int nthr, int bar) {
    const int KTILES = b.KTILES;
    int *ctr = b.ctr;
    if (b.zeroer && tid == 0) {
        const int nc = cta_of_tile(b.zb * KTILES + KTILES - 1, a.T, a.grid) - cta_of_tile(b.zb * KTILES, a.T, a.grid) + 1;
        if (mark_old == nc - 1) atomicExch(&ctr[b.zb], 0);
    }
    if (pend0 < 0 && pend1 < 0) return;
    const float *wsp = reinterpret_cast<const float *>(a.ws + ws_partial_offset());
    int *done = ctr + a.NB;
    // every consumer thread's partial-sum stores precede the arrivals
    named_barrier(bar, nthr);
    int my_bb = -1, my_nc = 0, done_before = 0;
    if (tid < 2) {
        my_bb = tid == 0 ? pend0 : pend1;
        if (my_bb >= 0) {
            my_nc = cta_of_tile(my_bb * KTILES + KTILES - 1, a.T, a.grid) - cta_of_tile(my_bb * KTILES, a.T, a.grid) + 1;
            red_add_release_gpu(&ctr[my_bb], 1);
            if (ok) ok = wait_count_bounded(&ctr[my_bb], my_nc + a.wait_extra, b.err, a.wait_ns);
            // passed the wait: count it now, the answer arrives during the sums
            done_before = atomicAdd(&done[my_bb], 1);
        }
    }
    // the acquires of threads 0 and 1 are ordered before every thread's loads below
    named_barrier(bar, nthr);
    // Shares of both pending n-blocks as one list of 4-channel output groups
    // (n0 from the first, then the second); two groups per iteration, with all
    // their loads in flight together.
    const int total = a.M * (BN / 4);
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
        // Every contributor after the first starts inside this n-block, so it
        // is their first n-block (slot 0); the first contributor used slot 1
        // if it started in an earlier n-block.
        e_slot[p] = tile_begin(c_lo, a.T, a.grid) < bb * KTILES ? 1 : 0;
    }
    const int n_all = e_cnt[0] + e_cnt[1];
    for (int base = 0; base < n_all; base += 2 * nthr) {
        float4 sum[2];
        int gis[2], ps[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int idx = base + hh * nthr + tid;
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
                        x[hh][v] = __ldcg(reinterpret_cast<const float4 *>(wsp + ((size_t)c2 * 2 + sl) * ws_slot_floats() +
                                                                           (size_t)gis[hh] * 4));
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
            float *yr = a.Y + (size_t)tok * a.N;
            if (nn + 0 < a.N) yr[nn + 0] = __fmul_rn(sxt, sum[hh].x);
            if (nn + 1 < a.N) yr[nn + 1] = __fmul_rn(sxt, sum[hh].y);
            if (nn + 2 < a.N) yr[nn + 2] = __fmul_rn(sxt, sum[hh].z);
            if (nn + 3 < a.N) yr[nn + 3] = __fmul_rn(sxt, sum[hh].w);
        }
    }
    // every contributor has passed its wait once all have counted
    if (my_bb >= 0 && done_before == my_nc - 1) {
        atomicExch(&ctr[my_bb], 0);
        atomicExch(&done[my_bb], 0);
    }
}

// One output of a segment that ends (the block's partial or full sum y of
// output (tok, nn)), written by the consumer thread that holds it:
//  - full: the segment is the n-block's whole K range -> Y = sx * y;
//  - deterministic split: published in the block's slot (first or last
//    n-block) for gemm_finish;
//  - accumulating split: Y += sx * y once the zeroing is visible (the caller
//    waited for the segment's flag).
enum SegKind { SEG_FULL = 0, SEG_PUBLISH = 1, SEG_ADD = 2 };
__device__ __forceinline__ void gemm_segment_out(const GemmArgs &a, int kind, float *slot_base, int tok, int nl, int nn,
                                                 float y) {
    if (tok >= a.M) return;
    if (kind == SEG_PUBLISH) {
        __stcg(slot_base + (size_t)tok * BN + nl, y);
    } else if (nn < a.N) {
        const float v = __fmul_rn(__ldg(a.sx + tok), y);
        if (kind == SEG_FULL)
            a.Y[(size_t)tok * a.N + nn] = v;
        else
            atomicAdd(a.Y + (size_t)tok * a.N + nn, v);
    }
}

}  // namespace hq
