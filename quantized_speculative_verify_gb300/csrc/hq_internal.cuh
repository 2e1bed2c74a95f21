// hq_internal.cuh -- blob geometry and device helpers shared by the kernels
// of the quantized speculative-verify linear layer (sm_103a).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/hq.h"

namespace hq {

// ---------------------------------------------------------------------------
// Packed weight blob.
//
// The weights of a layer are cut into tiles of BN = 128 output channels by
// KT input features (KT = max(128, group)).  Tiles are stored n-block major,
// K minor, so the tiles one thread block streams are one contiguous byte
// range and one bulk copy fetches a whole tile.  Inside a tile, with
// channel n = 0..127 and 64-feature chunk c = 0..KT/64-1:
//
//   codes   4-bit: [c][quarter p 0..1][n][16 bytes]: the 32 features
//           64c + 32p .. +31 of channel n as four 32-bit words of eight
//           nibbles; nibble i of word t (bits 4i..4i+3) holds feature
//           2t + 8i and nibble i + 4 feature 2t + 8i + 1, i = 0..3.  Word t
//           is then exactly what lane t of a quad needs for two 16-feature
//           MMA steps of one channel (feature pairs 2t, 2t+1 and 2t+8, 2t+9
//           of each step), and one mask (after a shift by 8 for the second
//           step) lifts each pair into the two halves of a 32-bit register.
//           8-bit: [c][quarter p 0..3][n][16 bytes]: the 16 features
//           64c + 16p .. of channel n as four words, word t holding features
//           2t, 2t+1, 2t+8, 2t+9 (bytes 0..3): lane t of a quad's A operand
//           for one 16-feature MMA step.
//           A tcgen05 widening thread owns one channel and reads 16 contiguous
//           bytes per quarter (the 32 lanes of a warp: 512 contiguous bytes);
//           an MMA lane reads the one word of its quad position.
//   scales  [n][group in tile] fp32
//   zeros   4-bit only: nibble n * GPT + g (low nibble first), uint4
//
// Every region and every tile is a multiple of 16 bytes, and the byte count
// of a tile equals its algorithmic size: BN*KT*(bits/8) for the codes plus
// 4 bytes (and half a byte for the zero point) per (channel, group).
// N and K are padded up to whole tiles with zero codes and zero scales.
// ---------------------------------------------------------------------------
constexpr int BN = 128;           // output channels per tile (= TMEM lanes)
constexpr int MAX_CTAS = 480;     // upper bound on GEMM thread blocks (up to three per SM; workspace sizing)
constexpr int MAX_M = HQ_MAX_M;

struct Geom {
    int K, N, G, fmt;
    int KT;          // features per tile
    int Kp;          // K rounded up to KT
    int NB;          // n-blocks (tiles along N)
    int KTILES;      // tiles along K
    int GPT;         // groups per tile
    int NGK;         // real groups along K (K / G)
    int code_bytes;  // per tile
    int scale_bytes; // per tile
    int zero_bytes;  // per tile
    int tile_bytes;
};

__host__ __device__ inline bool desc_valid(int K, int N, int G, int fmt) {
    if (K <= 0 || N <= 0) return false;
    if (K % 32 != 0) return false;
    if (!(G == 16 || G == 32 || G == 64 || G == 128 || G == 256)) return false;
    if (K % G != 0) return false;
    if (fmt != HQ_W4_ASYM && fmt != HQ_W8_SYM) return false;
    return true;
}

// Largest K a layer may have: the activation operand's limit (a row of X is
// rotated and quantized by one thread block), and far below the int range of
// the tile arithmetic (K + KT - 1 stays positive).
constexpr int MAX_K = 65536;

// A valid layer whose tile count fits the kernels' int tile indices (at most
// 2^30 tiles of 128 channels x max(128, group) features) and whose K is at
// most MAX_K.  Every entry point that takes a layer descriptor checks this
// before computing any geometry.
inline bool desc_ok(const hq_layer_desc *d) {
    if (!d || !desc_valid(d->K, d->N, d->group, d->format)) return false;
    if (d->K > MAX_K) return false;
    const long long kt = d->group > 128 ? d->group : 128;
    const long long tiles = ((long long)d->N + BN - 1) / BN * (((long long)d->K + kt - 1) / kt);
    return tiles <= (1LL << 30);
}

__host__ __device__ inline Geom make_geom(int K, int N, int G, int fmt) {
    Geom g;
    g.K = K;
    g.N = N;
    g.G = G;
    g.fmt = fmt;
    g.KT = G > 128 ? G : 128;
    g.Kp = (K + g.KT - 1) / g.KT * g.KT;
    g.NB = (N + BN - 1) / BN;
    g.KTILES = g.Kp / g.KT;
    g.GPT = g.KT / G;
    g.NGK = K / G;
    g.code_bytes = fmt == HQ_W4_ASYM ? BN * g.KT / 2 : BN * g.KT;
    g.scale_bytes = g.GPT * BN * 4;
    g.zero_bytes = fmt == HQ_W4_ASYM ? g.GPT * BN / 2 : 0;
    g.tile_bytes = g.code_bytes + g.scale_bytes + g.zero_bytes;
    return g;
}

__host__ __device__ inline size_t blob_bytes(const Geom &g) {
    return (size_t)g.NB * (size_t)g.KTILES * (size_t)g.tile_bytes;
}

// Workspace: [0, 16) error word; then the partial-sum slots, two per thread
// block, BN x MAX_M floats each (a call fills its first M rows); then two
// counters per n-block (arrivals [NB], then finished reductions [NB]).
// Every offset is independent of the layer and of M, so one workspace, large
// enough for each call, serves calls of any shape in turn.
__host__ __device__ inline size_t ws_slot_floats() { return (size_t)BN * (size_t)MAX_M; }
__host__ __device__ inline size_t ws_partial_offset() { return 16; }
__host__ __device__ inline size_t ws_counter_offset() {
    return ws_partial_offset() + (size_t)MAX_CTAS * 2 * ws_slot_floats() * 4;
}
__host__ __device__ inline size_t ws_counter_bytes(const Geom &g) { return ((size_t)g.NB * 8 + 15) / 16 * 16; }
__host__ __device__ inline size_t ws_bytes(const Geom &g) { return ws_counter_offset() + ws_counter_bytes(g); }

// Activation operand of the GEMM (private to the library).  Rows are padded
// to MT = 16, 32, 64 or 128 (the MMA's N); rows past M and features past K
// are zero.  It is a sequence of K tiles of KT = max(G, 128) features (the
// weight blob's K tiles), each holding what one weight tile's MMAs and
// epilogue read, so that a run of consecutive K tiles is one contiguous copy:
//   codes, KT / 128 blocks of 128 features, in one of three encodings
//   chosen by the GEMM that reads the operand (act_rs, act_e4):
//     fp16 rows (act_rs: the register-resident GEMM, 4-bit weights, up to
//             32 rows): [MT rows][128 fp16 + 16 bytes of padding]: a row of
//             272 bytes puts the 16-byte chunk c of the 8 rows of an
//             ldmatrix in 8 distinct bank quads (272 = 256 + 16), and the
//             activation kernel writes each row's 256 bytes in one run;
//     fp16:   [16 chunks of 8 features][MT rows][8 fp16] (exact for
//             |q| <= 127), the B operand of kind::f16 MMAs;
//     digits: [8 chunks of 16 features][2 MT rows][16 e4m3]: q = 16 h + l
//             with l in [-8, 7], h in [-8, 8], both exact in e4m3; row r < MT
//             holds the l of token r, row MT + r its h: the B operand of
//             kind::f8f6f4 MMAs whose N covers both digits;
//   the last two are the B operand of a tile's tcgen05 MMAs as 8-row x
//   16-byte core matrices (K-major, no swizzle), MT * 256 bytes; then, where the
//   consuming GEMM needs them (act_sums),
//   group sums [KT / G groups][MT] fp32: S[g][m] = sum of the int8 codes of
//   row m over the tile's group g (zero past K).
constexpr int ACT_BLOCK = 128;
__host__ __device__ inline int act_rows(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }
// The digit encoding: 4-bit weights (their codes are e4m3 bytes as they are)
// on the tensor-memory GEMM, rows that fit an MMA of N = 2 MT <= 128 (33 to
// 64 rows; up to 32 rows the register-resident GEMM takes the fp16
// encoding), and groups of at least 32 features (one f8f6f4 MMA covers 32).
__host__ __device__ inline bool act_e4(int fmt, int M, int G) {
    return fmt == HQ_W4_ASYM && act_rows(M) > 32 && act_rows(M) <= 64 && G >= 32;
}
__host__ __device__ inline int act_blocks(int K) { return (K + ACT_BLOCK - 1) / ACT_BLOCK; }
__host__ __device__ inline int act_kt(int G) { return G > ACT_BLOCK ? G : ACT_BLOCK; }
__host__ __device__ inline int act_ktiles(int K, int G) { return (K + act_kt(G) - 1) / act_kt(G); }
// Whether the operand carries the group sums: only the GEMM that applies a
// 4-bit layer's zero point through them (the tensor-memory GEMM, above 32
// rows).  Up to 32 rows the register-resident GEMM subtracts the zero point
// while widening the weights; 8-bit weights have none.
__host__ __device__ inline bool act_sums(int fmt, int M) { return fmt == HQ_W4_ASYM && act_rows(M) > 32; }
// The row encoding: the operand of the register-resident GEMM (every
// format, up to 32 rows).
__host__ __device__ inline bool act_rs(int fmt, int M) { return (fmt == HQ_W4_ASYM || fmt == HQ_W8_SYM) && act_rows(M) <= 32; }
constexpr int ACT_RS_PITCH = 272;  // bytes per row of a 128-feature block in the row encoding
// bytes of one 128-feature block's codes, of one K tile's codes, of its group
// sums, and of the whole K tile
__host__ __device__ inline int act_block_bytes(int M, int fmt) { return act_rows(M) * (act_rs(fmt, M) ? ACT_RS_PITCH : 256); }
__host__ __device__ inline int act_tile_code_bytes(int M, int G, int fmt) { return (act_kt(G) / ACT_BLOCK) * act_block_bytes(M, fmt); }
__host__ __device__ inline int act_tile_sum_bytes(int M, int G, int fmt) {
    return act_sums(fmt, M) ? (act_kt(G) / G) * act_rows(M) * 4 : 0;
}
__host__ __device__ inline int act_tile_bytes(int M, int G, int fmt) {
    return act_tile_code_bytes(M, G, fmt) + act_tile_sum_bytes(M, G, fmt);
}
__host__ __device__ inline size_t act_operand_bytes(int M, int K, int G, int fmt) {
    return (size_t)act_ktiles(K, G) * (size_t)act_tile_bytes(M, G, fmt);
}

// Device error codes written to the workspace error word.
constexpr int DEV_ERR_TIMEOUT = 1;
// Bounded waits give up after this long (normal waits last microseconds).
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;

// fp32 nearest to 1/sqrt(32): the overall scale of the Hadamard transform.
constexpr uint32_t HADAMARD_SCALE_BITS = 0x3E3504F3u;

// ---------------------------------------------------------------------------
// Device helpers (inline PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Test the phase; a thread whose phase is not complete is suspended by the
// hardware until the phase completes or about `hint_ns` elapse, so a waiting
// warp issues no instructions (polling would take issue slots from the warps
// that do the work).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns = 1000000u) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase (no suspension): the fast path of a wait
// whose phase has usually completed already.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with parity `parity` of barrier `bar` to complete, for
// at most `limit_ns`.  On time-out, records DEV_ERR_TIMEOUT in *err (if not
// NULL) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int *err,
                                                  unsigned long long limit_ns = WAIT_LIMIT_NS) {
    if (mbar_test_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    uint32_t it = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++it & 15u) == 0u && global_timer_ns() - t0 > limit_ns) {
            if (err) atomicExch(err, DEV_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// One-dimensional bulk copy global -> shared, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Add without returning the old value, release semantics at GPU scope.
__device__ __forceinline__ void red_add_release_gpu(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait until *p >= target (acquire), for at most WAIT_LIMIT_NS; polls with a
// short sleep in between.  On time-out records DEV_ERR_TIMEOUT in *err and
// returns false.
__device__ __forceinline__ bool wait_count_bounded(const int *p, int target, int *err,
                                                   unsigned long long limit_ns = WAIT_LIMIT_NS) {
    if (ld_acquire_gpu(p) >= target) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        __nanosleep(100);
        if (ld_acquire_gpu(p) >= target) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            if (err) atomicExch(err, DEV_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ int atom_add_acquire_gpu(int *p, int v) {
    int old;
    asm volatile("atom.acquire.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ int atom_add_release_gpu(int *p, int v) {
    int old;
    asm volatile("atom.release.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_release_cta_shared(uint32_t addr, int v) {
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_cta_shared(uint32_t addr) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Wait until the shared-memory word at addr is at least target (acquire, CTA
// scope), for at most WAIT_LIMIT_NS.  On time-out records DEV_ERR_TIMEOUT in
// *err and returns false.
__device__ __forceinline__ bool wait_count_shared_bounded(uint32_t addr, int target, int *err) {
    if (ld_acquire_cta_shared(addr) >= target) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        __nanosleep(32);
        if (ld_acquire_cta_shared(addr) >= target) return true;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
            if (err) atomicExch(err, DEV_ERR_TIMEOUT);
            return false;
        }
    }
}

// Wait until the shared-memory word at addr is non-zero (acquire, CTA scope),
// for at most WAIT_LIMIT_NS.  On time-out records DEV_ERR_TIMEOUT in *err and
// returns false.
__device__ __forceinline__ bool wait_flag_bounded(uint32_t addr, int *err) {
    if (ld_acquire_cta_shared(addr) != 0) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        __nanosleep(32);
        if (ld_acquire_cta_shared(addr) != 0) return true;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
            if (err) atomicExch(err, DEV_ERR_TIMEOUT);
            return false;
        }
    }
}

// Wait until *p >= mark, or until *p has fallen below `own` (the counter was
// reset, which happens only after the mark was added), for at most
// WAIT_LIMIT_NS; acquire.  On time-out records DEV_ERR_TIMEOUT in *err and
// returns false.
__device__ __forceinline__ bool wait_mark_bounded(const int *p, int mark, int own, int *err,
                                                  unsigned long long limit_ns = WAIT_LIMIT_NS) {
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        const int v = ld_acquire_gpu(p);
        if (v >= mark || v < own) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            if (err) atomicExch(err, DEV_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(64);
    }
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace hq

// Launchers (defined in the kernel translation units).
namespace hq {
cudaError_t launch_rotate_quant_act(const float *X, int M, int K, int G, bool rs, bool e4, bool sums, const uint32_t *signs, int8_t *qx,
                                    int32_t *gsum, uint8_t *qop, float *sx, bool pdl, cudaStream_t s);
cudaError_t launch_codes_to_operand(const int8_t *qx, int M, int K, int G, bool rs, bool e4, bool sums, uint8_t *qop,
                                    bool pdl, cudaStream_t s);
// rows of W -> n-blocks nb0.. of the blob of layer g
cudaError_t launch_pack(const Geom &g, const float *W, int rows, int nb0, const uint32_t *signs, void *blob,
                        cudaStream_t s);
cudaError_t launch_unpack(const Geom &g, const void *blob, uint8_t *codes, float *scales, uint8_t *zeros,
                          cudaStream_t s);
// flags: HQ_LAUNCH_* of hq_verify_gemm; wait_extra / wait_ns: the bounded-wait
// self-test (0 / 0 = normal call).
cudaError_t launch_verify_gemm(const Geom &g, const void *blob, const uint8_t *qop, const float *sx, int M, float *Y,
                               int32_t *partials, void *workspace, uint32_t flags, cudaStream_t s,
                               int wait_extra = 0, long long wait_ns = 0);
cudaError_t launch_wait_selftest(void *workspace, long long limit_ns, cudaStream_t s);
// Draft-tree acceptance: ACCEPT_CHUNK logits per thread block of the argmax.
constexpr int ACCEPT_CHUNK = 8192;
int accept_chunks(int V);
cudaError_t launch_tree_accept(const float *logits, int M, int V, const int32_t *parent, const int32_t *tokens,
                               int32_t *g_out, int32_t *path, int32_t *n_accept, int32_t *bonus, void *workspace,
                               bool pdl, cudaStream_t s);
// Tree-masked verify attention and the accepted-path cache commit.
size_t attn_workspace_bytes(int Hkv);
cudaError_t launch_tree_attention(const void *q, const void *k, const void *v, int cap, int L, int M, int Hq, int Hkv,
                                  const int32_t *parent, float scale, float *out, void *workspace, bool pdl,
                                  cudaStream_t s);
cudaError_t launch_tree_commit_kv(void *k, void *v, int cap, int L, int M, int Hkv, const int32_t *path,
                                  const int32_t *n_accept, bool pdl, cudaStream_t s);
// Rollback-free DeltaNet tree pass and the accepted-path state commit.
cudaError_t launch_delta_tree(const float *state, const float *q, const float *k, const float *v, const float *alpha,
                              const float *beta, const int32_t *parent, int M, int H, float *out, bool pdl,
                              cudaStream_t s);
cudaError_t launch_delta_commit(float *state, const float *k, const float *v, const float *alpha, const float *beta,
                                const int32_t *path, const int32_t *n_accept, int M, int H, bool pdl, cudaStream_t s);
int device_sm_count();

// Per-device results of one-time launch set-up (function attributes,
// occupancy), safe to use from several host threads at once.  cache[dev]
// holds value + 1 once known (0: not yet); devices >= CACHE_DEVICES are not
// cached.  compute(int *out) returns a cudaError_t and writes a non-negative
// value; concurrent first calls may both compute it, with the same result.
constexpr int CACHE_DEVICES = 64;
template <class F>
cudaError_t cached_per_device(std::atomic<int> (&cache)[CACHE_DEVICES], int dev, int *out, F compute) {
    const bool cached = dev >= 0 && dev < CACHE_DEVICES;
    if (cached) {
        const int c = cache[dev].load(std::memory_order_acquire);
        if (c > 0) {
            *out = c - 1;
            return cudaSuccess;
        }
    }
    int v = 0;
    const cudaError_t e = compute(&v);
    if (e != cudaSuccess) return e;
    if (cached) cache[dev].store(v + 1, std::memory_order_release);
    *out = v;
    return cudaSuccess;
}
}  // namespace hq
