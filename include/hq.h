/*
 * hq.h -- C ABI of the quantized speculative-verify linear layer for GB300
 * (sm_103a).
 *
 * The layer is the target model's linear layer in the verification pass of
 * speculative decoding: M drafted tree tokens (M = 1..128 rows) go through
 *   1. a block-diagonal randomized Hadamard rotation (blocks of 32, seeded
 *      +-1 sign flips, one overall scale 1/sqrt(32)) and per-row int8
 *      quantization of the activations, computed on the fly;
 *   2. an integer GEMM against weights that were rotated with the same
 *      transform and quantized offline, either to 4-bit asymmetric grouped
 *      integers ("Medium") or to 8-bit symmetric grouped integers ("Large");
 *   3. a per-group fp32 dequantization epilogue.
 * Source: page "Karpathy's Trick for Faster Local LLMs Finally Has Proper
 * Tooling" (blog.dailydoseofds.com): section "How Uzu optimizes bytes and
 * tokens per pass" (the two weight formats, 8-bit activations on the fly,
 * int8 matrix path, 32-block randomized Hadamard transform, transform block
 * independent of the quantization group) and section "Producing several
 * tokens from one model pass" (the verify batch is the 16-32 token draft
 * tree, "16 rows of work instead of 1").
 *
 * After the verify pass, the same library accepts the draft tree
 * (hq_tree_accept) and runs the two stateful layer kinds of the verified model
 * over the tree without changing their committed state, then commits the
 * accepted path: tree-masked attention over a KV cache (hq_tree_attention,
 * hq_tree_commit_kv) and the gated delta-rule DeltaNet layer (hq_delta_tree,
 * hq_delta_commit).  Source: the same page, section "Verifying a draft tree
 * without restoring model state".
 *
 * Conventions
 *   - Row-major everywhere.  X is [M][K], W is [N][K], Y = X W^T is [M][N].
 *   - Pointers are DEVICE pointers unless their name ends in _host.  The
 *     caller owns and allocates every buffer; the library allocates no
 *     memory and keeps no per-call state.
 *   - Every call that takes a `stream` (a cudaStream_t, NULL = legacy default
 *     stream) only enqueues work and returns without synchronizing.
 *   - Arguments are validated before anything is launched.  A call that
 *     returns an error launched nothing, except HQ_ERR_CUDA, which reports
 *     that the launch itself failed.  Faults of kernels that did launch show
 *     up, as always with CUDA, at the caller's next synchronization.
 *   - Calls are reentrant.  Two calls that share a workspace must not run
 *     concurrently (use one workspace per stream).
 */
#ifndef HQ_H
#define HQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HQ_OK = 0,
    HQ_ERR_INVALID_ARG = 1, /* NULL pointer, bad size, misaligned pointer   */
    HQ_ERR_UNSUPPORTED = 2, /* valid request the library does not implement */
    HQ_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed          */
    HQ_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up            */
} hq_status;

typedef enum {
    HQ_W4_ASYM = 0, /* "Medium": uint4 codes, fp32 scale + uint4 zero point per group */
    HQ_W8_SYM = 1   /* "Large":  int8 codes, fp32 scale per group                     */
} hq_format;

/* One linear layer.  K = input features (multiple of 32 and of `group`, at
 * most 65536), N = output features (>= 1), group = quantization group along
 * K, one of 16, 32, 64, 128, 256 (independent of the 32-element transform
 * block), format = hq_format.  The layer may have at most 2^30 weight tiles
 * of 128 output features x max(128, group) input features (a blob far larger
 * than any GPU memory); a descriptor beyond that is invalid. */
typedef struct {
    int32_t K;
    int32_t N;
    int32_t group;
    int32_t format;
} hq_layer_desc;

/* Launch flags. */
#define HQ_LAUNCH_DEFAULT 0u
/* Launch with programmatic dependent launch: the kernel may start while the
 * previous kernel of the stream is still running and waits for it (and for
 * its memory) before reading anything that kernel could have produced.
 * Some inputs are read before that wait, so with this flag they must not be
 * written by the operation launched immediately before in the same stream:
 * the blob (hq_verify_gemm streams the packed weights early), the committed
 * cache positions [0, L) (hq_tree_attention) and the committed state
 * (hq_delta_tree). */
#define HQ_LAUNCH_PDL 1u
/* hq_verify_gemm only: combine the thread blocks that share an output in a
 * fixed order, so that results repeat bit for bit from run to run (the blocks
 * wait for one another before that sum; slower).  Without it, their fp32
 * partial sums are added into Y atomically as each block finishes, and the
 * last bits of such outputs may differ between runs. */
#define HQ_LAUNCH_DETERMINISTIC 2u
/* hq_verify_gemm only: no output's K range is split between thread blocks:
 * each thread block takes whole blocks of 128 output channels, so every
 * output is summed over its groups in ascending order by one thread block,
 * each product scale * P rounded and then added (the definition's
 * arithmetic), and is bit-identical to the sequential fp32 sum of the
 * definition (see hq_verify_gemm).  Without this flag (and without check-mode
 * partials) a group is folded with one fused multiply-add, one rounding
 * fewer per group.  Slower on layers with few 128-channel blocks (fewer
 * thread blocks than SMs); implies HQ_LAUNCH_DETERMINISTIC. */
#define HQ_LAUNCH_EXACT_ORDER 4u

/* Maximum number of token rows per call. */
#define HQ_MAX_M 128

/* Human-readable name of a status code (static string, never NULL). */
const char *hq_status_string(int status);

/* ABI version of this library: (major << 16) | minor. */
int32_t hq_version(void);

/* Size in bytes of the packed weight blob of `desc` (0 if desc is invalid).
 * The blob layout is private to the library; hq_unpack_codes gives the
 * canonical view. */
size_t hq_packed_bytes(const hq_layer_desc *desc);

/* Size in bytes of the workspace hq_verify_gemm needs for `desc` and M rows
 * (0 if the arguments are invalid).  The workspace holds the device error
 * word, the split-K partial sums (two slots of 128 channels x 128 rows per
 * thread block, up to 480 blocks: 60 MiB) and two counters per 128 output
 * channels, at offsets
 * that depend on neither the layer nor M: one workspace of the largest size
 * serves calls of every layer and M in turn (calls that may overlap on the
 * GPU need workspaces of their own).  It must be zero-filled once after
 * allocation; every call leaves the error word and the counters at zero
 * again (except after a time-out, see hq_workspace_status); the partial sums
 * need no clearing. */
size_t hq_workspace_bytes(const hq_layer_desc *desc, int32_t M);

/* Sign vector of the randomized Hadamard transform ("random sign flips
 * applied before the mixing", section "How Uzu optimizes bytes and tokens
 * per pass").  Host-only.  Feature k is negated when the top bit of the k-th
 * output of SplitMix64 (Steele, Lea & Flood 2014) seeded with `seed` is set;
 * the result is bit-packed: bit (k % 32) of signs_host[k / 32].
 * K must be a positive multiple of 32; signs_host has K/32 words.  The same
 * vector must be used for the weights and for the activations of a layer. */
int hq_make_signs(uint64_t seed, int32_t K, uint32_t *signs_host);

/* Offline: rotate, quantize and pack the weights of one layer (section "How
 * Uzu optimizes bytes and tokens per pass": Medium = 4-bit asymmetric,
 * Large = 8-bit symmetric, transform before quantization).
 *   W      fp32 [N][K], 16-byte aligned
 *   signs  uint32 [K/32] (device copy of hq_make_signs' output)
 *   blob   hq_packed_bytes(desc) bytes, 16-byte aligned, written in full
 * Per (output channel n, group g): Medium: lo = min(0, min w), hi = max(0,
 * max w), scale = (hi - lo) / 15, zero = rint(-lo / scale), code =
 * clamp(rint(w / scale) + zero, 0, 15); Large: scale = max|w| / 127, code =
 * clamp(rint(w / scale), -127, 127); an all-zero group has scale 0 and
 * codes 0.  rint rounds half to even; divisions are IEEE. */
int hq_pack_weights(const hq_layer_desc *desc, const float *W, const uint32_t *signs, void *blob,
                    void *stream);

/* Offline, fused layers: pack `rows` rows of weights (fp32 [rows][K]) as the
 * output channels n0 .. n0 + rows - 1 of the layer `desc`, writing only the
 * blob's tiles of those channels.  Layers that read the same activations
 * (the q, k and v projections, or the gate and up projections) are packed
 * part by part into one blob of N = the sum of their widths and run as one
 * hq_verify_gemm; Y's columns n0 .. n0 + rows - 1 are that part's outputs,
 * identical to what the part alone would give (per output, the same
 * arithmetic).  n0 must be a multiple of 128, and the rows of the last part
 * may end anywhere before N; channels of the blob that no call packs are
 * left as they were.  Signs, formats and errors as in hq_pack_weights. */
int hq_pack_weights_at(const hq_layer_desc *desc, int32_t n0, int32_t rows, const float *W, const uint32_t *signs,
                       void *blob, void *stream);

/* Size in bytes of the GEMM's activation operand for M rows of the
 * activations of layers like `desc` (its K, group and format; N is not used),
 * 0 if the arguments are invalid or M = 0.  The operand is an opaque buffer
 * written by hq_rotate_quant_act and read by hq_verify_gemm of layers with the
 * same K, group and format; its layout is private to this version of the
 * library (it depends on the format and on M). */
size_t hq_act_operand_bytes(const hq_layer_desc *desc, int32_t M);

/* Verify pass, step 1: rotate and quantize the activations of M rows
 * (section "How Uzu optimizes bytes and tokens per pass": activations
 * quantized to 8 bits on the fly, after the same randomized Hadamard
 * transform as the weights).
 *   desc  the layers that read these activations: K (a multiple of 32, at
 *         most 65536), group (16, 32, 64, 128 or 256, dividing K) and format
 *         choose the operand's encoding; N is not used
 *   X     fp32 [M][K], 16-byte aligned, 0 <= M <= HQ_MAX_M (M = 0: no-op)
 *   signs uint32 [K/32]
 *   qx    int8 [M][K] (4-byte aligned) or NULL: clamp(rint(x' / sx), -127, 127)
 *   gsum  int32 [M][K/group] (4-byte aligned) or NULL: the sum of the codes
 *         qx over each group (the correction term of the Medium format:
 *         sum qx (q - z) = sum qx q - z * gsum)
 *   qop   the GEMM's activation operand (hq_act_operand_bytes(desc, M)
 *         bytes, 16-byte aligned, opaque) or NULL
 *   sx    fp32 [M]:  max_k |x'[m][k]| / 127  (0 for an all-zero row)
 * At least one of qx, gsum, qop must be given.  x' is the rotated row: per
 * 32-block, sign flip, unnormalized Walsh-Hadamard butterfly at strides 1, 2,
 * 4, 8, 16 in fp32 without fused multiply-add, then multiplication by
 * fp32(1/sqrt(32)).  flags: HQ_LAUNCH_DEFAULT or HQ_LAUNCH_PDL. */
int hq_rotate_quant_act(const hq_layer_desc *desc, const float *X, int32_t M, const uint32_t *signs, int8_t *qx,
                        int32_t *gsum, void *qop, float *sx, uint32_t flags, void *stream);

/* Verify pass, step 2: integer GEMM of the quantized activations against the
 * packed weights with the per-group dequantization epilogue (section "How
 * Uzu optimizes bytes and tokens per pass": both matmul operands integers).
 *   blob      packed by hq_pack_weights for the same desc (16-byte aligned)
 *   qop, sx   from hq_rotate_quant_act with the same M, a descriptor of the
 *             same K, group and format, and the same signs
 *   M         0..HQ_MAX_M (0: no-op); one launch for every M
 *   Y         fp32 [M][N]:
 *               Y[m][n] = sx[m] * sum_g ( scale[n][g] * P[m][n][g] )
 *             with P[m][n][g] = sum_{k in g} qx[m][k] * (code[n][k] - zero[n][g])
 *             (zero = 0 for Large), the sum over g in fp32.
 *   partials  check mode: NULL, or int32 [M][N][K/group] that receives P
 *             exactly (slower; for verification)
 *   workspace hq_workspace_bytes(desc, M) bytes, 16-byte aligned, zero-filled
 *             before its first use
 * The integer sums P are exact: the codes are multiplied on the tensor cores
 * with fp32 accumulation, exact for these ranges (up to 32 rows: warp-level
 * fp16 MMAs on the weight codes widened in registers, 4-bit codes to
 * q - z; above: tcgen05 MMAs with e4m3 or fp16 operands, the Medium zero
 * point entering through the group sums).  The fp32 sum over groups is taken in ascending
 * group order.  An output whose K range is
 * split across thread blocks is the sum of the blocks' partial sums: by
 * default each block adds sx[m] * (its partial sum) into Y with an fp32
 * atomic add when it finishes (Y is zeroed first by the kernel itself), so
 * the order of those adds, and the last bits of such outputs, may change from
 * run to run; with HQ_LAUNCH_DETERMINISTIC the blocks wait for one another
 * and sum the partial sums in ascending K order, then multiply by sx[m].
 * Outputs computed by one block are the same in both modes.  Every wait is
 * bounded; the grid never exceeds the blocks resident at once, but a kernel
 * running concurrently on another stream that holds SMs for longer than the
 * bound makes the call time out (HQ_ERR_TIMEOUT from hq_workspace_status;
 * zero the workspace again before reusing it after a time-out).  flags: any
 * of HQ_LAUNCH_PDL, HQ_LAUNCH_DETERMINISTIC, HQ_LAUNCH_EXACT_ORDER (see
 * above); with HQ_LAUNCH_PDL,
 * Y is written only after the wait for the previous kernel. */
int hq_verify_gemm(const hq_layer_desc *desc, const void *blob, const void *qop, const float *sx, int32_t M, float *Y,
                   int32_t *partials, void *workspace, uint32_t flags, void *stream);

/* The verify GEMM on int8 activation codes, the boundary's form with qx, sx
 * and the group sums (page "Karpathy's Trick for Faster Local LLMs Finally
 * Has Proper Tooling", section "How Uzu optimizes bytes and tokens per pass":
 * both matmul operands are integers).  The result is that of
 * hq_verify_gemm on the operand hq_rotate_quant_act would write for these
 * codes (same Y, same modes and flags, same errors).
 *   qx        int8 [M][K] (4-byte aligned): clamp(rint(x' / sx), -127, 127)
 *             from hq_rotate_quant_act or any other producer of the codes
 *   sx        fp32 [M]
 *   gsum      int32 [M][K/group] or NULL: not read (the group sums the
 *             Medium zero point needs are formed from qx, exactly)
 *   workspace hq_workspace_q8_bytes(desc, M) bytes, 16-byte aligned: the
 *             hq_workspace_bytes(desc, M) bytes of hq_verify_gemm (zero-filled
 *             before first use, as there), then room for the operand
 * One launch converts qx into the operand inside the workspace, the GEMM
 * follows on the same stream (with programmatic dependent launch: its weight
 * stream starts while the conversion runs). */
size_t hq_workspace_q8_bytes(const hq_layer_desc *desc, int32_t M);
int hq_verify_gemm_q8(const hq_layer_desc *desc, const void *blob, const int8_t *qx, const float *sx,
                      const int32_t *gsum, int32_t M, float *Y, int32_t *partials, void *workspace, uint32_t flags,
                      void *stream);

/* Canonical view of a blob (for verification and for saving in a portable
 * form): codes uint8 [N][K] (Medium: 0..15; Large: the int8 code's byte),
 * scales fp32 [N][K/group], zeros uint8 [N][K/group] (Medium only; may be
 * NULL for Large). */
int hq_unpack_codes(const hq_layer_desc *desc, const void *blob, uint8_t *codes, float *scales, uint8_t *zeros,
                    void *stream);

/* Synchronizes `stream`, then reads and clears the error word of a
 * workspace (of hq_verify_gemm or hq_tree_attention).  Returns
 * HQ_ERR_TIMEOUT if a bounded wait inside a call that used the workspace
 * gave up since the word was last cleared (the outputs of that call are then
 * incomplete), HQ_OK otherwise. */
int hq_workspace_status(void *workspace, void *stream);

/* hq_verify_gemm without a caller-supplied workspace, for callers that
 * cannot allocate device memory at the point of the call: code that runs
 * under an allocator that forbids new allocations (for example inside a
 * memory-capped serving process, or a plugin whose host owns all device
 * memory), or code that must not call cudaMalloc because it would
 * synchronize the device.  The pages have no counterpart of this call.
 *
 * The scratch lives in one file-scope device array of
 * HQ_NOALLOC_SCRATCH_BYTES (60 MiB + 128 KiB) that every GPU which loads the
 * library holds until the process exits.  A call is accepted when
 * hq_workspace_bytes(desc, M) fits in it (any M, for N up to about two
 * million outputs); larger calls return HQ_ERR_UNSUPPORTED and launch
 * nothing.  The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current
 * and zero-fills the array once (a synchronous cudaMemset); make that first
 * call before any stream capture.  Later calls only launch the GEMM: the
 * kernels leave the array's error word and counters at zero after every
 * call whose waits all succeed.  A bounded wait that gives up (see
 * hq_verify_gemm) leaves the outputs of that call incomplete and records
 * the time-out in the array; hq_noalloc_status reports it and cleans the
 * array up.  All calls on a device share the one array, so calls that may
 * overlap on the GPU (different streams, or graphs replayed concurrently)
 * race and must be serialized by the caller.  Arguments, outputs and flags
 * are those of hq_verify_gemm; HQ_LAUNCH_PDL works as there (nothing runs
 * between the previous kernel and the GEMM). */
#define HQ_NOALLOC_SCRATCH_BYTES (60u * 1024u * 1024u + 128u * 1024u)
int hq_verify_gemm_noalloc(const hq_layer_desc *desc, const void *blob, const void *qop, const float *sx,
                           int32_t M, float *Y, int32_t *partials, uint32_t flags, void *stream);

/* Status of the allocation-free calls on the current device: synchronizes
 * `stream`, then returns HQ_ERR_TIMEOUT if a bounded wait inside an
 * hq_verify_gemm_noalloc call gave up since the last status call (the
 * outputs of that call are incomplete; the array's error word and counters
 * are reset to zero before returning), HQ_OK otherwise (also when no such
 * call has run on the device).  Allocates nothing. */
int hq_noalloc_status(void *stream);

/* Draft-tree acceptance, after the verify pass (sections "Producing several
 * tokens from one model pass": the main model checks the drafted positions
 * together, accepts the valid prefix and adds its own token at the first
 * position it does not confirm; and "Verifying a draft tree without restoring
 * model state": on a tree, the longest valid path is accepted).
 *   logits    fp32 [M][V], row i = the main model's output after tree node i
 *   M         1..HQ_MAX_M tree nodes; node 0 is the root (the last committed
 *             token)
 *   parent    int32 [M], parent[0] ignored, 0 <= parent[i] < i otherwise
 *   tokens    int32 [M], the drafted token of each node (tokens[0] ignored)
 *   greedy    int32 [M] out: argmax of each row (lowest index among equal
 *             maxima; a NaN ranks above every number, the first NaN wins)
 *   path      int32 [M] out: the accepted drafted nodes from the root's child
 *             down, n_accept of them; the other entries -1
 *   n_accept  int32 out: accepted drafted tokens (the sequence advances by
 *             n_accept + 1); -1 (and bonus -1) if parent is not a tree listed
 *             parents-first
 *   bonus     int32 out: greedy[accepted node], the main model's own token
 *   workspace hq_tree_accept_workspace_bytes(M, V) bytes, 16-byte aligned
 * A node i > 0 is valid when its parent is and tokens[i] == greedy[parent[i]];
 * the deepest valid node is accepted, the lowest index among equally deep
 * ones.  All pointers are device memory.  flags: HQ_LAUNCH_DEFAULT or
 * HQ_LAUNCH_PDL. */
size_t hq_tree_accept_workspace_bytes(int32_t M, int32_t V);
int hq_tree_accept(const float *logits, int32_t M, int32_t V, const int32_t *parent, const int32_t *tokens,
                   int32_t *greedy, int32_t *path, int32_t *n_accept, int32_t *bonus, void *workspace, uint32_t flags,
                   void *stream);

/* Tree-masked verify attention (section "Verifying a draft tree without
 * restoring model state": an attention layer keeps a cache of every past
 * token, and the main model checks every branch of the draft tree in one pass
 * without changing its committed state).  The page gives no mask; node i
 * attends to the L committed positions, to its ancestors and to itself (the
 * prefix its branch would have had if decoded alone).  The ancestor walk
 * follows parent[] while the parent lies in [0, node); a parent outside that
 * range ends it.  Textbook softmax attention with grouped heads: query head h
 * reads key/value head h / (Hq / Hkv).
 *   q        fp16 [M][Hq][D], the tree nodes' queries
 *   k_cache  fp16 [Hkv][cap][D]: positions [0, L) committed, position L + j
 *   v_cache  = tree node j (written by this pass's key/value projection)
 *   cap      positions per head in the cache, >= L + M
 *   M        1..HQ_MAX_M tree nodes (node 0 the root); L >= 0
 *   Hq, Hkv  Hq a multiple of Hkv; 64 a multiple of Hq / Hkv
 *   D        HQ_ATTN_HEAD_DIM
 *   parent   int32 [M] (device)
 *   scale    softmax scale (typically 1/sqrt(D)), finite
 *   out      fp32 [M][Hq][D]
 *   workspace hq_tree_attention_workspace_bytes(Hkv) bytes, 16-byte aligned;
 *            its first word is the error word read by hq_workspace_status
 * The probabilities are rounded to fp16 for the product with V (fp32
 * accumulation everywhere): |out - exact| <= 2^-11 * max|v| + fp32 rounding.
 * All pointers are device memory, 16-byte aligned.  flags: HQ_LAUNCH_DEFAULT
 * or HQ_LAUNCH_PDL.  With HQ_LAUNCH_PDL the committed positions [0, L) are
 * read before waiting for the previous kernel of the stream, so that kernel
 * must not write them (the tree rows, q and parent may be its outputs).
 * Launches two kernels (chunks of key positions, then their merge). */
#define HQ_ATTN_HEAD_DIM 128
size_t hq_tree_attention_workspace_bytes(int32_t Hkv);
int hq_tree_attention(const void *q, const void *k_cache, const void *v_cache, int32_t cap, int32_t L, int32_t M,
                      int32_t Hq, int32_t Hkv, int32_t D, const int32_t *parent, float scale, float *out,
                      void *workspace, uint32_t flags, void *stream);

/* Commit of the accepted path into the attention cache (same section: state
 * is committed only along the chosen path).  The root stays at position L;
 * accepted node path[d] (depth d + 1) moves to position L + 1 + d for
 * d < *n_accept, in k_cache and v_cache (layout as in hq_tree_attention);
 * nothing moves when *n_accept <= 0 (no drafted token accepted, or the -1 of
 * a malformed tree) or when L + 1 + *n_accept > cap.  path and n_accept are
 * hq_tree_accept's outputs in device memory, so no host round trip is
 * needed; path entries outside [1, M) are skipped.  The next committed length
 * is L + 1 + *n_accept. */
int hq_tree_commit_kv(void *k_cache, void *v_cache, int32_t cap, int32_t L, int32_t M, int32_t Hkv, int32_t D,
                      const int32_t *path, const int32_t *n_accept, uint32_t flags, void *stream);

/* Rollback-free DeltaNet tree pass (section "Verifying a draft tree without
 * restoring model state": a Gated DeltaNet layer keeps a fixed-size state that
 * every accepted token changes; the verify pass computes every branch's
 * outputs without changing it, and the state is updated only along the
 * accepted path).  The page gives no equations; the recurrence is the
 * published gated delta rule, per head with a D x D state S (rows: value
 * dimensions, columns: key dimensions):
 *     S_i = alpha_i S_p (I - beta_i k_i k_i^T) + beta_i v_i k_i^T,  o_i = S_i q_i
 * with p the parent of tree node i, or the committed state for the root and
 * for a node whose parent lies outside [0, i).
 *   state  fp32 [H][D][D], the committed state; only read
 *   q, k, v  fp32 [M][H][D] (q, k as they enter the recurrence: any
 *          normalization is applied before); alpha, beta fp32 [M][H]
 *   parent int32 [M]; M 1..HQ_MAX_M; D = HQ_DELTA_HEAD_DIM
 *   out    fp32 [M][H][D]
 * Computed without forming any node's state: o_i = S w_i + sum_j c_j v_j over
 * node i's root path (w_i, c_j from D-vector steps), fp32 arithmetic.  With
 * HQ_LAUNCH_PDL the state is read before waiting for the previous kernel of
 * the stream, which therefore must not write it.  All pointers are device
 * memory, 16-byte aligned. */
#define HQ_DELTA_HEAD_DIM 128
int hq_delta_tree(const float *state, const float *q, const float *k, const float *v, const float *alpha,
                  const float *beta, const int32_t *parent, int32_t M, int32_t H, int32_t D, float *out,
                  uint32_t flags, void *stream);

/* Commit of the accepted path into the DeltaNet state (same section): in
 * place, one step for the root and one for each accepted node path[d],
 * d < *n_accept, in order (the new state is the accepted node's state).
 * path and n_accept are hq_tree_accept's outputs in device memory; path
 * entries outside [1, M) are skipped; nothing changes when *n_accept < 0.
 * Arguments as in hq_delta_tree. */
int hq_delta_commit(float *state, const float *k, const float *v, const float *alpha, const float *beta,
                    const int32_t *path, const int32_t *n_accept, int32_t M, int32_t H, int32_t D, uint32_t flags,
                    void *stream);

/* Self-test of the bounded-wait path: launches one block that waits on a
 * shared-memory barrier nothing will ever complete, giving up after
 * `limit_ns` nanoseconds (1000..100000000) and setting the error word of
 * `workspace` (>= 16 bytes, zero-filled).  hq_workspace_status then
 * returns HQ_ERR_TIMEOUT.  No fault and no hang: the kernel returns. */
int hq_selftest_wait_timeout(void *workspace, int64_t limit_ns, void *stream);

/* Self-test of the GEMM's bounded waits between thread blocks: runs
 * hq_verify_gemm (arguments as there, HQ_LAUNCH_DETERMINISTIC) with every
 * wait for the other contributors of a split output asking for one arrival
 * more than there are and giving up after `limit_ns` nanoseconds
 * (1000..100000000).  On a layer with split outputs (K of several 128-feature
 * tiles and more tiles than SMs) the waits run out: hq_workspace_status then
 * returns HQ_ERR_TIMEOUT; Y is unspecified.  No fault and no hang: the kernel
 * returns.  Zero the workspace before reusing it. */
int hq_selftest_gemm_wait_timeout(const hq_layer_desc *desc, const void *blob, const void *qop, const float *sx,
                                  int32_t M, float *Y, void *workspace, int64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* HQ_H */
