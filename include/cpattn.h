/*
 * cpattn.h — C ABI of the GB300 (sm_103a) context-parallel ring-attention library.
 *
 * The operations follow the page "G5 上下文并行建模设计规格" (G5 context-parallel
 * modelling design spec, v1.1.1).  The cp ranks of that spec are VIRTUAL ranks
 * that all live on one GPU: the pass-KV rotation is an index change (rank r at
 * ring step t reads the K/V rows of source rank s = (r - t) mod cp straight from
 * HBM) and the pass-Q dispatch is a shared buffer.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Ownership: the caller allocates and owns every buffer and the CUDA stream.
 *   The library never allocates device memory, never frees, keeps no state
 *   between calls except the device status word read by
 *   cp_take_device_status() and the kernel-choice settings of
 *   cp_set_kernel_choice(), and never synchronises a stream (except in
 *   cp_take_device_status()).  Device calls are asynchronous on `cuda_stream`
 *   (a cudaStream_t; NULL = the legacy default stream).
 * - Errors are returned BEFORE any launch and nothing is launched on error;
 *   there is no fallback path.  A CUDA launch error maps to CP_ERR_CUDA.
 * - Device pointers must be non-NULL and 16-byte aligned.
 * - Layouts are token-major (rows of tokens, then heads, then head_dim):
 *     Q        [b, S, h_q,  d]  bf16        K, V  [b, S, h_kv, d]  bf16
 *     O        [b, S, h_q,  d]  fp32        m, l  [b, h_q, S]      fp32
 *   Grouped-query heads map as kv_head = h / (h_q / h_kv).
 * - The triple (m, l, O) of a query row over a key set J, x_j = scale*<q,k_j>:
 *     m = max_j x_j (natural-log units), l = sum_j exp(x_j - m),
 *     O = sum_j exp(x_j - m) v_j  (unnormalised).  The identity is (-inf, 0, 0).
 *   ("Partial attention" row of the Terms table: max / numerator / denominator,
 *   merged associatively and in any order.)
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CPATTN_API __attribute__((visibility("default")))
#else
#define CPATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARGUMENT = 1, /* bad size, pointer, alignment, step range, mode */
  CP_ERR_UNSUPPORTED = 2,      /* valid request outside what the kernels implement (e.g. head_dim) */
  CP_ERR_OVERFLOW = 3,         /* a byte count does not fit uint64 */
  CP_ERR_CUDA = 4,             /* a CUDA runtime/driver call or launch failed */
  CP_ERR_TIMEOUT = 5           /* a device-side wait gave up (reported by cp_take_device_status) */
} cp_status;

/* Modes of cp_ring_step_partial_attn.  FINALIZE and OVERLAP_PREVIOUS may be OR-ed
 * into either of EMIT and ACCUMULATE. */
enum {
  CP_MODE_EMIT = 0,       /* write the triple of the steps [step_begin, step_end) */
  CP_MODE_ACCUMULATE = 1, /* merge that triple into the triple already in (o, m, l) */
  CP_MODE_FINALIZE = 2,   /* after that, write o = O / l (0 where l = 0); m, l stay */
  /* Launch as a programmatic dependent of the kernel before it on the stream: the
   * CTAs may start while that kernel still runs, read q, k, v at once and wait for
   * it to finish before they read or write o, m, l.  The caller promises that the
   * kernel before this launch on the stream writes none of q, k, v (true in a chain
   * of ring-step launches over the same inputs, where each launch's tail then
   * overlaps the next one's start).  The results are the same bits as without it. */
  CP_MODE_OVERLAP_PREVIOUS = 4
};

/* Chunk layouts.  BALANCED is the method (Terms table, "Balanced chunk split"):
 * rank r holds chunks r and 2cp-1-r.  SEQUENTIAL is the plain split the same row
 * contrasts it with (rank r holds tokens [r*S/cp, (r+1)*S/cp) = chunks 2r, 2r+1),
 * provided to measure the imbalance the balanced split removes. */
enum { CP_LAYOUT_BALANCED = 0, CP_LAYOUT_SEQUENTIAL = 1 };

/* Largest number of partial triples one cp_merge_partials call merges. */
#define CP_MAX_MERGE_PARTS 256

/* Static description of one attention problem (prefill or decode). */
typedef struct {
  int64_t b;      /* batch (sequences) */
  int64_t S;      /* prefill: sequence length; decode: KV length L per sequence */
  int64_t h_q;    /* query heads */
  int64_t h_kv;   /* key/value heads, divides h_q */
  int64_t d;      /* head dimension */
  int64_t cp;     /* virtual ranks (prefill) or KV shards (decode); explicit, >= 1 */
  float scale;    /* softmax scale, > 0 (the spec prints none; callers pass 1/sqrt(d)) */
  int32_t causal; /* prefill: must be 1; decode: must be 0 */
} cp_attn_desc;

/* Human-readable name of a cp_status value (static storage, never NULL). */
CPATTN_API const char* cp_status_string(int32_t status);

/*
 * Balanced head/tail chunk plan (Terms table, row "Balanced chunk split"; design
 * rationale paragraph on balanced splitting; eq. g5cp-step-flops).
 * The sequence is cut into 2*cp chunks of C = S/(2cp) tokens.  Rank r owns chunk
 * r (head) and chunk 2cp-1-r (tail).  At ring step t rank r holds the K/V block of
 * source rank (r - t) mod cp (step 0 = its own block; cp-1 rotations follow).
 * Host-only; all arrays are caller-allocated host memory:
 *   chunk_begin [2cp+1]  int64   first token of chunk k, chunk_begin[2cp] = S
 *   rank_chunks [cp][2]  int32   {r, 2cp-1-r}
 *   step_src    [cp][cp] int32   source rank of rank r at step t
 *   step_pairs  [cp][cp] int64   visible (query,key) pairs per head of rank r at step t:
 *                                2C^2, plus C at t = 0 (the two causal diagonals)
 * Errors: cp < 1, S < 1, S % (2cp) != 0, or a NULL array -> CP_ERR_INVALID_ARGUMENT.
 */
CPATTN_API cp_status cp_plan_balanced_chunks(int64_t S, int32_t cp, int64_t* chunk_begin,
                                  int32_t* rank_chunks, int32_t* step_src,
                                  int64_t* step_pairs);

/*
 * The same plan for either layout (cp_plan_balanced_chunks == layout BALANCED).
 * SEQUENTIAL: rank_chunks[r] = {2r, 2r+1}; with n = S/cp rows per rank,
 * step_pairs[r][t] = n^2 when the source rank s < r, n(n+1)/2 when s == r, 0 when
 * s > r (per-rank totals differ: the imbalance the Terms table describes).
 * Errors: as cp_plan_balanced_chunks, plus an unknown layout -> CP_ERR_INVALID_ARGUMENT.
 */
CPATTN_API cp_status cp_plan_chunks(int64_t S, int32_t cp, int32_t layout, int64_t* chunk_begin,
                                    int32_t* rank_chunks, int32_t* step_src, int64_t* step_pairs);

/*
 * Ring-step partial attention (Terms table rows "Pass-KV", "Ring step", "Partial
 * attention"; eq. g5cp-step-flops) for ALL cp virtual ranks at once, over the ring
 * steps [step_begin, step_end).  For every rank r, local query row i (global
 * position) and step t, the visible keys are the rows of the two chunks of
 * source rank s = (r - t) mod cp with key position <= i.  The steps are merged in
 * ring order inside the kernel; the merged triple of each row is then
 *   EMIT        written to (o, m, l) (rows that saw no key get the identity);
 *   ACCUMULATE  merged into the triple already held in (o, m, l);
 *   | FINALIZE  followed by o = O / l.
 * EMIT | FINALIZE over [0, cp) is the complete causal attention in one launch.
 * q, k, v: bf16 device, layouts above; o, m, l: fp32 device, layouts above.
 * Tiling: each CTA computes two 128-row query tiles that share every K/V tile: two
 * heads of one kv group (even h_q / h_kv) or two consecutive row tiles of one head
 * (odd).  With h_q == h_kv, a launch with at most one wave (SM count) of single tiles
 * keeps one tile per CTA; cp_set_kernel_choice(CP_KNOB_RING_PAIRING, ...) overrides
 * that choice, and every choice gives the same bits.  When such single tiles fill at
 * most half the GPU, each tile's key walk is split over a cluster of 2-8 CTAs whose
 * partial triples are merged on chip (CP_KNOB_RING_KV_SPLIT); the result then equals
 * the unsplit one within rounding.
 * Supported: d in {64, 128}; causal = 1; every pointer 16-byte aligned.
 * Errors: cp < 1, S % (2cp) != 0, h_q % h_kv != 0, any size < 1, scale <= 0 or
 * not finite, 0 <= step_begin < step_end <= cp violated, unknown mode bits, NULL or
 * misaligned pointer -> CP_ERR_INVALID_ARGUMENT; d outside {64,128} or causal != 1
 * -> CP_ERR_UNSUPPORTED; a failed tensor-map encode or launch -> CP_ERR_CUDA.
 */
CPATTN_API cp_status cp_ring_step_partial_attn(const cp_attn_desc* desc, int32_t step_begin,
                                    int32_t step_end, const void* q, const void* k,
                                    const void* v, float* o, float* m, float* l,
                                    int32_t mode, void* cuda_stream);

/*
 * Ring-step partial attention for the virtual ranks [rank_begin, rank_end) only,
 * under either chunk layout; cp_ring_step_partial_attn is layout BALANCED over all
 * ranks [0, cp).  Only the selected ranks' rows of (o, m, l) are read or written.
 * Used to time one virtual rank's work (the per-rank balance of a layout).
 * Errors: as cp_ring_step_partial_attn, plus an unknown layout or
 * 0 <= rank_begin < rank_end <= cp violated -> CP_ERR_INVALID_ARGUMENT.
 */
CPATTN_API cp_status cp_ring_rank_partial_attn(const cp_attn_desc* desc, int32_t layout, int32_t rank_begin,
                                               int32_t rank_end, int32_t step_begin, int32_t step_end,
                                               const void* q, const void* k, const void* v, float* o, float* m,
                                               float* l, int32_t mode, void* cuda_stream);

/*
 * The whole balanced ring for tensors held in HOST memory, with the host<->device
 * copies overlapped with the computation inside the call.  The operation is
 * cp_ring_step_partial_attn over all cp steps in EMIT | FINALIZE mode (Terms table
 * rows "Balanced chunk split", "Pass-KV", "Ring step" and "Partial attention"):
 *   q_host [b, S, h_q, d] bf16, k_host / v_host [b, S, h_kv, d] bf16 (read);
 *   o_host [b, S, h_q, d] fp32 = O / l, m_host / l_host [b, h_q, S] fp32 (written).
 * All six are caller-owned host memory; page-locked (pinned) memory lets the
 * copies overlap the kernels, pageable memory gives the same results more slowly.
 * `workspace` (device, caller-owned, 256-byte aligned, at least
 * cp_ring_attn_host_workspace_bytes bytes) receives the device copies of all six.
 * Pipeline, in units of chunks: the head chunks in ascending order, then the tail
 * chunks in descending order (up to 8 units each).  Head chunk c sees only keys
 * [0, (c+1) S/(2cp)), so K and V are copied in chunk order and a head unit waits
 * only for the prefix it reads; the tail units wait for all of K and V.  A unit's Q
 * rows are copied in, one launch runs all cp ring steps for those rows, and its
 * O, m and l rows are copied out.  Copies in, launches (two streams, so one
 * launch's last CTAs overlap the next) and copies out run on separate streams
 * that the library creates once per device, so one unit's copies overlap other
 * units' computation.  The call is ordered on `cuda_stream`: it starts after the
 * work queued there before it, later work queued there starts after its last
 * copy, and the workspace is in use until then.  The host is not blocked:
 * synchronise `cuda_stream` before reading the outputs.  Calls from several host
 * threads are safe with one workspace each; on one device they share the library's
 * streams, so their copies and launches interleave rather than run side by side.
 * Errors: as cp_ring_step_partial_attn, plus a NULL host pointer or a misaligned
 * or too small workspace -> CP_ERR_INVALID_ARGUMENT; a failed copy, launch or
 * stream/event call -> CP_ERR_CUDA.
 */
CPATTN_API cp_status cp_ring_attn_host_workspace_bytes(const cp_attn_desc* desc, size_t* bytes);
CPATTN_API cp_status cp_ring_attn_host(const cp_attn_desc* desc, const void* q_host, const void* k_host,
                                       const void* v_host, float* o_host, float* m_host, float* l_host,
                                       void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * LSE merge of n_parts partial triples (Terms table, row "Partial attention":
 * the merge is associative and order-free; pass-Q paragraph of the
 * Algorithm/formulas section: the reduce carries O, the max and the denominator).
 *   o_parts [n_parts, batch, rows, heads, d]  m_parts, l_parts [n_parts, batch, heads, rows]
 *   o_out   [batch, rows, heads, d]           m_out, l_out     [batch, heads, rows]
 * (the prefill triple layout with rows = S; the decode partial layout with rows = 1).
 * m = max_p m_p; l = sum_p e^{m_p - m} l_p; O = sum_p e^{m_p - m} O_p, the sums
 * taken in the order given by `order` (a HOST array, a permutation of
 * 0..n_parts-1; NULL = index order).  Parts with m_p = -inf weigh 0; a row whose
 * parts are all the identity stays the identity.  finalize != 0 writes O / l
 * (0 where l = 0) into o_out instead of O.  Outputs must not alias inputs.
 * With d = 128 and at most 64 parts the O rows are streamed by TMA;
 * cp_set_kernel_choice(CP_KNOB_MERGE_KERNEL, 0) selects the plain-load kernel, which
 * gives the same bits.
 * A device-side wait that gives up records CP_ERR_TIMEOUT for cp_take_device_status.
 * Errors: any size < 1, n_parts > CP_MAX_MERGE_PARTS, d % 4 != 0, `order` not a
 * permutation, NULL or misaligned device pointer -> CP_ERR_INVALID_ARGUMENT;
 * d > 512 -> CP_ERR_UNSUPPORTED; a failed tensor-map encode or launch -> CP_ERR_CUDA.
 */
CPATTN_API cp_status cp_merge_partials(int64_t batch, int64_t rows, int64_t heads, int64_t d,
                            int32_t n_parts, const float* o_parts, const float* m_parts,
                            const float* l_parts, const int32_t* order, float* o_out,
                            float* m_out, float* l_out, int32_t finalize,
                            void* cuda_stream);

/*
 * Tree-structured reduction of n_parts triples (n_parts a power of two, 2..256),
 * the O(log cp)-depth reduce topology the spec lists as later work (Limitations
 * table, "pass-Q 归约拓扑固定": Tree Attention's log-depth steps).  Level k merges
 * part i with part i + n/2 for every i, halving n, until one triple is left; every
 * node is the two-part LSE merge.  The kernel computes the whole tree in one pass
 * over the parts (the tree is a pairwise tree over the parts in bit-reversed index
 * order), with the same arithmetic at every node as the multi-row merge applies to
 * two parts, so for rows > 1 the result is bit for bit what level-by-level two-part
 * cp_merge_partials calls give (the one-row merge adds in blocks).  It equals the
 * flat cp_merge_partials up to rounding (the merge is associative).  Same layouts
 * as cp_merge_partials.  No workspace is needed: cp_merge_tree_workspace_bytes
 * gives 0 and `workspace` may be NULL.  Inputs are not modified.
 * Errors: n_parts not a power of two in 2..256, sizes < 1, d % 4 != 0, a NULL or
 * misaligned part or output pointer -> CP_ERR_INVALID_ARGUMENT; d > 512 ->
 * CP_ERR_UNSUPPORTED.
 */
CPATTN_API cp_status cp_merge_tree_workspace_bytes(int64_t batch, int64_t rows, int64_t heads, int64_t d,
                                                   int32_t n_parts, size_t* bytes);
CPATTN_API cp_status cp_merge_partials_tree(int64_t batch, int64_t rows, int64_t heads, int64_t d,
                                            int32_t n_parts, const float* o_parts, const float* m_parts,
                                            const float* l_parts, float* workspace, size_t workspace_bytes,
                                            float* o_out, float* m_out, float* l_out, int32_t finalize,
                                            void* cuda_stream);

/*
 * Bytes of device workspace cp_passq_decode needs for `desc` on the CURRENT
 * device (the split count depends on its SM count).  Host-only.
 * Errors: as cp_passq_decode's argument checks.
 */
CPATTN_API cp_status cp_passq_workspace_bytes(const cp_attn_desc* desc, size_t* bytes);

/*
 * Pass-Q decode (Terms table row "Pass-Q"; use-case decode paragraph; pass-Q
 * paragraph of the Algorithm/formulas section).  One query per sequence is
 * scored against cp KV shards: shard s holds keys [s*L/cp, (s+1)*L/cp) with
 * L = desc->S; every key is visible.  Each shard is further split into key
 * ranges so the whole GPU streams K/V (equal ranges for the streaming kernel; whole
 * 128-key tiles of at most one tile's difference for the shared-K/V kernel, the
 * count chosen so that the SMs get even work); every range writes a partial triple
 * to `workspace`, then the three-quantity reduce (the LSE merge, in shard order)
 * writes
 *   out   [b, h_q, d] fp32 = O / l,   m_out, l_out [b, h_q] fp32 (each nullable).
 * q [b, h_q, d] bf16; k, v [b, L, h_kv, d] bf16.  The query dispatch of the spec
 * is the shared q buffer.
 * Supported: g = h_q / h_kv in {1, 2, 4} with d in {64, 128, 256, 512} and
 * g * d <= 1024 (a streaming kernel on the FP32 pipes); or g in {16, 32} with d in
 * {128, 256, 512} (query heads sharing one K/V head, MQA / MLA-style: both
 * contractions on the tensor cores; k and v may be the same buffer);
 * cp * splits <= CP_MAX_MERGE_PARTS; causal = 0.
 * Errors: cp < 1, L % cp != 0, sizes < 1, h_q % h_kv != 0, scale <= 0, NULL or
 * misaligned pointer, workspace_bytes below cp_passq_workspace_bytes ->
 * CP_ERR_INVALID_ARGUMENT; unsupported d, group or causal -> CP_ERR_UNSUPPORTED.
 */
CPATTN_API cp_status cp_passq_decode(const cp_attn_desc* desc, const void* q, const void* k,
                          const void* v, float* workspace, size_t workspace_bytes,
                          float* out, float* m_out, float* l_out, void* cuda_stream);

/*
 * Pass-Q decode that allocates nothing (the pages have no counterpart to this
 * call; it exists for callers that cannot allocate device memory).
 * Same operation, layouts, support limits and argument errors as cp_passq_decode,
 * but without a workspace argument: the per-range partial triples go to a fixed
 * scratch array of CP_PASSQ_NOALLOC_SCRATCH_BYTES built into the library, which
 * every GPU that loads the library holds until the process exits.  Callers that
 * cannot allocate are, for example, a plug-in whose host runtime owns all device
 * memory and hands it only its input and output buffers, or a token loop that
 * must not call cudaMalloc because it may synchronise the device.
 * - It calls no cudaMalloc, cudaFree or other allocating routine.
 * - The first call on a device looks up the scratch's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.  Each call checks that the device's context is still the one the
 *   address was looked up in; after a device reset (cudaDeviceReset) the next
 *   call looks it up again in the new context, so that call too should come
 *   before any capture.
 * - All calls share the scratch, which keeps the last call's contents (nothing in
 *   it needs to start at zero).  Calls that overlap on the GPU (other streams,
 *   or other host threads) race on it and must be serialised by the caller.
 * - The shards are split as in cp_passq_decode while the partials fit; otherwise
 *   into fewer ranges.  A problem whose partials do not fit even one range per
 *   shard (cp * b * h_q * (d + 2) * 4 bytes, rounded up per section, above the
 *   limit) returns CP_ERR_UNSUPPORTED before any launch.
 */
#define CP_PASSQ_NOALLOC_SCRATCH_BYTES (8u << 20)
CPATTN_API cp_status cp_passq_decode_noalloc(const cp_attn_desc* desc, const void* q, const void* k,
                                             const void* v, float* out, float* m_out, float* l_out,
                                             void* cuda_stream);

/* Inputs of the closed-form byte counts (all >= 0; cp >= 1). */
typedef struct {
  int64_t S;       /* sequence length */
  int64_t cp;      /* CP degree */
  int64_t c_kv;    /* K+V bytes per token per layer (both K and V already counted) */
  int64_t b;       /* decode batch */
  int64_t d;       /* model hidden size (length of the partial output vector) */
  int64_t n_h;     /* attention heads */
  int64_t s_dtype; /* bytes per element of the pass-Q messages */
  int64_t layers_local; /* attention layers held by one rank (L_local of the memory paragraph) */
} cp_comm_query;

typedef struct {
  uint64_t passkv_total;    /* (cp-1) * (S/cp) * c_kv        eq. g5cp-passkv-bytes */
  uint64_t passkv_per_step; /* (S/cp) * c_kv                 bytes of one ring step */
  uint64_t passq_dispatch;  /* b * d * s_dtype               pass-Q query dispatch */
  uint64_t passq_reduce;    /* b * (d + 2 n_h) * s_dtype     pass-Q reduce message */
  uint64_t kv_bytes_per_rank; /* b * S * c_kv * L_local / cp  per-rank KV footprint */
} cp_comm_result;

/*
 * Closed-form communication volumes and the per-rank KV footprint (Algorithm /
 * formulas section: eq. g5cp-passkv-bytes, the pass-Q paragraph and the memory
 * paragraph), exact in uint64.  Host-only.  The footprint is computed as
 * b * (S/cp) * c_kv * L_local, exact because S % cp == 0.
 * The pass-KV formula carries no batch factor, as printed (per rank per layer).
 * Errors: NULL pointer, a negative field, cp < 1, S % cp != 0 ->
 * CP_ERR_INVALID_ARGUMENT; any result above 2^64-1 -> CP_ERR_OVERFLOW (the
 * result struct is then left untouched).
 */
CPATTN_API cp_status cp_comm_bytes(const cp_comm_query* query, cp_comm_result* result);

/*
 * Kernel-choice settings, for tests and diagnostics (the pages have no counterpart:
 * each knob picks between kernels of this library that compute the same result).
 *   CP_KNOB_RING_PAIRING  -1 automatic (default); 0 one query tile per CTA for
 *                         launches with h_q == h_kv; 1 two tiles per CTA always.
 *   CP_KNOB_MERGE_KERNEL  -1 automatic (default: TMA-fed where supported);
 *                         0 the plain-load kernel; 1 the same as -1.
 *   CP_KNOB_RING_KV_SPLIT -1 automatic (default); 0 never split a query tile's key
 *                         walk over a CTA cluster; 1 the same as -1.  The split
 *                         merges the parts' triples in another order, so its results
 *                         equal the unsplit ones within rounding, not bit for bit.
 * The setting is process-wide, applies to every device and to launches made after
 * the call returns, and is read once per launch (no environment variable is read
 * anywhere in the library).
 * Errors: an unknown knob or a value outside {-1, 0, 1} -> CP_ERR_INVALID_ARGUMENT.
 */
enum { CP_KNOB_RING_PAIRING = 0, CP_KNOB_MERGE_KERNEL = 1, CP_KNOB_RING_KV_SPLIT = 2 };
CPATTN_API cp_status cp_set_kernel_choice(int32_t knob, int32_t value);

/*
 * Synchronise `cuda_stream`, then read and clear the library's device status
 * word on the current device.  Kernels never trap: a device-side wait that gives
 * up records CP_ERR_TIMEOUT there and the kernel returns early (its outputs are
 * then undefined).  *status receives CP_OK or the recorded error.
 * Errors: NULL status -> CP_ERR_INVALID_ARGUMENT; a failed CUDA call -> CP_ERR_CUDA.
 */
CPATTN_API cp_status cp_take_device_status(void* cuda_stream, int32_t* status);

/*
 * Self-test of the failure path (no counterpart on the pages, which leave failure
 * handling out; their design rationale forbids silent fallbacks).  Launches one
 * CTA on `cuda_stream` that waits, with the same bounded mbarrier wait the ring
 * kernel uses, on a barrier nothing will complete.  After about one second the
 * wait gives up and records CP_ERR_TIMEOUT in the ring kernel's device status
 * word; until cp_take_device_status() clears it, ring launches return at once
 * without writing.  Nothing faults, traps or hangs.
 * Errors: a failed launch -> CP_ERR_CUDA.
 */
CPATTN_API cp_status cp_selftest_wait_timeout(void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */
