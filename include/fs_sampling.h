/*
 * fs_sampling.h -- sorting-free top-k / top-p / min-p sampling on GB300 (sm_103a).
 *
 * C ABI of libfs_sampling.so.  Sources of the operations (three web pages on one
 * subject):
 *   [blog]      "Sorting-Free GPU Kernels for LLM Sampling" (FlashInfer blog):
 *               Top-K / Top-P / Min-P, inverse transform sampling, rejection
 *               sampling, dual-pivot rejection sampling, correctness proof,
 *               implementation details (guarded parallel prefix sums).
 *   [drill]     "F4: top-k / top-p without sorting" (GPU kernel drills hint page):
 *               sections 2-4 (threshold by bisection on count / mass, bisection on
 *               the fp32 bit pattern), section 8 (signed values need their sign
 *               handled before a bit-pattern comparison).
 *   [explainer] FlashInfer sorting-free sampling explainer: the allowed set S and
 *               renormalised distribution, top-k-first vs joint order, the API list
 *               (direct sampling vs filter-only), seed/offset and RNG ownership,
 *               degenerate rows.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless stated.
 *    Each call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 *    the legacy default stream) and may be made from several host threads at once.
 *  - Scratch memory.  The top-k-first samplers, the joint order with a top-k or a
 *    min-p filter on rows of probabilities (fs_top_k_top_p_sampling*,
 *    fs_top_k_sampling, fs_min_p_sampling) and fs_sampling_from_probs run as two
 *    launches: a scan that reads every input row
 *    once, spread evenly over the GPU, and writes a small summary of each row (a few
 *    bytes per 128 values; the joint order adds one byte per 4 values), then one CTA
 *    per output row that finishes the row from that summary.  The summaries live in a
 *    scratch buffer that the library owns, one per (device, stream): calls on one
 *    stream run in order and share it; calls on different streams do not touch each
 *    other's.  The first call that needs more than the stream's buffer holds
 *    allocates it (cudaMalloc, in relaxed stream-capture mode, so this may happen
 *    while the stream is being captured; the buffer then belongs to the library, not
 *    to the graph).  fs_workspace_reserve allocates ahead of time and
 *    fs_release_workspaces frees every buffer.  A new buffer is set to zero on `stream`
 *    (the scan's claim counters in it must start at zero; each call leaves them at
 *    zero).  A CUDA graph captured on a stream uses
 *    that stream's buffer on every replay: do not replay it while other calls of
 *    this library on that stream, or other replays of graphs captured on it, may run
 *    at the same time.  No other call allocates, and no state but these buffers
 *    outlives a call.
 *  - `probs` / `logits` are row-major [batch_in, vocab] float32, contiguous (row
 *    stride = vocab).  Rows are probabilities (or unnormalised non-negative scores;
 *    every filter is scale-invariant, see top-p below).
 *  - Sampling entries produce one token per OUTPUT row b in [0, batch_out).
 *    `indices` (nullable) maps output row b to input row indices[b]; when NULL,
 *    batch_out must equal batch_in and row b reads input row b.  Several output rows
 *    may share an input row (parallel samples); each still draws its own numbers.
 *  - Per-row parameter arrays are indexed by OUTPUT row (length batch_out):
 *      top_k[b] <= 0 or >= vocab     : no top-k filter;
 *      top_p[b] >= 1                 : no top-p filter; top_p[b] <= 0 keeps the arg-max;
 *      min_p[b] <= 0                 : no min-p filter; min_p[b] > 1 keeps nothing.
 *  - Random numbers: Philox4x32-10 (Salmon et al., SC'11) with
 *      key = (seed lo, seed hi), counter = (round, output row b, offset lo, offset hi);
 *    u = (first word >> 8) * 2^-24.  A caller must advance `offset` on every call
 *    ([explainer] seed/offset: reusing it repeats the same draws).  The same inputs,
 *    seed, offset and launch give the same tokens (no atomics decide a result).
 *  - Outputs of sampling entries: out_token[b] (int32), out_valid[b] (uint8: 1 valid,
 *    0 invalid) and, if out_rounds != NULL, out_rounds[b] = number of draws made.
 *    A row is INVALID -- token -1, valid 0, never token 0 ([explainer] degenerate
 *    rows) -- when its input row holds a NaN or a negative entry, sums to 0 (or its
 *    float32 total overflows), keeps no token (e.g. min_p > 1), has a NaN parameter,
 *    indices[b] is out of range, or FS_MAX_ROUNDS draws end without acceptance.
 *  - Return value (fs_status): only what the host can check -- NULL required
 *    pointers, vocab < 1, vocab > FS_MAX_VOCAB, batch < 0, indices == NULL with
 *    batch_out != batch_in, a bad order value -- or a CUDA launch error
 *    (FS_ERR_CUDA; fs_last_error_string() then holds the CUDA message).  A call
 *    with batch_out == 0 (or batch == 0) does nothing and returns FS_OK.  Data
 *    problems of single rows never become a status; they become valid = 0.
 */
#ifndef FS_SAMPLING_H
#define FS_SAMPLING_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fs_status {
    FS_OK = 0,
    FS_ERR_INVALID_ARG = 1,
    FS_ERR_UNSUPPORTED = 2,
    FS_ERR_CUDA = 3
} fs_status;

/* Order of top-k and top-p ([explainer] filter order; [blog] footnote 1).
 * TOP_K_FIRST: keep the top k, then apply top-p inside them with their mass
 *              renormalised (top-p measured against F_k = mass of the k kept);
 * JOINT:       the filters are checked together in every rejection round, each on
 *              the original row (S = S_k intersect S_p intersect S_min). */
typedef enum fs_order {
    FS_ORDER_TOP_K_FIRST = 0,
    FS_ORDER_JOINT = 1
} fs_order;

#define FS_MAX_VOCAB 2097152   /* largest supported vocab */
#define FS_MAX_ROUNDS 256      /* rejection rounds before a row is reported invalid */
#define FS_NOALLOC_SCRATCH_BYTES (8u << 20)  /* fixed scratch of fs_top_k_top_p_sampling_noalloc */

/* Plain categorical sampling: one draw by inverse transform over the whole row.
 * [blog] "inverse transform sampling": u ~ U[0,1), the token k with
 * F_{k-1} <= u * M < F_k, located tile by tile with a guarded prefix sum
 * ([blog] "implementation details"). */
fs_status fs_sampling_from_probs(const float* probs, int32_t batch_in, int32_t vocab,
                                 const int32_t* indices, int32_t batch_out,
                                 uint64_t seed, uint64_t offset,
                                 int32_t* out_token, uint8_t* out_valid,
                                 int32_t* out_rounds, void* stream);

/* Top-k sampling by dual-pivot rejection ([blog] "dual-pivot rejection sampling",
 * proof section: Pr[out = j] = p_j / Z on the k largest).  top_k: [batch_out] int32. */
fs_status fs_top_k_sampling(const float* probs, int32_t batch_in, int32_t vocab,
                            const int32_t* indices, int32_t batch_out,
                            const int32_t* top_k,
                            uint64_t seed, uint64_t offset,
                            int32_t* out_token, uint8_t* out_valid,
                            int32_t* out_rounds, void* stream);

/* Top-p (nucleus) sampling: S = the smallest descending prefix whose mass reaches
 * top_p * M, M = the row's own total ([explainer] Top-p, ">=" form).
 * top_p: [batch_out] float32. */
fs_status fs_top_p_sampling(const float* probs, int32_t batch_in, int32_t vocab,
                            const int32_t* indices, int32_t batch_out,
                            const float* top_p,
                            uint64_t seed, uint64_t offset,
                            int32_t* out_token, uint8_t* out_valid,
                            int32_t* out_rounds, void* stream);

/* Min-p sampling: S = {i : p_i >= min_p * max_j p_j} ([blog] Min-P).  The threshold
 * is the float32 rounded up from the exact product, so p_i >= threshold holds exactly
 * when p_i >= min_p * max.  min_p: [batch_out] float32. */
fs_status fs_min_p_sampling(const float* probs, int32_t batch_in, int32_t vocab,
                            const int32_t* indices, int32_t batch_out,
                            const float* min_p,
                            uint64_t seed, uint64_t offset,
                            int32_t* out_token, uint8_t* out_valid,
                            int32_t* out_rounds, void* stream);

/* Combined top-k + top-p (+ optional min-p) sampling, order = fs_order value
 * ([explainer] filter order).  top_k and top_p are required ([batch_out] each);
 * min_p is nullable and, when given, is intersected in either order. */
fs_status fs_top_k_top_p_sampling(const float* probs, int32_t batch_in, int32_t vocab,
                                  const int32_t* indices, int32_t batch_out,
                                  const int32_t* top_k, const float* top_p,
                                  const float* min_p, int32_t order,
                                  uint64_t seed, uint64_t offset,
                                  int32_t* out_token, uint8_t* out_valid,
                                  int32_t* out_rounds, void* stream);

/* Sampling with caller-owned generator state ([explainer] RNG ownership: per-request
 * seed / offset, and a device-resident offset so that a captured CUDA graph advances
 * its own state between replays).  Arguments as fs_top_k_top_p_sampling, except:
 *   top_k, top_p   nullable here (NULL: that filter is off);
 *   seeds          [batch_out] uint64, nullable: Philox key of output row b;
 *   offsets        [batch_out] uint64, nullable: counter offset of output row b;
 *   offset_dev     one uint64 in device memory, nullable: added to every row's offset
 *                  (read when the kernel runs, after earlier work on the stream);
 *   seed, offset   used for rows whose seeds / offsets array is NULL.
 * Row b draws Philox4x32-10 with key = seed_b and counter = (round, s_b, lo, hi) of
 * offset_b + *offset_dev, where s_b = b when `seeds` is NULL and 0 otherwise: with
 * per-request seeds a request's draws do not depend on its position in the batch.
 * A consequence: two output rows with the same seed and the same offset draw the same
 * numbers, hence the same token when they read the same input row.  Parallel samples
 * of one request (several output rows mapped to one input row through `indices`) need
 * distinct seeds or distinct offsets here; without `seeds` they differ by b.
 * Nothing is advanced by this call; see fs_advance_offset. */
fs_status fs_top_k_top_p_sampling_rng(const float* probs, int32_t batch_in, int32_t vocab,
                                      const int32_t* indices, int32_t batch_out,
                                      const int32_t* top_k, const float* top_p,
                                      const float* min_p, int32_t order,
                                      const uint64_t* seeds, const uint64_t* offsets,
                                      const uint64_t* offset_dev,
                                      uint64_t seed, uint64_t offset,
                                      int32_t* out_token, uint8_t* out_valid,
                                      int32_t* out_rounds, void* stream);

/* Sampling from logits with the softmax fused in ([explainer] the sampling pipeline:
 * p = softmax(z / T) before the filters).  logits: [batch_in, vocab] float32.  The row
 * is read from HBM once (an online softmax: the first pass keeps each segment's
 * largest logit and, where needed, its mass relative to it; the row maximum m follows
 * from the CTAs'); the rest of the path (every filter, order and the dual-pivot
 * rounds, exactly as fs_top_k_top_p_sampling) then runs on the weights
 * w = exp((z - m) / T) in float32 -- the unnormalised softmax, read again from L2 --
 * so no probability matrix is written.  temperature: [batch_out] float32, nullable
 * (1); T <= 0 or NaN makes the row invalid.  top_k, top_p, min_p: nullable.  A NaN
 * or +inf logit makes the row invalid; -inf logits have weight 0.  Top-k and top-p
 * are decided on the float32 weights (two logits whose weights round to the same
 * float32 count as equal). */
fs_status fs_top_k_top_p_sampling_from_logits(const float* logits, int32_t batch_in, int32_t vocab,
                                              const int32_t* indices, int32_t batch_out,
                                              const float* temperature,
                                              const int32_t* top_k, const float* top_p,
                                              const float* min_p, int32_t order,
                                              uint64_t seed, uint64_t offset,
                                              int32_t* out_token, uint8_t* out_valid,
                                              int32_t* out_rounds, void* stream);

/* Ablation of the pivot rule: as fs_top_k_top_p_sampling (top_k and top_p nullable),
 * with pivots = 2 the dual-pivot sampler and pivots = 1 the one-pivot rejection
 * sampler of [blog] "rejection sampling" (after a rejection low <- pivot1; no second
 * pivot).  Both draw from the same distribution; the one-pivot rule needs more rounds
 * when many tokens lie below the cut.  pivots outside {1, 2}: FS_ERR_INVALID_ARG. */
fs_status fs_top_k_top_p_sampling_pivots(const float* probs, int32_t batch_in, int32_t vocab,
                                         const int32_t* indices, int32_t batch_out,
                                         const int32_t* top_k, const float* top_p,
                                         const float* min_p, int32_t order, int32_t pivots,
                                         uint64_t seed, uint64_t offset,
                                         int32_t* out_token, uint8_t* out_valid,
                                         int32_t* out_rounds, void* stream);

/* *offset_dev += delta on the device, ordered on `stream` (one thread; no status
 * beyond launch errors).  Placed after the sampling call inside a captured graph it
 * gives every replay fresh draws.  offset_dev must not be NULL. */
fs_status fs_advance_offset(uint64_t* offset_dev, uint64_t delta, void* stream);

/* Filter-only: keep x >= t, t = the largest threshold with count(x >= t) >= k, found
 * exactly on the fp32 bit pattern ([drill] sections 2-4); write x / (kept mass), 0
 * elsewhere.  top_k: [batch] int32 (<= 0 or >= vocab: keep all).  out_probs:
 * [batch, vocab] float32, may equal probs (in place).  out_valid: [batch] uint8,
 * nullable; an invalid row (NaN, negative, zero or overflowing total) is written as
 * zeros. */
fs_status fs_top_k_renorm_probs(const float* probs, int32_t batch, int32_t vocab,
                                const int32_t* top_k, float* out_probs,
                                uint8_t* out_valid, void* stream);

/* Filter-only top-p: t = the largest threshold with mass(x >= t) >= top_p * M
 * ([drill] sections 2-4); writes x / mass(x >= t) or 0.  top_p: [batch] float32
 * (>= 1 keeps all, <= 0 keeps the arg-max, NaN makes the row invalid).  out_probs
 * may equal probs. */
fs_status fs_top_p_renorm_probs(const float* probs, int32_t batch, int32_t vocab,
                                const float* top_p, float* out_probs,
                                uint8_t* out_valid, void* stream);

/* Filter-only on logits: keep the k largest, write -inf elsewhere.  The threshold is
 * found on an order-preserving integer key of the signed float ([drill] section 8:
 * negative bit patterns sort backwards, so the key flips them).  A row holding a NaN
 * is invalid and written as -inf.  top_k: [batch] int32 (<= 0 or >= vocab: copy).
 * out_logits may equal logits. */
fs_status fs_top_k_mask_logits(const float* logits, int32_t batch, int32_t vocab,
                               const int32_t* top_k, float* out_logits,
                               uint8_t* out_valid, void* stream);

/* Chain speculative-sampling verification (speculative decoding), one cluster per
 * batch row.  The pages name it as a use of the sampler ([blog] community adoption)
 * without an algorithm; this follows Leviathan et al. 2023, Algorithm 1 / Chen et
 * al. 2023, Algorithm 2.  For row b, draft token d_i (drawn by the caller from draft
 * row q_i) is accepted while u_i * q_i(d_i) < p_i(d_i); at the first rejection i the
 * emitted token is drawn from the residual max(p_i - q_i, 0), and after num_draft
 * acceptances from p_{num_draft+1}.  Rows are used as given (not renormalised); a
 * draft token outside [0, vocab) is rejected.  The draw is the sampler's inverse
 * transform over the weights.  Randomness: the Philox stream of row b as in the
 * samplers (key = seed, counter = (round, b, offset)): round i for the test of draft
 * i, round num_draft for the draw.
 *   draft_probs  [batch, num_draft, vocab] float32, device (may be null if num_draft = 0)
 *   draft_tokens [batch, num_draft] int32, device (idem)
 *   target_probs [batch, num_draft + 1, vocab] float32, device
 *   out_tokens   [batch, num_draft + 1] int32, device: the accepted draft tokens, then
 *                the emitted token, then -1
 *   out_accepted [batch] int32: accepted draft tokens
 *   out_emitted  [batch] int32: accepted + 1, or accepted when the draw's weights are
 *                not a valid row (a NaN or infinite value, a negative value in the
 *                bonus row, or no positive mass); the emitted slot is then -1
 * Pointers are device memory owned by the caller; nothing is allocated.  Errors:
 * FS_ERR_INVALID_ARG for negative sizes, vocab < 1 or a required null pointer;
 * FS_ERR_UNSUPPORTED for vocab > FS_MAX_VOCAB or batch * (num_draft + 1) >= 2^31. */
fs_status fs_chain_speculative_sampling(const float* draft_probs, const int32_t* draft_tokens,
                                        const float* target_probs, int32_t batch, int32_t num_draft,
                                        int32_t vocab, uint64_t seed, uint64_t offset,
                                        int32_t* out_tokens, int32_t* out_accepted, int32_t* out_emitted,
                                        void* stream);

/* The launch plan of the sampling kernels for `batch_out` rows of `vocab` elements on
 * the current device.  order = FS_ORDER_TOP_K_FIRST gives the plan of the
 * top-k-first entries (fs_top_k_top_p_sampling*, order top-k-first) and of
 * fs_sampling_from_probs: a scan of every row with *ctas_per_sm CTAs on every SM,
 * then one CTA per row (*cluster = 1) that finishes the row from its summary
 * (*segments_per_cta = the row's segments; fs_sampling_from_probs finishes with one
 * warp per row); the joint order with a top-k or a min-p filter on rows of
 * probabilities (fs_top_k_sampling, fs_min_p_sampling) runs the same two launches.
 * FS_ORDER_JOINT gives the plan of the cluster kernel: fs_top_p_sampling, whose
 * rejection rounds pass over the row several times on a cluster of CTAs, for rows of
 * probabilities that are 16-byte aligned with vocab % 4 = 0 (other rows run a
 * scalar-load build of the same kernel).  Outputs (host pointers): CTAs per row
 * (*cluster), elements per segment, segments per CTA and the most CTAs resident on
 * one SM (*ctas_per_sm; below the occupancy limit when the plan caps it through its
 * shared-memory request).  Host only; nothing is launched.
 * FS_ERR_INVALID_ARG: batch_out or vocab < 1, a null output, an unknown order. */
fs_status fs_sampling_plan(int32_t batch_out, int32_t vocab, int32_t order, int32_t* cluster,
                           int32_t* segment_len, int32_t* segments_per_cta, int32_t* ctas_per_sm);

/* The counter-based generator the samplers draw from, exposed for checking:
 * out[4i..4i+3] = Philox4x32-10(counter = ctr[4i..4i+3], key = key[2i..2i+1]).
 * ctr: [n,4] uint32, key: [n,2] uint32, out: [n,4] uint32 (device pointers). */
fs_status fs_philox4x32_10(const uint32_t* ctr, const uint32_t* key, int64_t n,
                           uint32_t* out, void* stream);

/* Static description of a status code. */
const char* fs_status_string(int32_t status);

/* Message of the last FS_ERR_CUDA returned to the calling host thread ("" if none). */
const char* fs_last_error_string(void);

/* FS_MAX_VOCAB, for bindings that cannot read the macro. */
int32_t fs_max_vocab(void);

/* Bytes of scratch that the row summaries of `batch_in` input rows of `vocab` values
 * take on the path that needs the most (see "Scratch memory" above): 2 KB of counters,
 * then per row 8 bytes per segment of the launch plan (128 values per segment up to
 * vocab 2^19), 16 bytes per 512 values and, for the joint order, 1 byte per 4 values.
 * *bytes is a host pointer.  FS_ERR_INVALID_ARG: null bytes, batch_in < 0, vocab < 1. */
fs_status fs_workspace_bytes(int32_t batch_in, int32_t vocab, size_t* bytes);

/* Make sure the scratch buffer of the current device and `stream` holds the summaries
 * of `batch_in` rows of `vocab` values, allocating (cudaMalloc) now if it does not.
 * Host-side; launches nothing.  FS_ERR_CUDA if the allocation fails. */
fs_status fs_workspace_reserve(int32_t batch_in, int32_t vocab, void* stream);

/* fs_top_k_top_p_sampling without any allocation (the pages have no counterpart: this
 * is a deployment variant).  Some callers cannot let a library call cudaMalloc: a
 * serving engine that reserves nearly all of device memory for its KV cache up front
 * and fails or fragments on a later allocation; code that runs under a memory pool
 * or allocator that must see every device allocation; a process that must not risk
 * the device-wide synchronisation an allocation can cause in the middle of a decode
 * step.  This entry takes the same arguments and gives the same results as
 * fs_top_k_top_p_sampling, but both orders keep their row summaries in one fixed
 * array of FS_NOALLOC_SCRATCH_BYTES (8 MiB) that is part of the library's module
 * image: every device that loads the library holds it until the process exits, and no
 * call allocates or frees anything.
 *  - Limit: the summaries of the call must fit FS_NOALLOC_SCRATCH_BYTES: 64 rows of
 *    151936 values take 0.9 MB in the top-k-first order and 3.3 MB in the joint order
 *    (which adds one byte per 4 values), 256 rows of 256000 values 6.1 MB in the
 *    top-k-first order (too many for the joint order); larger batches return
 *    FS_ERR_UNSUPPORTED and fs_last_error_string() says why.
 *  - Set-up: the first call on a device looks the array's device address up
 *    (cudaGetSymbolAddress, which may load the module); make that first call before
 *    any stream capture.
 *  - Sharing: every call on every stream of a device uses the same array, and it keeps
 *    the last call's contents.  Each call first sets the scan's 16 claim counters in it
 *    to zero (an asynchronous memset on `stream`, which allocates nothing); every
 *    other word it reads it has written itself.  Calls whose work overlaps on the GPU
 *    (other streams, or graph replays running at the same time) race on it: order
 *    them. */
fs_status fs_top_k_top_p_sampling_noalloc(const float* probs, int32_t batch_in, int32_t vocab,
                                          const int32_t* indices, int32_t batch_out,
                                          const int32_t* top_k, const float* top_p,
                                          const float* min_p, int32_t order,
                                          uint64_t seed, uint64_t offset,
                                          int32_t* out_token, uint8_t* out_valid,
                                          int32_t* out_rounds, void* stream);

/* Free every scratch buffer of the library on every device.  Only when no call of
 * this library is in flight on any stream (and no captured graph that uses one will
 * be replayed again); later calls allocate afresh. */
fs_status fs_release_workspaces(void);

#ifdef __cplusplus
}
#endif

#endif /* FS_SAMPLING_H */
