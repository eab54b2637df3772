/*
 * lmhead.h -- C ABI of the chunked LM-head log-prob + entropy head for
 * NVIDIA GB300 (sm_103a).
 *
 * For every scored token t, with hidden row h_t (length H), vocabulary table
 * W (V rows of length H), target id y_t and temperature tau:
 *
 *   z_v      = h_t . W_v / tau                         (v = 0 .. V-1)
 *   lse_t    = log sum_v exp(z_v)
 *   logp_t   = z_{y_t} - lse_t
 *   entropy_t = lse_t - sum_v softmax(z)_v z_v         (nats)
 *
 * and the exact backward for per-token cotangents g_l (of logp) and g_e (of
 * entropy):
 *
 *   dz_v        = g_l (onehot(y_t)_v - p_v) - g_e p_v (log p_v + entropy_t)
 *   d_hidden_t  = sum_v (dz_v / tau) W_v
 *   d_weight_v += sum_t (dz_v / tau) h_t
 *
 * Sources (cited by page and section): SkyRL issue #891 "[tx] support long
 * sequence", section "What Each Optimization Does", item 4 -- the loss is
 * computed chunk by chunk so the [T, V] logits never exist at once; tunix
 * PR #2913, section "How the fused log-prob head works" -- a single pass
 * over a chunk's logits yields the target logit (one-hot selection), the
 * row maximum and exponential sum, and the entropy from those same
 * exponentials, the maximum and sum being saved for the backward, which
 * recomputes the logits, turns them into their cotangent elementwise, and
 * feeds that single cotangent to both gradient products; the palingenesis guide
 * "Long Sequences (SeCO)", section "Efficiency" -- partial results are
 * combined by their log-sum-exp.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller, on the
 *    current CUDA device, which is where the library launches (the Python
 *    binding makes the tensors' device current and refuses mixed devices).
 *    The library allocates no device memory, never synchronises the stream
 *    in the compute calls, and enqueues all work on `stream`.
 *  - bf16 tensors are passed as raw bfloat16 bit patterns (uint16_t).
 *  - Matrices are row-major and dense: hidden [T, H], weight [V, H],
 *    d_hidden [T, H], d_weight [V, H].
 *  - Argument errors are returned synchronously and nothing is launched:
 *    LMHEAD_ERR_INVALID_ARG for a NULL required pointer, T < 0, H <= 0,
 *    V <= 0, a temperature that is not finite and > 0, chunk_size <= 0;
 *    LMHEAD_ERR_UNSUPPORTED for H not a multiple of 64, T >= 2^31 - 256,
 *    or a bf16 / fp32 matrix pointer that is not 16-byte aligned;
 *    LMHEAD_ERR_WORKSPACE_TOO_SMALL when workspace_bytes is below
 *    lmhead_workspace_size().  A failed launch returns LMHEAD_ERR_CUDA.
 *  - T == 0 is a no-op that returns LMHEAD_OK (the backward still zeroes
 *    d_weight unless accumulate_dweight is set).
 *  - Conditions found on the device (an unmasked target outside [-V, V), a
 *    bounded wait that gave up, a tile store refused at an invalid
 *    coordinate) are recorded in a status word inside the workspace;
 *    lmhead_read_device_status() returns it.
 *  - Calls are reentrant as long as concurrent calls use distinct
 *    workspaces.  Results are deterministic: the same inputs, shapes and
 *    chunk_size give the same bits.
 *  - Three environment variables, read by the library, change how the work
 *    is launched, never what is computed: LMHEAD_CTA_PAIR=0 (single-CTA
 *    tiles instead of CTA pairs; results within the same tolerances),
 *    LMHEAD_BWD_PERSISTENT (0: two launches per backward block, 1: one
 *    persistent launch, 2: one launch per block window; unset: chosen by
 *    block size; every form gives the same bits) and LMHEAD_FWD_GROUP_MB (MB
 *    of hidden rows per group of token blocks in the forward's work order,
 *    default 32, 0 for one group; same bits).  They are for diagnosis and
 *    measurement.
 *  - After a kernel's first use in the process (which configures it), the
 *    compute calls make no allocation, synchronisation or configuration
 *    call, so a sequence of them can be captured in a CUDA graph.  Their
 *    kernels use programmatic dependent launch: each may start while the
 *    previous work on `stream` drains, and waits for it before touching
 *    memory.
 */
#ifndef LMHEAD_H_
#define LMHEAD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* lmhead_stream_t;

typedef enum {
  LMHEAD_OK = 0,
  LMHEAD_ERR_INVALID_ARG = 1,
  LMHEAD_ERR_UNSUPPORTED = 2,
  LMHEAD_ERR_WORKSPACE_TOO_SMALL = 3,
  LMHEAD_ERR_CUDA = 4,
  LMHEAD_ERR_DEVICE_TIMEOUT = 5, /* a device-side wait exceeded its limit */
  LMHEAD_ERR_BAD_TARGET = 6,     /* a scored target outside [-V, V) */
  LMHEAD_ERR_INTERNAL = 7        /* a kernel refused a tile store at an invalid coordinate
                                    instead of issuing it (a defect of this library) */
} lmhead_status;

enum { LMHEAD_OP_FWD = 0, LMHEAD_OP_BWD = 1, LMHEAD_OP_FWD_BWD = 2 };

/* How lmhead_logps_fwd_bwd runs (see there). */
enum {
  LMHEAD_STRATEGY_AUTO = 0,        /* the library's cost model chooses */
  LMHEAD_STRATEGY_RECOMPUTE = 1,   /* lmhead_logps_fwd, then lmhead_logps_bwd */
  LMHEAD_STRATEGY_KEEP_LOGITS = 2  /* keep each token block's logits; no recompute */
};

/*
 * Bytes of device workspace that lmhead_logps_fwd (op = LMHEAD_OP_FWD),
 * lmhead_logps_bwd (op = LMHEAD_OP_BWD) or lmhead_logps_fwd_bwd (op =
 * LMHEAD_OP_FWD_BWD, any strategy) needs for these sizes; 0 for invalid sizes.  The workspace holds the compacted scored rows (2*T*H bytes at
 * most), per-token statistics (tens of bytes per token) and, for the
 * backward, a bf16 logit-cotangent block of at most about chunk_size * V
 * elements.  It never grows with T * V: chunk_size alone bounds the
 * vocabulary-wide scratch (SkyRL issue #891: the loss memory is set by the
 * chunk, 300 MB at chunk_size 512 on a 152k vocabulary).
 */
size_t lmhead_workspace_size(int op, int64_t T, int32_t H, int32_t V, int32_t chunk_size);

/*
 * Forward: per-token log-prob of the target, entropy and log-sum-exp.
 *
 *  hidden     [T, H] bf16, weight [V, H] bf16
 *  targets    [T] int32; ids in [-V, 0) wrap to id + V (tunix PR #2913,
 *             _target_hit review thread); a scored id outside [-V, V) gives
 *             logp = NaN and sets LMHEAD_ERR_BAD_TARGET in the device status
 *  loss_mask  [T] uint8, nonzero = scored; NULL = every token scored.
 *             Unscored tokens are skipped whole: their hidden rows are never
 *             read by the GEMMs and their outputs are +0.0.
 *  temperature  tau > 0; the logits are h.W / tau
 *  chunk_size   tokens per chunk; sets the backward's scratch bound.  The
 *             forward's results do not depend on it.
 *  logp       [T] fp32 out
 *  entropy    [T] fp32 out, or NULL to skip
 *  lse        [T] fp32 out; keep it for lmhead_logps_bwd
 *  workspace  device buffer of at least lmhead_workspace_size(LMHEAD_OP_FWD, ...)
 *             bytes, 256-byte aligned
 */
lmhead_status lmhead_logps_fwd(const uint16_t* hidden, const uint16_t* weight,
                               const int32_t* targets, const uint8_t* loss_mask, int64_t T,
                               int32_t H, int32_t V, float temperature, int32_t chunk_size,
                               float* logp, float* entropy, float* lse, void* workspace,
                               size_t workspace_bytes, lmhead_stream_t stream);

/*
 * Backward: exact d_hidden and d_weight for per-token cotangents.
 *
 *  hidden, weight, targets, loss_mask, T, H, V, temperature, chunk_size:
 *             as given to lmhead_logps_fwd
 *  grad_logp    [T] fp32 cotangent of logp, or NULL (zeros)
 *  grad_entropy [T] fp32 cotangent of entropy, or NULL: the log-prob-only
 *             backward (tunix PR #2913: GRPO stops the entropy's gradient)
 *  lse        [T] fp32 from lmhead_logps_fwd (required)
 *  entropy    [T] fp32 from lmhead_logps_fwd; required iff grad_entropy
 *  d_hidden   [T, H] fp32 out, overwritten; unscored rows are +0.0
 *  d_weight   [V, H] fp32 out; overwritten, or added to when
 *             accumulate_dweight != 0 (micro-batch accumulation).  The
 *             reduction over tokens runs in a fixed order (deterministic).
 *  workspace  at least lmhead_workspace_size(LMHEAD_OP_BWD, ...) bytes
 *
 * The logits are recomputed chunk by chunk from hidden and weight; the
 * logit cotangent is formed once per block and read by both gradient
 * contractions.
 */
lmhead_status lmhead_logps_bwd(const uint16_t* hidden, const uint16_t* weight,
                               const int32_t* targets, const uint8_t* loss_mask, int64_t T,
                               int32_t H, int32_t V, float temperature, int32_t chunk_size,
                               const float* grad_logp, const float* grad_entropy,
                               const float* lse, const float* entropy, float* d_hidden,
                               float* d_weight, int accumulate_dweight, void* workspace,
                               size_t workspace_bytes, lmhead_stream_t stream);

/*
 * Forward and backward in one call, for losses whose per-token cotangents
 * are known before the forward (a GRPO-style sum of advantage-weighted
 * log-probs plus an entropy term; tunix PR #2913, commit "fused sharded
 * log-prob head": one cotangent, read by both gradient matmuls).
 *
 * Arguments and results are those of lmhead_logps_fwd followed by
 * lmhead_logps_bwd with the same cotangents (entropy is required when
 * grad_entropy is given).  `strategy`:
 *  LMHEAD_STRATEGY_RECOMPUTE    exactly the two calls (logits recomputed in
 *                               the backward);
 *  LMHEAD_STRATEGY_KEEP_LOGITS  token blocks of T_b tokens spanning the whole
 *                               vocabulary (T_b x V <= chunk_size x V): the
 *                               forward keeps the block's logits (16-bit, relative
 *                               to each 256-column tile's running maximum), one
 *                               elementwise pass turns them into the cotangent,
 *                               and no logit is recomputed.  Counted flops stay
 *                               6 T H V, executed flops drop from 8 to 6 T H V;
 *                               results agree with RECOMPUTE within the
 *                               head's tolerances, not bit for bit;
 *  LMHEAD_STRATEGY_AUTO         whichever the library's cost model expects to
 *                               be faster (KEEP_LOGITS needs large chunks, since
 *                               its smaller token blocks add fp32 passes over
 *                               d_weight; lmhead_fwd_bwd_keeps_logits reports the
 *                               choice).
 * workspace: at least lmhead_workspace_size(LMHEAD_OP_FWD_BWD, ...) bytes.
 */
lmhead_status lmhead_logps_fwd_bwd(const uint16_t* hidden, const uint16_t* weight,
                                   const int32_t* targets, const uint8_t* loss_mask, int64_t T,
                                   int32_t H, int32_t V, float temperature, int32_t chunk_size,
                                   const float* grad_logp, const float* grad_entropy,
                                   float* logp, float* entropy, float* lse, float* d_hidden,
                                   float* d_weight, int accumulate_dweight, int strategy,
                                   void* workspace, size_t workspace_bytes,
                                   lmhead_stream_t stream);

/*
 * 1 if LMHEAD_STRATEGY_AUTO keeps the logits for these sizes, 0 if it
 * recomputes them, -1 for invalid sizes; *block_tokens (if not NULL) gets the
 * token block T_b that KEEP_LOGITS would use.
 */
int lmhead_fwd_bwd_keeps_logits(int64_t T, int32_t H, int32_t V, int32_t chunk_size,
                                int32_t* block_tokens);

/*
 * Vocabulary-sharded head.  The vocabulary table is split by rows into
 * shards; a call holds rows [vocab_offset, vocab_offset + V_shard) of a
 * vocabulary of vocab_total ids (weight_shard [V_shard, H] bf16 is those rows,
 * for instance a view into the whole table, or one GPU's shard of it).  A
 * token's statistics over disjoint parts of the vocabulary combine exactly by
 * their log-sum-exp (the rule by which the "Long Sequences (SeCO)" guide,
 * section "Efficiency", merges partial attention results, and by which the
 * forward merges its own vocabulary splits), so the head over the whole
 * vocabulary is:
 *   1. lmhead_logps_fwd_shard on every shard -> 16 bytes of statistics per
 *      token and shard;
 *   2. the shards' statistics brought together (on several GPUs: one
 *      all-gather of 16 bytes per token), and lmhead_combine_shards -> logp,
 *      entropy, lse of the whole vocabulary, as lmhead_logps_fwd gives them;
 *   3. lmhead_logps_bwd_shard on every shard with that lse and entropy ->
 *      the shard's rows of d_weight and its share of d_hidden; d_hidden is the
 *      sum of the shares (on several GPUs: one all-reduce).
 * The shards must tile [0, vocab_total) without overlap.  Results agree with
 * the unsharded calls within the head's tolerances (fp32 summation order
 * differs), not bit for bit.
 *
 * lmhead_logps_fwd_shard: arguments as lmhead_logps_fwd with V = V_shard, plus
 *  targets      ids of the whole vocabulary: ids in [-vocab_total, 0) wrap to
 *               id + vocab_total; an id held by another shard is no error; a
 *               scored id outside [-vocab_total, vocab_total) sets
 *               LMHEAD_ERR_BAD_TARGET in the device status
 *  partials     [T][4] fp32 out, 16-byte aligned: per token {m, s, S1, zy} in
 *               base-2 units of u = z log2(e) over this shard's rows: m the
 *               largest u, s = sum 2^(u - m), S1 = sum 2^(u - m) (u - m), zy the
 *               target's u if the target is in this shard, else -inf.
 *               Unscored tokens get zeros.
 *  workspace    lmhead_workspace_size(LMHEAD_OP_FWD, T, H, V_shard, chunk_size)
 * LMHEAD_ERR_INVALID_ARG also for V_shard <= 0, vocab_offset < 0 or
 * vocab_offset + V_shard > vocab_total; LMHEAD_ERR_UNSUPPORTED for partials
 * not 16-byte aligned.
 */
lmhead_status lmhead_logps_fwd_shard(const uint16_t* hidden, const uint16_t* weight_shard,
                                     const int32_t* targets, const uint8_t* loss_mask,
                                     int64_t T, int32_t H, int32_t V_shard, int32_t vocab_offset,
                                     int32_t vocab_total, float temperature, int32_t chunk_size,
                                     float* partials, void* workspace, size_t workspace_bytes,
                                     lmhead_stream_t stream);

/*
 * logp, entropy (NULL to skip) and lse [T] fp32 of the whole vocabulary from
 * n_shards sets of shard statistics, partials [n_shards][T][4] fp32 (16-byte
 * aligned; set j from lmhead_logps_fwd_shard on shard j, in any fixed shard
 * order: the result depends on the order only through fp32 rounding).
 * Unscored tokens (loss_mask 0) give +0.0; a scored id outside
 * [-vocab_total, vocab_total) gives logp = NaN.  HBM-bound: one read of the
 * statistics.
 */
lmhead_status lmhead_combine_shards(const float* partials, int32_t n_shards,
                                    const int32_t* targets, const uint8_t* loss_mask, int64_t T,
                                    int32_t vocab_total, float* logp, float* entropy, float* lse,
                                    lmhead_stream_t stream);

/*
 * Backward of one vocabulary shard: arguments as lmhead_logps_bwd with
 * V = V_shard and targets as in lmhead_logps_fwd_shard, given the WHOLE
 * vocabulary's lse (and entropy, with grad_entropy) from lmhead_combine_shards.
 *  d_hidden        [T, H] fp32 out, overwritten: this shard's share,
 *                  sum over v in the shard of (dz_v / tau) W_v; the gradient of
 *                  hidden is the sum of every shard's share
 *  d_weight_shard  [V_shard, H] fp32: the gradient of this shard's rows,
 *                  overwritten or accumulated as in lmhead_logps_bwd
 *  workspace       lmhead_workspace_size(LMHEAD_OP_BWD, T, H, V_shard, chunk_size)
 */
lmhead_status lmhead_logps_bwd_shard(const uint16_t* hidden, const uint16_t* weight_shard,
                                     const int32_t* targets, const uint8_t* loss_mask,
                                     int64_t T, int32_t H, int32_t V_shard, int32_t vocab_offset,
                                     int32_t vocab_total, float temperature, int32_t chunk_size,
                                     const float* grad_logp, const float* grad_entropy,
                                     const float* lse, const float* entropy, float* d_hidden,
                                     float* d_weight_shard, int accumulate_dweight,
                                     void* workspace, size_t workspace_bytes,
                                     lmhead_stream_t stream);

/*
 * Logits-level scoring, for callers that already hold one chunk's logits
 * (the per-chunk cross-entropy of a chunked trainer; "Long Sequences (SeCO)"
 * guide, section "Efficiency").  logits [T, V] fp32 row-major; the scored
 * logits are z = logits / temperature.  Outputs as lmhead_logps_fwd.
 *
 * Non-finite logits (the pages test fused scoring on inf, -inf and NaN
 * logits and on a row with no finite logit, and require an isfinite mask in
 * the cotangent -- tunix PR #2913, FusedScoringTest -- without printing
 * values; this is the reading implemented):
 *  - a -inf entry has probability 0 and contributes nothing; a -inf target
 *    logit gives logp = -inf;
 *  - a NaN or +inf entry anywhere in a row makes its lse, logp and entropy NaN;
 *  - a row with no finite entry has lse = -inf and NaN logp and entropy.
 * Unscored rows give +0.0; an id outside [-V, V) gives logp = NaN (there is
 * no device status word for these calls).  HBM-bound: one read of the logits.
 */
lmhead_status lmhead_score_logits_fwd(const float* logits, const int32_t* targets,
                                      const uint8_t* loss_mask, int64_t T, int32_t V,
                                      float temperature, float* logp, float* entropy, float* lse,
                                      lmhead_stream_t stream);

/*
 * d_logits [T, V] fp32 (overwritten; may be the logits buffer itself) =
 * d loss / d logits for cotangents grad_logp / grad_entropy (NULL = zero;
 * entropy required with grad_entropy), given lse (and entropy) from
 * lmhead_score_logits_fwd.  Non-finite logits get a zero cotangent
 * (isfinite mask); finite entries of a NaN row get NaN; unscored rows get
 * zeros.  HBM-bound: one read and one write of [T, V].
 */
lmhead_status lmhead_score_logits_bwd(const float* logits, const int32_t* targets,
                                      const uint8_t* loss_mask, int64_t T, int32_t V,
                                      float temperature, const float* grad_logp,
                                      const float* grad_entropy, const float* lse,
                                      const float* entropy, float* d_logits,
                                      lmhead_stream_t stream);

/*
 * Self-test of failure detection (the pages have no counterpart; the
 * kernels need it on shared GPUs): launches one CTA that allocates tensor
 * memory and waits, with the same bounded mbarrier wait every GEMM pipeline
 * stage uses, on a barrier nothing arrives on.  After `limit_ms` (1..10000)
 * the wait gives up, LMHEAD_ERR_DEVICE_TIMEOUT is recorded in the workspace's
 * status word (read it with lmhead_read_device_status), tensor memory is
 * freed and the kernel exits; the context stays usable.  workspace: at
 * least 256 bytes, 256-byte aligned.
 */
lmhead_status lmhead_selftest_bounded_wait(void* workspace, size_t workspace_bytes,
                                           uint32_t limit_ms, lmhead_stream_t stream);

/*
 * Synchronises `stream`, then returns the device status word that the last
 * call using `workspace` left (LMHEAD_OK, LMHEAD_ERR_BAD_TARGET,
 * LMHEAD_ERR_DEVICE_TIMEOUT or LMHEAD_ERR_INTERNAL), or LMHEAD_ERR_CUDA if the
 * read failed.
 */
lmhead_status lmhead_read_device_status(const void* workspace, lmhead_stream_t stream);

/* Number of scored tokens found by the last call using `workspace`
   (synchronises `stream`); -1 on error. */
int64_t lmhead_read_scored_count(const void* workspace, lmhead_stream_t stream);

/*
 * Size of the static device scratch that lmhead_logps_fwd_noalloc uses:
 * 64 MiB on every GPU where the library's module is loaded, held until the
 * process exits.
 */
#define LMHEAD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * Forward without a caller workspace, for callers that cannot allocate
 * device memory: a plugin running inside a host program that owns every
 * device allocation and hands it no allocator, or code on a path where a
 * cudaMalloc would synchronise the device and stall other work.  The pages
 * have no counterpart to this entry point; it exists only for such callers.
 *
 * Same arguments and results as lmhead_logps_fwd, minus the workspace: the
 * scratch comes from one file-scope device array of
 * LMHEAD_NOALLOC_SCRATCH_BYTES per GPU.  The call allocates nothing (no
 * cudaMalloc, no cudaFree, no allocating library call).
 *  - Errors are those of lmhead_logps_fwd, checked in the same order (sizes,
 *    pointers, alignment); sizes whose forward workspace
 *    (lmhead_workspace_size(LMHEAD_OP_FWD, ...)) exceeds
 *    LMHEAD_NOALLOC_SCRATCH_BYTES then return LMHEAD_ERR_WORKSPACE_TOO_SMALL
 *    before anything is launched (about 11,000 tokens at H = 2560).
 *  - Set-up happens in the first call on each device (and in each CUDA
 *    context on it): the call looks up the array's device address with that
 *    device current (cudaGetSymbolAddress) and caches it per context.  With
 *    CUDA's default lazy module loading that lookup also loads the library's
 *    module, which is when the array's memory is taken, so the first call can
 *    fail with LMHEAD_ERR_CUDA when the device lacks that much free memory.
 *    Make the first call at set-up time, before any stream capture.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's contents; each call re-initialises the parts that must start
 *    from a known state.  Calls whose work overlaps on the GPU (different
 *    streams, or different host threads without ordering) race on it.
 *  - lmhead_read_device_status cannot see this scratch; check logp for NaN
 *    to detect invalid targets.
 */
lmhead_status lmhead_logps_fwd_noalloc(const uint16_t* hidden, const uint16_t* weight,
                                       const int32_t* targets, const uint8_t* loss_mask,
                                       int64_t T, int32_t H, int32_t V, float temperature,
                                       int32_t chunk_size, float* logp, float* entropy,
                                       float* lse, lmhead_stream_t stream);

/* Static, human-readable name of a status code. */
const char* lmhead_status_string(lmhead_status status);

/*
 * Plan the library uses for these sizes on the current device:
 *  fwd_splits   vocabulary splits per token block in the forward
 *  bwd_tokens   tokens per backward block (T_b)
 *  bwd_vocab    vocabulary rows per backward block (V_b); the bf16 cotangent
 *               scratch holds bwd_tokens * bwd_vocab elements
 * Returns LMHEAD_ERR_INVALID_ARG for invalid sizes.
 */
lmhead_status lmhead_plan_info(int64_t T, int32_t H, int32_t V, int32_t chunk_size,
                               int32_t* fwd_splits, int32_t* bwd_tokens, int32_t* bwd_vocab);

/*
 * Instrumentation (off by default).  While enabled, every kernel launch is
 * bracketed by CUDA events on its stream.  lmhead_profile_enable(1) clears
 * earlier records.  lmhead_profile_record() synchronises on the i-th
 * record's end event and returns its kernel name (static string) and
 * duration in milliseconds.
 */
void lmhead_profile_enable(int on);
int lmhead_profile_count(void);
lmhead_status lmhead_profile_record(int i, const char** name, float* ms);

/* Kernels this library has launched in this process. */
uint64_t lmhead_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* LMHEAD_H_ */
