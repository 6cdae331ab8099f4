/*
 * pe.h -- C ABI of one P-EAGLE parallel-drafting round on one GPU (sm_103a).
 *
 * P-EAGLE drafts all K speculative tokens of a sequence in ONE drafter pass
 * instead of K sequential passes (P-EAGLE: Parallel Speculative Decoding in
 * vLLM, "TL;DR" and "Solving the autoregressive drafting bottleneck").  One
 * round is five stages, each an entry point below:
 *
 *   pe_prepare_batch   rebuild the drafter batch (metadata, slot mapping)
 *   pe_scatter_hidden  gather/broadcast the drafter input rows
 *   pe_draft_forward   drafter pass + LM head with fused argmax -> K drafts
 *   pe_verify          greedy verification -> acceptance length, bonus token
 *   pe_step            all of the above on one stream
 *
 * Non-greedy drafting and verification (from the forward pass's logits):
 *
 *   pe_sample_drafts   draw the drafts from the drafter's temperature softmax
 *   pe_verify_sampled  rejection-sampling verification against the target's
 *                      distributions
 *
 * The DFlash-style variant: pe_inject_kv projects the verifier's hidden states
 * straight into the drafter's KV cache.
 *
 * Conventions shared by every entry point:
 *
 * - Memory.  Unless stated otherwise a pointer argument is a DEVICE pointer to
 *   memory the caller owns; structs passed by pointer (pe_config, pe_weights,
 *   pe_kv) and the per-layer pointer arrays inside them are HOST memory and
 *   are only read during the call.  The library never allocates or frees
 *   device memory: scratch comes from the caller's workspace.
 * - Streams.  Every call enqueues work on `stream` (a cudaStream_t; NULL is the
 *   legacy default stream) and returns without synchronising.  Inputs must
 *   stay valid and outputs must not be read until the stream reaches that point.
 * - Host-side validation.  Bad sizes, null or misaligned pointers and a short
 *   workspace return an error status BEFORE anything is launched.  A launch
 *   failure returns PE_ERR_CUDA.
 * - Device-side checks.  Out-of-range token ids, accepted counts, page ids or
 *   positions found on the device write an error code into *err_word (the
 *   first error wins; 0 = none) and the offending access is skipped.  The
 *   caller zeroes *err_word once and reads it after synchronising.  Codes:
 *   the low byte is a pe_status, the next byte says which check fired
 *   (PE_DEV_* below).
 * - Determinism.  Same inputs give bit-identical outputs: no floating-point
 *   atomics; every reduction runs in a fixed order.
 * - Layouts are row-major.  Weights use the nn.Linear [out][in] layout.  The
 *   storage type of every weight, hidden state, input row and cache entry is
 *   pe_config.dtype (fp32 or bf16).
 *
 * Row layout of the drafter batch (P-EAGLE pages, "vLLM implementation
 * details", fused Triton kernel): every sequence b owns S = 2K consecutive
 * padded rows b*S .. b*S+S-1: first the K+1 copy slots of its previous verify
 * batch, in verify order, then K-1 MASK slots.  With a = num_accepted[b] and
 * P = prev_pos[b][0], copy slot r is an accepted context row (r < a), the
 * next-token-prediction row (r == a) or a rejected row (r > a, slot -1, not
 * computed); MASK slot m (row K+m) sits at position P+a+m.  Rejected rows are
 * dropped by compaction: the drafter pass runs only over the n_valid rows of
 * row_list (a+K per sequence).
 */
#ifndef PE_H
#define PE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pe_stream_t; /* same type as cudaStream_t */

typedef enum {
    PE_OK = 0,
    PE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad value */
    PE_ERR_SHAPE = 2,        /* sizes inconsistent or outside the supported range */
    PE_ERR_UNSUPPORTED = 3,  /* valid config this build has no kernel for */
    PE_ERR_CUDA = 4,         /* a launch or CUDA runtime call failed */
    PE_ERR_DEVICE_CHECK = 5, /* (err_word only) a device-side check fired */
    PE_ERR_TIMEOUT = 6       /* (err_word only) a bounded device wait gave up */
} pe_status;

/* Detail codes written to *err_word: (check << 8) | pe_status. */
#define PE_DEV_BAD_TOKEN    0x0105 /* token id outside [0, vocab] */
#define PE_DEV_BAD_ACCEPTED 0x0205 /* num_accepted outside [0, K] */
#define PE_DEV_BAD_PAGE     0x0305 /* block-table entry outside [0, num_pages) */
#define PE_DEV_BAD_POSITION 0x0405 /* position beyond the block table, or negative */
#define PE_DEV_NONFINITE    0x0505 /* LM head: a logit was NaN or infinite; draws: NaN or +inf */
#define PE_DEV_BAD_ROW      0x0605 /* a row index outside the batch */
#define PE_DEV_TIMEOUT      0x0106 /* a pipeline wait exceeded its time limit */

typedef enum { PE_F32 = 0, PE_BF16 = 1 } pe_dtype;

/*
 * Drafter and batch shape.  The drafter (fc 2d->d, then per layer: RMSNorm,
 * GQA attention with rotate-half RoPE over the paged cache, RMSNorm, SwiGLU
 * MLP; then a final RMSNorm and the LM head) is the one the GPT-OSS-20B and
 * Qwen3-Coder-30B P-EAGLE heads use; the pages name "N transformer layers and
 * an LM head" (P-EAGLE: Parallel Speculative Decoding in vLLM, step 2
 * "Parallel Drafting").
 */
typedef struct {
    int32_t B;                 /* sequences in the batch, >= 1 */
    int32_t K;                 /* draft depth (num_speculative_tokens), >= 1 */
    int32_t d;                 /* drafter width (bf16: a multiple of 64) */
    int32_t n_q, n_kv;         /* query / key-value heads; n_kv divides n_q */
    int32_t head_dim;          /* 64 or 128 */
    int32_t ffn;               /* SwiGLU width F (bf16: a multiple of 64) */
    int32_t vocab;             /* V; the MASK token id is V (row V of emb) */
    int32_t n_layers;          /* L >= 1 */
    int32_t page_size;         /* KV page size; must be 16 */
    int32_t max_pages_per_seq; /* block-table row length */
    pe_dtype dtype;            /* storage type of weights, hidden states, cache */
    float rms_eps;             /* RMSNorm epsilon (1e-6) */
    float rope_theta;          /* RoPE base (10000) */
} pe_config;

/* Drafter weights (device pointers; the arrays of per-layer pointers are host memory). */
typedef struct {
    const void *emb;       /* [(V+1)][d]; row V = learned emb(mask) */
    const void *h_shared;  /* [d]; learned shared hidden state of MASK rows */
    const void *fc;        /* [d][2d]; input = concat(emb, hidden), emb first */
    const void *const *norm_attn; /* [L] -> [d] */
    const void *const *wqkv;      /* [L] -> [(n_q+2*n_kv)*head_dim][d]: q heads, k heads, v heads */
    const void *const *wo;        /* [L] -> [d][n_q*head_dim] */
    const void *const *norm_mlp;  /* [L] -> [d] */
    const void *const *w_gate_up; /* [L] -> [2F][d]: F gate rows then F up rows */
    const void *const *w_down;    /* [L] -> [d][F] */
    const void *norm_final;       /* [d] */
    const void *lm_head;          /* [V][d] */
} pe_weights;

/* Paged drafter KV cache: per layer separate K and V pools
 * [num_pages][page_size][n_kv][head_dim]; post-RoPE keys are stored. */
typedef struct {
    void *const *k_cache; /* [L] device pointers (host array) */
    void *const *v_cache; /* [L] device pointers (host array) */
    int32_t num_pages;
} pe_kv;

/*
 * Stage (a): rebuild the drafter batch in one pass (P-EAGLE: Parallel
 * Speculative Decoding in vLLM, "vLLM implementation details": the fused
 * kernel copies previous token ids and positions, inserts the bonus token,
 * fills the parallel-draft slots with the MASK id, and emits the rejected
 * mask, the MASK mask and the hidden-state map; "KV cache and CUDA Graphs":
 * rejected tokens get PADDING_SLOT_ID = -1).
 *
 * In : prev_tokens [B][K+1], prev_pos [B][K+1] (the previous verify batch
 *      [last, d_1..d_K] and its positions), num_accepted [B], bonus [B],
 *      block_table [B][max_pages_per_seq] (physical page ids, -1 unused).
 * Out: per padded row (B*2K rows): input_ids, positions, slot_mapping (int64,
 *      -1 on rejected rows), is_rejected, is_mask (uint8 0/1), hidden_map
 *      (row of target_hidden, -1 on MASK rows); row_list [B*2K] (the valid
 *      rows in increasing order, then -1 padding), *n_valid (device int32),
 *      draft_rows [B*K] (index into row_list of t_1..t_K of each sequence:
 *      the NTP row, then the MASK rows).
 * Row r of sequence b: r < a: token prev_tokens[b][r+1] at prev_pos[b][r]
 * with hidden row b*(K+1)+r (shifted by one); r == a: bonus at prev_pos[b][a]
 * with hidden row b*(K+1)+a; a < r <= K: rejected (token 0, slot -1);
 * r = K+m: MASK id V at prev_pos[b][a]+m, hidden_map -1.
 * slot(p) = block_table[b][p/16]*16 + p%16.
 * num_pages bounds the page ids (device check PE_DEV_BAD_PAGE).
 */
pe_status pe_prepare_batch(const pe_config *cfg, const int32_t *prev_tokens, const int32_t *prev_pos,
                           const int32_t *num_accepted, const int32_t *bonus, const int32_t *block_table,
                           int32_t num_pages, int32_t *input_ids, int32_t *positions, int64_t *slot_mapping,
                           uint8_t *is_rejected, uint8_t *is_mask, int32_t *hidden_map, int32_t *row_list,
                           int32_t *n_valid, int32_t *draft_rows, int32_t *err_word, pe_stream_t stream);

/*
 * Stage (b): drafter input rows (P-EAGLE: Parallel Speculative Decoding in
 * vLLM, step 2 "Parallel Drafting" -- context rows pair emb(token) with the
 * target hidden state, the NTP row pairs emb(new) with h_context, MASK rows
 * pair emb(mask) with h_shared; "Hidden-state management" -- a dedicated copy
 * kernel broadcasts h_shared to the MASK slots and maps target hidden states
 * to their new rows).
 *
 * For i < *n_valid, with row = row_list[i]:
 *   x0[i] = concat(emb[input_ids[row]], is_mask[row] ? h_shared : target_hidden[hidden_map[row]])
 * target_hidden [B*(K+1)][d]; x0 [B*2K][2d] (compacted: only the first
 * *n_valid rows are written).  Rows are moved with bulk async copies, so
 * emb, target_hidden, h_shared and x0 must be 16-byte aligned and
 * d * sizeof(dtype) a multiple of 16.
 */
pe_status pe_scatter_hidden(const pe_config *cfg, const pe_weights *w, const void *target_hidden,
                            const int32_t *input_ids, const uint8_t *is_mask, const int32_t *hidden_map,
                            const int32_t *row_list, const int32_t *n_valid, void *x0, int32_t *err_word,
                            pe_stream_t stream);

/*
 * Stages (c)+(d): one drafter pass over the n_valid compacted rows and the LM
 * head with a fused argmax (P-EAGLE: Parallel Speculative Decoding in vLLM,
 * step 2 "Parallel Drafting": all positions pass through the N layers and
 * the LM head, predicting t_1..t_K at once).
 *
 * Per layer, each row's post-RoPE k and v are written to the cache at
 * slot_mapping[row] (skipped when -1) BEFORE attention; a row at position p
 * attends to its sequence's cache positions 0..p (prefix + this round's rows:
 * causal inside the draft block).  Only the B*K draft rows reach the LM head;
 * draft_tokens[b][k] = argmax over the vocabulary (the lowest index wins a
 * tie); logits are not written unless logits_dbg is non-null
 * ([B*K][V] fp32, debug only, costs a full write of the logits).
 *
 * x0 is pe_scatter_hidden's output; positions/slot_mapping/row_list/n_valid/
 * draft_rows are pe_prepare_batch's.  workspace: >= pe_workspace_bytes(cfg)
 * bytes, 256-byte aligned, contents need not be initialised; it must not be
 * used by two calls that run concurrently.
 */
pe_status pe_draft_forward(const pe_config *cfg, const pe_weights *w, const pe_kv *kv,
                           const int32_t *block_table, const void *x0, const int32_t *positions,
                           const int64_t *slot_mapping, const int32_t *row_list, const int32_t *n_valid,
                           const int32_t *draft_rows, void *workspace, size_t workspace_bytes,
                           int32_t *draft_tokens, float *logits_dbg, int32_t *err_word, pe_stream_t stream);

/*
 * pe_draft_forward for callers that cannot allocate device memory.  The P-EAGLE
 * pages have no counterpart of this call; it exists for deployment.
 *
 * Some callers have no way to obtain a workspace.  Examples are a plugin whose
 * host framework owns all device memory through its own pool and offers
 * plugins no allocation hook, and a latency-critical serving loop where
 * cudaMalloc is forbidden because it can synchronise the device.  For these
 * callers the scratch lives in one fixed array of PE_NOALLOC_SCRATCH_BYTES
 * inside this library.  Every GPU that loads the library reserves that array
 * until the process exits.
 *
 * Arguments and results are those of pe_draft_forward, without the workspace.
 * A config whose pe_workspace_bytes(cfg) exceeds PE_NOALLOC_SCRATCH_BYTES is
 * rejected with PE_ERR_SHAPE before any launch.  The first call on a device
 * looks up the array's device address on the current device (and so does the
 * first call after cudaDeviceReset gave the device a new context); make that
 * first call before any stream capture.  This call allocates nothing and calls no
 * allocating routine.  Every call shares the one array, and the array keeps
 * whatever the last call left in it.  The pass zeroes every counter and
 * accumulator it needs at its start, so leftover contents do no harm.  Two
 * calls that overlap on the GPU (different streams, or different host threads
 * without ordering) race on the array and corrupt each other's results.
 */
#define PE_NOALLOC_SCRATCH_BYTES (48u << 20)
pe_status pe_draft_forward_noalloc(const pe_config *cfg, const pe_weights *w, const pe_kv *kv,
                                   const int32_t *block_table, const void *x0, const int32_t *positions,
                                   const int64_t *slot_mapping, const int32_t *row_list, const int32_t *n_valid,
                                   const int32_t *draft_rows, int32_t *draft_tokens, float *logits_dbg,
                                   int32_t *err_word, pe_stream_t stream);

/*
 * Stage (e): greedy verification (vLLM Speculators: parallel drafting for
 * speculative decoding, "Production integration in vLLM": verification keeps
 * the target's output; greedy form).
 *   num_accepted_out[b] = max{ j <= K : draft[b][i] == target[b][i] for all i < j }
 *   bonus_out[b]        = target[b][num_accepted_out[b]]
 * draft_tokens [B][K], target_tokens [B][K+1] (the target's token after each
 * position of the verify batch [bonus, t_1..t_K]).
 */
pe_status pe_verify(const pe_config *cfg, const int32_t *draft_tokens, const int32_t *target_tokens,
                    int32_t *num_accepted_out, int32_t *bonus_out, pe_stream_t stream);

/*
 * DFlash-style KV injection (vLLM Speculators: parallel drafting for speculative
 * decoding, "DFlash": the verifier's hidden states are projected and injected
 * straight into the drafter's KV cache, so that the drafter attends to the
 * verifier's state without more input rows).  The page gives no formula; here the
 * projected state stands where a row's residual stream would, so each layer turns
 * it into k and v exactly as it does for its own rows.
 *
 * For sequence b and element j <= num_accepted[b] of its previous verify batch
 * (the accepted drafts and the bonus token's position), with
 * h = target_hidden[b*(K+1) + j] and p = prev_pos[b][j]:
 *   x = W_inj . h                          (w_inj [d][d], nn.Linear layout, no bias)
 *   per layer l: y = rms(x) * norm_attn[l]; k = RoPE(W_k[l] . y, p); v = W_v[l] . y
 * (W_k, W_v: the k and v head blocks of wqkv[l]) are written to layer l's cache
 * at slot(p) = block_table[b][p/16]*16 + p%16.  Elements j > num_accepted[b] are
 * not written.  Only w->norm_attn and w->wqkv are read from w.  prev_pos,
 * num_accepted, target_hidden are pe_step's / pe_prepare_batch's arrays of the
 * same names; workspace as for pe_draft_forward.  Device checks: an accepted
 * count outside [0, K] (PE_DEV_BAD_ACCEPTED: nothing of that sequence is
 * written), a position outside the block table (PE_DEV_BAD_POSITION), a page id
 * outside [0, num_pages) (PE_DEV_BAD_PAGE).
 */
pe_status pe_inject_kv(const pe_config *cfg, const pe_weights *w, const void *w_inj, const pe_kv *kv,
                       const int32_t *block_table, const int32_t *prev_pos, const int32_t *num_accepted,
                       const void *target_hidden, void *workspace, size_t workspace_bytes, int32_t *err_word,
                       pe_stream_t stream);

/*
 * Non-greedy drafting (vLLM Speculators: parallel drafting for speculative
 * decoding, "Production integration in vLLM": verification by rejection
 * sampling keeps the target's output distribution).  Draft row r = b*K + k
 * draws its token from the drafter's distribution
 *   q_r(v) = exp(logits[r][v] / temperature - lse[r]),
 *   lse[r] = log sum_v exp(logits[r][v] / temperature)       (natural log)
 * with the uniform u_draft[r] in [0, 1): the first v at which the running sum
 * of q_r exceeds u_draft[r] (inverse CDF; the sum runs in a fixed order, so the
 * draw is deterministic).  logits [B*K][V] fp32 are pe_draft_forward's
 * logits_dbg output; draft_tokens [B][K] and lse [B*K] are written.  workspace:
 * 256-byte aligned, >= pe_workspace_bytes(cfg) bytes (the same workspace as
 * pe_draft_forward may be passed; its contents are scratch).  Two launches:
 * statistics of every 512-entry step of every row, then one warp per row for the
 * draw.  A -inf logit is a masked entry: probability 0, never drawn (a row may
 * mask whole 512-entry steps).  A NaN or +inf logit sets PE_DEV_NONFINITE and
 * leaves the row's distribution undefined: the row's token is 0 and its lse NaN;
 * so does a row whose every logit is -inf.  temperature must be positive and
 * finite (else PE_ERR_INVALID_ARG).
 */
pe_status pe_sample_drafts(const pe_config *cfg, const float *logits, const float *u_draft, float temperature,
                           void *workspace, size_t workspace_bytes, int32_t *draft_tokens, float *lse,
                           int32_t *err_word, pe_stream_t stream);

/*
 * Verification by rejection sampling (speculative sampling) of drafts drawn by
 * pe_sample_drafts from the same logits, lse and temperature.
 * target_probs [B][K+1][V] fp32: p_k = target_probs[b][k] is the target's
 * distribution for the position of draft k (after element k of the verify
 * batch [bonus, t_1..t_K]); p_K follows the last draft.  For k = 0, 1, ...:
 * draft x = draft_tokens[b][k] is accepted when u_accept[b][k] * q(x) < p_k(x),
 * i.e. with probability min(1, p_k(x) / q(x)).  At the first rejection
 * num_accepted_out[b] = k and bonus_out[b] is drawn with u_resample[b] (inverse
 * CDF, as above) from the residual max(0, p_k - q), or from p_k when that
 * residual is all zero; with every draft accepted, num_accepted_out[b] = K and
 * the bonus is drawn from p_K.  u_accept [B][K], u_resample [B] in [0, 1).
 * workspace as for pe_sample_drafts.  A draft outside [0, V) sets
 * PE_DEV_BAD_TOKEN (and
 * counts as rejected); a target row with no positive finite mass sets
 * PE_DEV_NONFINITE (bonus 0).
 */
pe_status pe_verify_sampled(const pe_config *cfg, const int32_t *draft_tokens, const float *logits, const float *lse,
                            float temperature, const float *target_probs, const float *u_accept,
                            const float *u_resample, void *workspace, size_t workspace_bytes,
                            int32_t *num_accepted_out, int32_t *bonus_out, int32_t *err_word, pe_stream_t stream);

/*
 * One whole round on one stream: pe_prepare_batch -> pe_scatter_hidden ->
 * pe_draft_forward -> pe_verify, plus the next round's verify batch:
 * next_prev_tokens[b] = [bonus[b], t_1..t_K] and next_prev_pos[b][j] =
 * prev_pos[b][num_accepted[b]] + 1 + j (both [B][K+1]).  target_tokens are
 * the target's tokens for that verify batch (the target model is outside this
 * library).  Batch metadata and x0 live in the workspace
 * (>= pe_workspace_bytes(cfg)).
 *
 * In-place state.  The round's state arrays are read only by the batch rebuild
 * (the first launch), so the next state may overwrite them: next_prev_tokens may
 * be prev_tokens, next_prev_pos may be prev_pos, num_accepted_out may be
 * num_accepted and bonus_out may be bonus (each pair exactly the same pointer).
 * With all four in place, one call -- or a CUDA graph captured from it -- run
 * again after the caller refills target_hidden and target_tokens is the next
 * round (the multi-round drafting loop; the prefix grows by num_accepted + 1
 * positions per round, which the block table must cover).  No other output may
 * overlap an input or another output (err_word and the first
 * pe_workspace_bytes(cfg) bytes of the workspace count as outputs): such a call
 * returns PE_ERR_INVALID_ARG before anything is launched.
 */
pe_status pe_step(const pe_config *cfg, const pe_weights *w, const pe_kv *kv, const int32_t *block_table,
                  const int32_t *prev_tokens, const int32_t *prev_pos, const int32_t *num_accepted,
                  const int32_t *bonus, const void *target_hidden, const int32_t *target_tokens,
                  void *workspace, size_t workspace_bytes, int32_t *draft_tokens, int32_t *num_accepted_out,
                  int32_t *bonus_out, int32_t *next_prev_tokens, int32_t *next_prev_pos, float *logits_dbg,
                  int32_t *err_word, pe_stream_t stream);

/*
 * Tracing (optional).  pe_draft_forward and pe_step can record caller-created
 * CUDA events (cudaEvent_t) at their stage boundaries, on the launch stream,
 * so a caller can time every stage with cudaEventElapsedTime.  Boundary i:
 *   0 start, 1 after pe_prepare_batch, 2 after pe_scatter_hidden (pe_draft_forward
 *   records 0..2 at its start), 3 after the forward prologue, 4 after fc, then
 *   for each layer l the 7 points after: attention RMSNorm, QKV+RoPE+KV write,
 *   attention (incl. the chunk merge), o-proj, MLP RMSNorm, gate/up+SwiGLU,
 *   down -- i.e. 5 + 7*l + {0..6} -- then after the final RMSNorm, after the
 *   LM head + argmax, after verification (pe_step only).
 * pe_trace_points(cfg) = 8 + 7*n_layers boundaries.  Events beyond n_events
 * are not recorded; n_events = 0 turns tracing off.  The event array is host
 * memory and is copied; the events themselves must outlive their recording.
 * pe_step runs the rebuild, the input rows and the forward prologue in one
 * launch: its points 1, 2 and 3 all follow that launch.
 */
pe_status pe_set_trace_events(void *const *events, int32_t n_events);
int32_t pe_trace_points(const pe_config *cfg);

/* Number of kernels this library has launched since it was loaded (all threads). */
uint64_t pe_kernel_launches(void);

/*
 * Failure detection.  Inside a CTA the pipeline roles (copy issue, MMA issue,
 * softmax, epilogue) wait on each other through shared-memory barriers; no CTA
 * ever waits for another CTA.  Every such wait gives up after a time limit:
 * it records PE_DEV_TIMEOUT in *err_word, raises the CTA's abort flag (the
 * CTA's other roles stop waiting), waits for the CTA's own copies and MMAs in
 * flight, frees its tensor memory and returns; the rest of the call's kernels
 * still run (their results are then undefined) and the stream stays usable.
 * pe_set_wait_limit_ns sets that limit, in nanoseconds, for the kernels
 * launched afterwards by any thread (0 restores the default of one second; a
 * round takes well under a millisecond, so only a lost arrival reaches it).
 * Kernels captured into a CUDA graph keep the limit of the capture.
 */
pe_status pe_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook of the wait-expiry path above (for failure-detection tests only).
 * The next tensor-core GEMM launch (bf16 configs), from any thread, leaves
 * pipeline stage `stage` of its first CTA unarmed: no copy is issued into it
 * and no byte count is expected on its barrier, so the MMA role's wait on it
 * runs out after the wait limit.  One-shot: the launch that applies it clears
 * it; -1 clears it beforehand.  PE_ERR_INVALID_ARG for stage < -1.  A stage
 * beyond the CTA's pipeline leaves the launch unchanged.
 */
pe_status pe_test_skip_pipeline_stage(int32_t stage);

/* Workspace bytes needed by pe_draft_forward, pe_step, pe_sample_drafts,
 * pe_verify_sampled and pe_inject_kv for this config (0 if invalid); one workspace
 * serves them all. */
size_t pe_workspace_bytes(const pe_config *cfg);

/*
 * Validate a config without launching anything.  PE_ERR_SHAPE: a size out of range
 * (B*2K > 65536, n_kv not dividing n_q, ...); PE_ERR_UNSUPPORTED: a valid shape this
 * build has no kernel for: page_size other than 16, head_dim other than 64 or 128,
 * d > 10240 in bf16 or 5120 in fp32 (the input-row copy stages ten d-wide row halves in
 * shared memory), or for bf16 d or ffn not a multiple of 64 (the tensor-core GEMMs tile every
 * contraction in 64-wide k atoms) or more than 128 query vectors per (sequence, kv head).
 */
pe_status pe_check_config(const pe_config *cfg);

/* Static description of a status code. */
const char *pe_status_str(pe_status s);

#ifdef __cplusplus
}
#endif

#endif /* PE_H */
