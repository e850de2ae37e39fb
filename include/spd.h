/*
 * spd.h — C ABI of the GB300 speculative-pipeline-decoding hot path.
 *
 * Method: "Speculative Pipeline Decoding: Higher-Accuracy Drafting with Hidden Latency
 * via Pipeline Parallelism" (arXiv 2605.30852).  The target decoder is cut into n
 * pipeline stages; n in-flight tokens of one sequence each advance through their own
 * stage in one step (abstract; machine review, "The reading").  A Pipeline Draft
 * Module concatenates the step's INPUT hidden states at depth anchors, projects them,
 * runs Ls draft layers and the LM head to propose the next token, concurrently with
 * the step (review, "What carries the argument" / "Core claim").  Streaming
 * verification checks the draft behind each exiting token and, on rejection,
 * truncates the KV cache, flushes the pipeline and reseeds it (same section).  At
 * T > 0 verification is standard speculative rejection sampling (review,
 * "Assumptions", section 3.5).
 *
 * On one GPU the n stages are rows of grouped kernels; the draft module runs on a
 * second CUDA stream; verification and rollback run on the device with no host
 * round trip per step.
 *
 * Conventions for every call:
 *   - Return value: SPD_OK (0) or a positive SPD_E* code.  No call aborts or throws;
 *     spd_last_error() gives the text of the handle's last failure.
 *   - Ownership: weight, prompt and output pointers are BORROWED device pointers
 *     unless a call says otherwise; they must stay valid while the handle uses them.
 *     The workspace is borrowed too (caller allocates spd_workspace_bytes()).
 *     The library itself allocates no device memory.
 *   - Ordering: all device work is issued on the stream given to spd_create (plus an
 *     internal second stream joined back to it); calls return after issuing work,
 *     except where an argument named *_host receives a result (those synchronise).
 *   - Layout: matrices are row-major [out][in] in the dtype of spd_dims.dtype;
 *     norm gains are fp32 vectors.  The KV caches hold fp32 rows for every weight type
 *     (the cache's rounding would otherwise reach every later token's logits).
 */
#ifndef SPD_H
#define SPD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define SPD_OK 0
#define SPD_EINVAL 1     /* bad argument or unsupported shape                          */
#define SPD_ENOMEM 2     /* workspace too small                                        */
#define SPD_ECUDA 3      /* a CUDA runtime call failed (text in spd_last_error)        */
#define SPD_ESTATE 4     /* call out of order (e.g. spd_step before spd_prefill)       */
#define SPD_ECAPACITY 5  /* max_seq, max_new or the step-trace capacity would overflow */
#define SPD_EDEVICE 6    /* a kernel reported an error flag (bounds check failed)      */

/* element types: weights are SPD_F32 or SPD_BF16; the KV caches of a handle are fp32.
 * SPD_F16 names an fp16 K/V operand of the stand-alone attention call below */
#define SPD_F32 0
#define SPD_BF16 1
#define SPD_F16 2

#define SPD_MAX_ANCHORS 8
#define SPD_MAX_STAGES 31
#define SPD_MAX_LAYERS 128
#define SPD_MAX_PDM_LAYERS 16

/* Model shape.  Dense pre-norm decoder: RMSNorm, RoPE (rotate-half, base rope_theta),
 * grouped-query attention (Hq / Hkv in {1, 2, 4, 8}; head dim 64 or 128), SwiGLU FFN of width F, vocabulary V.  The
 * pages leave the architecture to the workloads they evaluate (Qwen3.5 dense shapes). */
typedef struct spd_dims {
    int32_t L, d, Hq, Hkv, hd, F, V;
    float rope_theta;
    float rms_eps;
    int32_t dtype; /* SPD_F32 or SPD_BF16 */
} spd_dims;

/* One decoder layer: wq [Hq*hd][d], wk/wv [Hkv*hd][d], wo [d][Hq*hd], w_gate/w_up [F][d],
 * w_down [d][F] (dtype), attn_norm/ffn_norm [d] fp32.  All device pointers, borrowed. */
typedef struct spd_layer_weights {
    const void *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down;
    const float *attn_norm, *ffn_norm;
} spd_layer_weights;

/* Target model: embed [V][d], layers = HOST array of L entries (copied at spd_create),
 * final_norm [d] fp32, lm_head [V][d]. */
typedef struct spd_target_weights {
    const void *embed;
    const spd_layer_weights *layers;
    const float *final_norm;
    const void *lm_head;
} spd_target_weights;

/* Pipeline Draft Module (a learned speculation network followed by an LM head; review
 * "Assumptions & free parameters", invented entities):
 * proj [d][n_anchors*d] (one bias-free projection of the concatenated anchors),
 * Ls target-shaped layers (HOST array, copied), its own final_norm [d] fp32, and an
 * LM head [V][d] that may alias the target's (tied; the usual case). */
typedef struct spd_pdm_weights {
    int32_t Ls;
    const void *proj;
    const spd_layer_weights *layers;
    const float *final_norm;
    const void *lm_head;
} spd_pdm_weights;

/* Run configuration.
 *   n            pipeline stages, 1 <= n <= min(L, SPD_MAX_STAGES); stage s holds target
 *                layers [floor(sL/n), floor((s+1)L/n)) unless stage_bounds says otherwise
 *                (machine review, "The reading": L/n layers per stage).
 *   anchors      strictly increasing depths in [0, L] with anchors[0] == 0 (the
 *                embedding; the paper reports training is unstable without it,
 *                review "free parameters", App. A.1).  Depth a = residual stream
 *                after a layers.
 *   temperature  0 = greedy (argmax, lowest id on ties); > 0 = sampling from
 *                softmax(z / T) with Philox4x32-10 uniforms keyed by seed.
 *   max_seq      KV capacity in positions (>= prompt_len + max_new + n).
 *   max_new      tokens to generate per spd_generate (the prefill's token counts).
 *   force_p      < 0: drafts come from the draft module.  In [0, 1]: forced-draft
 *                test mode — the draft for position p is forced_ref[p] with
 *                probability force_p, else a uniformly chosen other id; the draft
 *                module still runs (and is traced) but its token is not used.
 *   forced_ref   device int32 array indexed by absolute position (prompt included),
 *                length forced_ref_len; borrowed.
 *   graph        1: each spd_step launch replays a captured CUDA graph of one step.
 *   timing       1: CUDA events bracket every launch of the gate/up projection kernel
 *                (the largest weight stream); read them with spd_kernel_timing.
 *   stage_bounds all zero: the uniform split above.  Otherwise the n + 1 layer indices
 *                0 = b_0 < b_1 < ... < b_n = L, stage s holding layers [b_s, b_{s+1}): a
 *                non-uniform partition (review, referee report, minor comment on
 *                Appendix C.1, which gives such assignments without trying them).
 *   speculate    SPD_SPEC_INPUT: the draft module reads the step's INPUT states and runs
 *                on a second stream concurrently with the step (the paper's early-start
 *                schedule).  SPD_SPEC_OUTPUT: it runs after the step's target layers on
 *                their OUTPUT states (stage s's token at depth b_{s+1}, the exiting token
 *                at full depth): the input- vs output-state ablation the referee report
 *                lists.  Tokens and verification are the same; the drafts differ. */
#define SPD_SPEC_INPUT 0
#define SPD_SPEC_OUTPUT 1
typedef struct spd_config {
    int32_t n;
    int32_t n_anchors;
    int32_t anchors[SPD_MAX_ANCHORS];
    float temperature;
    uint64_t seed;
    int32_t max_seq;
    int32_t max_new;
    float force_p;
    const int32_t *forced_ref;
    int32_t forced_ref_len;
    int32_t graph;
    int32_t timing;
    int32_t stage_bounds[SPD_MAX_STAGES + 1];
    int32_t speculate;
} spd_config;

/* Per-run statistics.  N = committed tokens after the prefill's, K = pipeline steps,
 * alpha = N / K (commits per step, <= 1), S0 = alpha * n: the draft-free theoretical
 * speedup of the paper's Eq. 9 (review, "Circularity Check").  mean_kept_run is the
 * mean number of consecutive kept drafts between rejections (reported apart from
 * alpha: the page's identification of alpha with the acceptance length is garbled).
 * weight_bytes: bytes of weights the steps streamed (only occupied stages stream). */
typedef struct spd_stats {
    int64_t N, K, accepts, rejects;
    double alpha, S0, mean_kept_run;
    double weight_bytes;
    int32_t ls_exceeds_masking; /* 1 when Ls > floor(L/n): draft latency not hidden (sec. 3.4) */
    int32_t device_error;       /* nonzero: a kernel bounds check fired (code)            */
} spd_stats;

/* One step of the trace.  exit_pos: position of the token leaving the last stage
 * (-1 if none); draft/target: the verified draft and the target's token for
 * exit_pos+1; accept: 1 kept / 0 rejected / -1 no check; commit: the committed
 * token (-1 none); pdm_top: the draft module's argmax for the newest position;
 * new_draft: the token proposed for stage 0 (forced, argmax or sampled);
 * n_committed: N after the step; n_active: occupied stages during the step;
 * target_logit / pdm_logit: fp32 logits of target and pdm_top. */
typedef struct spd_trace_rec {
    int32_t t, exit_pos, draft, target, accept, commit, pdm_top, new_draft, n_committed, n_active;
    float target_logit, pdm_logit;
} spd_trace_rec;

typedef struct spd_handle spd_handle;

/* Bytes of device workspace spd_create needs for these shapes (no device work).  Of
 * pdm_shape_only only the Ls field is read (the draft module's shape; its pointers may be
 * NULL); NULL means no draft module. */
int spd_workspace_bytes(const spd_dims *d, const spd_pdm_weights *pdm_shape_only, const spd_config *cfg,
                        size_t *bytes);

/* Bind weights and workspace, build the stage plan and launch schedule.  stream is a
 * cudaStream_t (NULL = legacy default stream).  Returns SPD_EINVAL for bad shapes,
 * anchors or n; SPD_ENOMEM if ws_bytes is too small.  *out is NULL on failure. */
int spd_create(const spd_dims *d, const spd_target_weights *tw, const spd_pdm_weights *pw,
               const spd_config *cfg, void *workspace, size_t ws_bytes, void *stream, spd_handle **out);

/* Prefill (untimed part of the method): run the whole prompt (device int32 ids,
 * 1 <= prompt_len, prompt_len + max_new + n <= max_seq) through all target layers,
 * fill the draft module's cached prefix with full-depth features of every prompt
 * position (verified prefixes use depth-maximised features: machine review, "What
 * carries the argument"), pick the first token y0 (committed) and seed stage 0 with
 * it.  Resets the step counter, trace and statistics.  Errors: SPD_EINVAL (empty
 * prompt), SPD_ECAPACITY (too long for max_seq), SPD_ECUDA. */
int spd_prefill(spd_handle *h, const int32_t *prompt_dev, int32_t prompt_len);

/* Issue up to n_steps pipeline steps (steps after completion are no-ops on the
 * device).  One step (machine review, "The reading" and "What carries the argument"):
 * every occupied stage runs its layers on its own in-flight token; the draft module
 * proposes the token after the newest one from the anchor states; the token leaving the
 * last stage yields the target's token, the draft one position behind it is verified
 * (streaming verification; at T > 0 speculative rejection sampling, review
 * "Assumptions", section 3.5), and a rejection truncates the KV caches after the exiting
 * position, flushes the pipeline and reseeds stage 0 with the target's token.  No host
 * round trip happens inside a step.  If committed_host is non-NULL, synchronise and
 * store 1 + N (tokens generated so far, y0 included).  Errors: SPD_ESTATE before
 * spd_prefill, SPD_EINVAL for n_steps < 0, SPD_ECUDA, SPD_EDEVICE (a kernel's error flag,
 * reported when committed_host is given).  The caller's stream is joined back on every
 * return after work was issued. */
int spd_step(spd_handle *h, int32_t n_steps, int32_t *committed_host);

/* Generation of one sequence (abstract: n tokens of a single sequence advance per
 * step): spd_prefill, then spd_step batches until max_new tokens are committed,
 * polling the device between batches (never more steps than tokens still missing).
 * If buffers_on_host is 0, prompt and out_tokens are device pointers; if 1, they are
 * host pointers (prompt_len <= max_steps * L) and the copies happen inside the call.
 * out_tokens receives max_new ids (y0 first); *n_out_host (nullable) the count;
 * *stats_host (nullable) the statistics.  Errors as spd_prefill and spd_step, plus
 * SPD_ECAPACITY for a host prompt too long to stage; on every error after work was
 * issued the caller's stream is still ordered after it. */
int spd_generate(spd_handle *h, const int32_t *prompt, int32_t prompt_len, int32_t buffers_on_host,
                 int32_t *out_tokens, int32_t *n_out_host, spd_stats *stats_host);

/* Copy the first min(max_recs, K) trace records and, if len_host is non-NULL, the
 * per-layer KV valid lengths after each step ([rec][L] int32) to host memory;
 * *count_host = K.  The records are what the streaming verification decided each step
 * (exit position, verified draft, target token, keep flag, committed token; machine
 * review, "What carries the argument"), and the KV lengths show every truncation.
 * Synchronises.  SPD_ECUDA on a failed copy. */
int spd_get_trace(spd_handle *h, spd_trace_rec *recs_host, int32_t max_recs, int32_t *len_host,
                  int32_t *count_host);

/* Device view of the trace: records [count] and per-layer KV valid lengths [count][L],
 * both in the handle's workspace (valid until the next spd_prefill / spd_generate /
 * spd_reset / spd_destroy; read them on or after the handle's stream).  Synchronises to read
 * the count.  The same records as spd_get_trace without a copy. */
typedef struct spd_trace_view {
    const spd_trace_rec *recs;
    const int32_t *kv_len;
    int32_t count;
    int32_t L;
} spd_trace_view;
int spd_get_trace_view(spd_handle *h, spd_trace_view *out);

/* Statistics so far (synchronises). */
int spd_get_stats(spd_handle *h, spd_stats *stats_host);

/* Generated tokens so far (y0 first) into host memory; *count_host = 1 + N. */
int spd_get_tokens(spd_handle *h, int32_t *tokens_host, int32_t max_tokens, int32_t *count_host);

/* Internal buffers readable for inspection (tests): see spd_read_buffer. */
#define SPD_BUF_RESIDUAL 0   /* fp32 [n+1][d]: per-slot residual stream (slot ring)       */
#define SPD_BUF_ANCHORS 1    /* fp32 [n+1][n_anchors][d]: per-slot anchor states          */
#define SPD_BUF_LOGITS 2     /* fp32 [2][V]: last step's target-exit and draft logits     */
#define SPD_BUF_KCACHE 3     /* fp32 [max_seq][Hkv][hd] of target layer `index`          */
#define SPD_BUF_VCACHE 4
#define SPD_BUF_PDM_KCACHE 5 /* same, draft layer `index`                                */
#define SPD_BUF_PDM_VCACHE 6
#define SPD_BUF_SLOTS 7      /* int32 [3][n+1]: valid, position, token per slot           */
#define SPD_BUF_STATE 8      /* int32 [8]: head, t, N, done, pending, error, pdm_len, 0   */
#define SPD_BUF_PREFILL_LOGITS 9 /* fp32 [V]: logits at the last prompt position          */
#define SPD_BUF_PDM_RESIDUAL 10  /* fp32 [n+1][d]: draft rows' final residual streams     */

/* Copy `bytes` from internal buffer `which` (instance `index` for per-layer buffers),
 * starting at byte `offset`, to host memory.  Synchronises.  SPD_EINVAL when the
 * range falls outside the buffer. */
int spd_read_buffer(spd_handle *h, int32_t which, int32_t index, size_t offset, void *host_dst, size_t bytes);

/* Accumulated CUDA-event time (ms) and launch count of the timed kernel since the
 * last spd_prefill (config.timing must be 1).  Synchronises. */
int spd_kernel_timing(spd_handle *h, double *total_ms_host, int64_t *launches_host);

/* ---- standalone decode attention ------------------------------------------------------
 * The attention of one decode token, as each pipeline stage runs it (machine review "The
 * reading": every in-flight token attends to all earlier positions of its layer's KV
 * cache): out[h] = softmax(q[h] . K[:, h/G]^T / sqrt(hd)) V[:, h/G] over positions
 * 0..seq_len-1, G = Hq / Hkv.
 *   q      device fp32 [Hq][hd] (already rotated by RoPE)
 *   k, v   device [seq_len][Hkv][hd] in dtype (SPD_F32, SPD_BF16 or SPD_F16) — the KV-cache
 *          layout
 *   out    device fp32 [Hq][hd]
 *   Hq / Hkv in {1, 2, 4, 8}; hd 64 or 128; 1 <= seq_len <= 16384; q, k, v, out 16-byte
 *   aligned.  Split-K over 128-position chunks merged in chunk order (deterministic).
 * spd_attention_scratch_bytes gives the scratch size; the scratch (device, 256-byte
 * aligned, borrowed) needs no initialisation.  Work is queued on `stream`; the call does
 * not synchronise.  Errors: SPD_EINVAL (shape, pointer, alignment), SPD_ENOMEM (scratch
 * too small), SPD_ECUDA; text in spd_ops_last_error(). */
int spd_attention_scratch_bytes(int32_t Hq, int32_t Hkv, int32_t hd, int32_t seq_len, size_t *bytes);
int spd_attention_decode(int32_t dtype, int32_t Hq, int32_t Hkv, int32_t hd, int32_t seq_len, const float *q,
                         const void *k, const void *v, float *out, void *scratch, size_t scratch_bytes, void *stream);

/* Scratch-free spd_attention_decode (no counterpart in the paper; a library convenience).
 * For callers that cannot lend device memory — all of theirs is owned by another
 * allocator, or a cudaMalloc and its implicit synchronisation is not acceptable where
 * they run.  Same arguments, result and errors as spd_attention_decode minus the
 * scratch: the split-K partials live in a 1 MiB array inside the library, reserved on
 * every GPU that loads it until the process exits.  A call fits when
 * 256 + Hq * ceil(seq_len / 128) * (hd + 4) * 4 <= 1048576 bytes (e.g. Hq 32, hd 128:
 * seq_len up to 7936).  Larger shapes fail with SPD_ECAPACITY.  The entry point itself allocates
 * nothing (no cudaMalloc / cudaFree).  Its first call on a device looks up the array's
 * device address for that device (make that first call before any stream capture).
 * Every call shares the array: each clears what must start at zero, and calls that
 * overlap on the GPU (other streams, other threads) race and give wrong results. */
int spd_attention_decode_noalloc(int32_t dtype, int32_t Hq, int32_t Hkv, int32_t hd, int32_t seq_len,
                                 const float *q, const void *k, const void *v, float *out, void *stream);

/* Text of the calling thread's last failure of a standalone entry point ("" if none). */
const char *spd_ops_last_error(void);

/* Return to the post-create state (keeps weights and workspace): the run state
 * (step counter, committed count, slot ring, statistics) is cleared; the next call must
 * be spd_prefill or spd_generate.  Synchronises.  SPD_ECUDA on failure. */
int spd_reset(spd_handle *h);

/* Release streams, events and graphs (not the borrowed memory).  NULL is a no-op. */
void spd_destroy(spd_handle *h);

/* Text of the handle's last error ("" if none); with h == NULL the last error of a
 * failed spd_create / spd_workspace_bytes on this thread. */
const char *spd_last_error(const spd_handle *h);

#ifdef __cplusplus
}
#endif
#endif /* SPD_H */
