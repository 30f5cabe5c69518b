/*
 * k2.h -- C ABI of libk2, the GB300 (sm_103a) token-generation hot path of a
 * dense decoder-only GQA transformer of the K2-Horizon-3.7B shape.
 *
 * What the calls compute is the model of the k2-burn README:
 *   - "Model shape": hidden 2560, 36 layers, 32 query heads over 8 KV heads
 *     (GQA, 4x repeat), head_dim 128, SwiGLU intermediate 10240,
 *     layernorm_num_groups 2, vocab 250624, rms_norm_eps 1e-6, untied lm_head;
 *   - "Status: v0": GroupedRMSNorm, split-half RoPE, GQA attention, SwiGLU MLP,
 *     a preallocated per-layer KV cache with a configurable context window and
 *     storage dtype, prefill + single-token decode, temperature 0 = greedy
 *     argmax;
 *   - "KV cache storage": the context bounds the cache; a prompt that does not
 *     fit is rejected, not truncated; KV stored as fp32, f16, or symmetric int8
 *     with per-row fp16 scales;
 *   - "Project layout": decoder layer = norm+attn residual, norm+mlp residual;
 *     model = embed -> layers -> norm -> lm_head.
 * The error conventions follow kimi-k3-in-c k3_run.c: refuse rather than
 * clamp (argument validation), and never hand back an output that was not
 * written (forward failure / "RUN INVALID").
 *
 * Conventions common to every call:
 *   - Pointers named d_* and every weight pointer are DEVICE pointers of the
 *     current CUDA device; all other pointers are host pointers.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued asynchronously on it; outputs are valid once
 *     the stream has reached the end of the call's work.
 *   - The library allocates no device memory.  The caller provides the
 *     workspace (k2_workspace_bytes) and every input/output buffer, and keeps
 *     them alive until k2_free.  k2_init_weights packs every projection
 *     matrix (Wq, Wk, Wv, Wo, W_gate, W_up, W_down, lm_head) into the
 *     workspace in the layout the kernels stream; once its work has completed
 *     on the stream the caller may free those.  The embedding table and the
 *     norm gains are read in place and must outlive the context.
 *   - A non-zero k2_status means the call had no effect on the context and
 *     enqueued no work; k2_last_error(ctx) says why.  Faults detected on the
 *     device (a token id outside the vocabulary, a NaN logit, a bounded wait
 *     that ran out, a position outside the cache, a weight or activation
 *     beyond fp16's range in the fp16-operand prefill) never trap: they set a
 *     device guard word that k2_sync_status reports.
 */
#ifndef K2_H
#define K2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  K2_OK = 0,
  K2_ERR_ARG = 1,          /* null pointer, bad index, bad option */
  K2_ERR_SHAPE = 2,        /* inconsistent shape (e.g. hidden % norm_groups != 0) */
  K2_ERR_UNSUPPORTED = 3,  /* a shape/dtype the kernels are not built for */
  K2_ERR_TOKEN_RANGE = 4,  /* reserved for host-checked token ids */
  K2_ERR_CONTEXT_FULL = 5, /* the tokens do not fit the remaining context */
  K2_ERR_WORKSPACE = 6,    /* workspace missing, misaligned or too small */
  K2_ERR_CUDA = 7,         /* a CUDA runtime call failed */
  K2_ERR_DEVICE_GUARD = 8, /* the device guard word is set (k2_sync_status) */
  K2_ERR_STATE = 9         /* a saved cache state that is not this library's, is damaged, or was
                              written for another model architecture or KV format */
} k2_status;

typedef enum { K2_F32 = 0, K2_BF16 = 1, K2_F16 = 2, K2_I8 = 3, K2_F8 = 4, K2_Q4 = 5 } k2_dtype;

/* Model shape and run limits (k2-burn README, "Model shape" and "KV cache
 * storage").  weight_dtype is K2_F32, K2_BF16, K2_F8 or K2_Q4; kv_dtype is
 * K2_F32, K2_F16 or K2_I8.  K2_F8 and K2_Q4 (k2-burn README, "Post-training
 * quantization" and "Quantization": fp8 E4M3 and int4 block-64 checkpoints;
 * only the Linear weights are quantized): the weights are given in bf16 and
 * k2_init_weights stores every projection matrix and the lm_head as fp8 E4M3
 * rows with one fp32 scale per row (K2_F8, see k2_quantize_fp8), or as int4
 * codes with one fp32 scale per 64 weights of a row (K2_Q4, see
 * k2_quantize_q4); the embedding and the norm gains stay bf16.  Such a model
 * decodes on the persistent step only and is refused where that step is not
 * available.  Prompts of >= 8 tokens with K2_F8 weights run through the
 * tensor-core GEMMs over bf16 copies of the codes (exact), each row's scale
 * applied to its outputs, the last token through the persistent step; with
 * K2_Q4 weights each layer's matrices are first dequantized (code * scale)
 * into bf16 high and low halves in a one-layer scratch, and the GEMMs add the
 * low halves' products (~16 bits of every weight), the last token again
 * through the persistent step.  max_context = KV rows per sequence (prompt + generated tokens);
 * max_batch = number of independent sequences. */
typedef struct {
  int32_t hidden, n_layers, n_heads, n_kv_heads, head_dim, intermediate, norm_groups, vocab;
  int32_t max_context, max_batch;
  float eps, rope_theta;
  int32_t weight_dtype, kv_dtype;
} k2_config;

/* Device pointers to the weights, nn.Linear layout [out_features, in_features],
 * row-major, in weight_dtype.  The per-layer members are HOST arrays of
 * n_layers device pointers.  Shapes: embed, lm_head [vocab, hidden];
 * *_norm [hidden]; wq [n_heads*head_dim, hidden]; wk, wv
 * [n_kv_heads*head_dim, hidden]; wo [hidden, n_heads*head_dim];
 * w_gate, w_up [intermediate, hidden]; w_down [hidden, intermediate].
 * Every pointer must be 16-byte aligned. */
typedef struct {
  const void* embed;
  const void* lm_head;
  const void* final_norm;
  const void* const* attn_norm;
  const void* const* wq;
  const void* const* wk;
  const void* const* wv;
  const void* const* wo;
  const void* const* mlp_norm;
  const void* const* w_gate;
  const void* const* w_up;
  const void* const* w_down;
} k2_weights;

typedef struct k2_ctx k2_ctx;

/* Facts about a context, for tests and measurement. */
typedef struct {
  int32_t kv_capacity;   /* allocated KV rows per sequence (>= max_context) */
  int32_t num_sms;
  int32_t attn_splits;   /* key-range splits of the batch-1 attention launch */
  int32_t gemv_grid;     /* CTAs of the batch-1 GEMV launches */
  int64_t kv_bytes;      /* bytes of the KV cache region */
  int64_t repack_bytes;  /* bytes of the packed projection weights */
  int64_t scratch_bytes; /* everything else in the workspace */
  int32_t persistent_grid;   /* CTAs of the persistent batch-1 step (0: not available) */
  int32_t persistent_splits; /* its key-range splits per KV head */
  int32_t tc_prefill;        /* 1: prompts of >= 8 tokens run through the tensor-core GEMMs
                                (bf16 weights, or fp8 weights through bf16 copies of their codes) */
  int32_t tc_batched;        /* 1: batched decode and speculative verification on the tensor
                                cores (bf16 weights only) */
} k2_info;

/* ---- set-up -------------------------------------------------------------- */

/* Bytes of workspace k2_init_weights needs for this config on the current
 * device: repacked weights + KV cache + rope table + activations.  0 if the
 * config is invalid or unsupported (k2_init_weights then says why). */
size_t k2_workspace_bytes(const k2_config* cfg);

/* Validates the config (kimi-k3-in-c k3_run.c: an untrusted config aborts
 * rather than falls back; k2-burn README "Limitations": out-of-scope
 * checkpoints hard-error), carves the workspace (256-byte aligned, at least
 * k2_workspace_bytes), packs the projection weights into it (QKV fused with
 * RoPE pair order, gate/up interleaved, every matrix in row pairs of
 * 512-byte chunks), builds the RoPE table and zeroes the sequence lengths.  Enqueued on
 * `stream`.  On success *out owns host memory only; release with k2_free. */
k2_status k2_init_weights(const k2_config* cfg, const k2_weights* w, void* d_workspace, size_t ws_bytes,
                          void* stream, k2_ctx** out);

/* Releases the host-side context.  The workspace is the caller's. */
void k2_free(k2_ctx* ctx);

/* Message of the last failed call on this context ("" if none). */
const char* k2_last_error(const k2_ctx* ctx);

k2_status k2_get_info(const k2_ctx* ctx, k2_info* info);

/* ---- the hot path --------------------------------------------------------- */

/* Prefill: appends the n tokens d_tokens[0..n) to sequence `seq` at its
 * current length (k2-burn README, "Status: v0": prefill + single-token decode)
 * and writes the greedy next token (first index of the max logit, kimi-k3-in-c
 * k3_run.c `argmax_`) to *d_next_token.  If d_logits is not NULL, the last
 * position's fp32 logits [vocab] are written there (kimi-k3-in-c k3_run.c:
 * `forward` returns last-position logits).  K2_ERR_CONTEXT_FULL if
 * length + n > max_context: the prompt is rejected, not truncated. */
/* With bf16 or fp8 weights (and option K2_OPT_TC_PREFILL) a prompt of 8 or more
 * tokens is processed in blocks of up to 2048 tokens: the projections as tcgen05
 * tensor-core GEMMs (activations split into two bf16 halves, fp32 accumulation;
 * fp8: the codes as bf16, each output row times its scale), causal attention over
 * the cache, the residual stream in fp32.  With fp8 weights the last token takes
 * the persistent step, which ends in the fp8 lm_head. */
k2_status k2_prefill(k2_ctx* ctx, int32_t seq, const int32_t* d_tokens, int32_t n, int32_t* d_next_token,
                     float* d_logits, void* stream);

/* One decode step for sequences 0..batch-1: sequence b consumes d_tokens[b]
 * at position length(b), appends its K/V, and gets its greedy next token in
 * d_next[b] (logits in d_logits[b*vocab ..] if d_logits is not NULL).
 * d_next may equal d_tokens (the step then feeds itself when replayed).
 * K2_ERR_CONTEXT_FULL if any of the sequences is at max_context. */
k2_status k2_decode_step(k2_ctx* ctx, const int32_t* d_tokens, int32_t batch, int32_t* d_next, float* d_logits,
                         void* stream);

/* The decoder layers alone for one new token per sequence: d_x [batch, hidden]
 * fp32 is the residual stream entering layer 0 and is overwritten with the
 * residual leaving the last layer.  K/V are appended and lengths advance as
 * in k2_decode_step; no embedding, final norm or lm_head. */
k2_status k2_decode_layers(k2_ctx* ctx, float* d_x, int32_t batch, void* stream);

/* ---- cache management ------------------------------------------------------ */

/* Sets the length of sequence `seq` (or of all sequences, seq = -1) to 0.
 * Memory is not cleared. */
k2_status k2_kv_reset(k2_ctx* ctx, int32_t seq, void* stream);

/* Sets the length of sequence `seq` to len (0 <= len <= max_context): rows
 * 0..len-1 are taken to be valid (e.g. filled through k2_kv_view). */
k2_status k2_kv_set_len(k2_ctx* ctx, int32_t seq, int32_t len, void* stream);

/* Device pointers of the cache of (layer, seq): K and V are
 * [n_kv_heads][kv_capacity][head_dim] in kv_dtype; for K2_I8 the fp16 row
 * scales are [n_kv_heads][kv_capacity] (NULL otherwise).  *len = current
 * length (host view). */
k2_status k2_kv_view(k2_ctx* ctx, int32_t layer, int32_t seq, void** k, void** v, void** k_scale, void** v_scale,
                     int32_t* len);

/* ---- sampling ------------------------------------------------------------------
 *
 * The pages' generation knobs (k2-burn README, "Sampling + greedy
 * generation"): temperature 0 is the greedy argmax of k2_decode_step and
 * k2_prefill, unchanged; temperature > 0 draws the next token instead, with
 * top-k / top-p / min-p truncation, a repetition penalty and a seed.  For a
 * row of logits l (fp32, one per vocabulary entry), in this order:
 *   1. repetition penalty r (1 = off): each DISTINCT id among the sequence's
 *      tokens so far (the prompt and every decode input, i.e. the rows of its
 *      cache) has l -> l / r if l > 0, l * r otherwise;
 *   2. z = l / temperature; z_max their maximum (NaN logits are excluded);
 *   3. top-k (0 = off): keep z >= the k-th largest z (ties at it all kept);
 *   4. weights w = exp(z - z_max) (fp32, computed by the library's own exp so
 *      that it is reproducible), masses m = floor(w * 2^32) of the top-k
 *      survivors, W their sum;
 *   5. top-p (1 = off): keep the tokens whose strictly heavier survivors weigh
 *      less than top_p * W (the smallest most-probable set reaching top_p;
 *      tied weights are kept or dropped together);
 *   6. min-p (0 = off): keep w >= min_p (the probability relative to the top one);
 *   7. draw: x = Philox4x32-10(counter = (position the token will take,
 *      sequence index, 0, 0), key = (seed low 32 bits, seed high 32 bits)),
 *      u = (x[0] >> 8) / 2^24; the token is the first index, in vocabulary
 *      order, whose running sum of kept masses exceeds floor(u * total).
 * Draws depend only on (seed, sequence, position) and the logits, so a
 * resumed sequence (k2_kv_load) continues with the same draws. */
typedef struct {
  float temperature;        /* 0 = greedy (the default) */
  int32_t top_k;            /* 0 = off */
  float top_p;              /* (0, 1]; 1 = off */
  float min_p;              /* [0, 1]; 0 = off */
  float repetition_penalty; /* > 0; 1 = off */
  uint64_t seed;
} k2_sampling;

/* Sets the sampling of this context's decode steps and prefills (NULL or
 * temperature 0: greedy).  The logits of a sampled step are written to d_logits
 * when the call passes one, else to workspace scratch; the sampler is one
 * cooperative launch after the step.  Recorded decode graphs are dropped.
 * K2_ERR_ARG for parameters outside the ranges below; K2_ERR_UNSUPPORTED if
 * max_batch rows of this vocabulary do not fit the device's shared memory. */
k2_status k2_set_sampling(k2_ctx* ctx, const k2_sampling* params);

/* The sampler alone, with this context's sampling parameters, on caller
 * logits d_logits [rows][vocab] (rows <= max_batch): row r draws into
 * d_next[r] with counter (d_position[r], first_seq + r); its repetition
 * penalty covers d_seen[r * seen_stride .. + d_seen_len[r]) (d_seen NULL: no
 * penalty).  All pointers are device memory.  K2_ERR_ARG if sampling is not
 * set (temperature 0). */
k2_status k2_sample_logits(k2_ctx* ctx, const float* d_logits, int32_t rows, const int32_t* d_seen,
                           int32_t seen_stride, const int32_t* d_seen_len, const int32_t* d_position,
                           int32_t first_seq, int32_t* d_next, void* stream);

/* The sampler's generator: d_out[4 * i + w] = word w of Philox4x32-10 with
 * counter (first + i, c1, c2, c3) and key (key low, key high), i < n. */
k2_status k2_philox(uint32_t first, int32_t n, uint32_t c1, uint32_t c2, uint32_t c3, uint64_t key, uint32_t* d_out,
                    void* stream);

/* ---- speculative decoding ------------------------------------------------------
 *
 * kimi-k3-in-c k3_run.c, --spec: draft ids by n-gram lookup in the sequence
 * itself and verify them in one batched pass; only the prefix the model
 * itself would have emitted greedily is accepted.
 *
 * Drafting (the rule stated for the page's spec_draft): for n = 4, then 3,
 * take the two latest earlier occurrences of the last n ids of h_tokens;
 * propose the ids that followed the latest one (at most max_draft, at most
 * 8, and not past the end of h_tokens); with a second occurrence, only as
 * far as the two continuations agree and the older one stays short of the
 * latest occurrence.  The first n giving a non-empty draft wins.  All
 * occurrences come from one linear pass (the Z-algorithm over the history
 * read backwards).  Returns the number of drafted ids written to h_out (host
 * memory; 0 = no draft).  No context, no GPU. */
int32_t k2_spec_draft(const int32_t* h_tokens, int32_t n_tokens, int32_t max_draft, int32_t* h_out);

/* One speculative step of sequence seq.  h_tokens [n_tokens] (host) holds
 * the sequence's cached ids followed by the next input id, so n_tokens =
 * its cache length + 1.  The input and up to max_draft drafted ids (see
 * k2_spec_draft, with max_draft capped so the rows fit max_context) are
 * appended in one tensor-core pass that computes the greedy id after every
 * one of them; draft i is accepted while it equals the greedy id after the
 * ids before it.  The cache keeps the rows of the input and of the accepted
 * drafts; h_out (room for max_draft + 1) receives the greedy ids after them
 * (accepted + 1 ids, the last one the next input), *n_out their count.
 * Without a draft (or without tensor-core prefill: fp32 weights) the step
 * is an ordinary decode step of seq.  Greedy only: K2_ERR_UNSUPPORTED while
 * sampling is set.  Waits for `stream`.  The verification pass runs the
 * prefill arithmetic, so where the top two logits of a step lie within its
 * ~1e-6 difference from the decode step's, the ids can differ from serial
 * decoding. */
k2_status k2_decode_speculative(k2_ctx* ctx, int32_t seq, const int32_t* h_tokens, int32_t n_tokens,
                                int32_t max_draft, int32_t* h_out, int32_t* n_out, void* stream);

/* Test hook: the fp32 logits [*rows][vocab] (device memory owned by the
 * context) of the last k2_decode_speculative call.  Row i holds the logits
 * after the input and drafts 0..i-1, for every position the pass verified
 * (the input and all drafts, accepted or not); a step without a draft leaves
 * one row.  *rows = 0 (and *d_logits NULL) for models without a tensor-core
 * path.  Valid until the next call on the context. */
k2_status k2_spec_logits_view(k2_ctx* ctx, float** d_logits, int32_t* rows);

/* ---- saved cache state ------------------------------------------------------
 *
 * A sequence's cache can be written to host memory and restored later, into
 * this or another context, so that a resumed conversation pays only for its
 * new tokens (kimi-k3-in-c k3_run.c, "conversation state").  The state holds
 * only the occupied rows, so the restoring context may have a different
 * max_context or max_batch.  Its header carries a fingerprint of the model
 * architecture and KV format; a state written for anything else is refused,
 * because restoring it would give fluent, wrong output.
 *
 * Layout (little-endian, all offsets from the start of the state):
 *   0   char magic[4] = "K2ST"; int32 version = 1
 *   8   int32 fp[12]: hidden, n_layers, n_heads, n_kv_heads, head_dim,
 *       intermediate, norm_groups, vocab, weight_dtype, kv_dtype, and the bit
 *       patterns of eps and rope_theta
 *   56  int32 cached (rows per layer and KV head), int32 n_tokens
 *   64  int64 row_bytes (one K or V row), int64 scale_bytes (2 for K2_I8, else 0),
 *       int64 total_bytes
 *   88  int32 reserved[2] = 0
 *   96  int32 tokens[n_tokens] (the caller's token ids, e.g. the conversation so far)
 *   then, 16-byte aligned, per layer: K [n_kv_heads][cached] rows, V the same,
 *       and for K2_I8 the fp16 scales of K [n_kv_heads][cached], then of V. */
#define K2_STATE_HEADER_BYTES 96

/* Bytes of the state k2_kv_save writes for sequence seq with n_tokens ids. */
k2_status k2_kv_state_bytes(const k2_ctx* ctx, int32_t seq, int32_t n_tokens, size_t* bytes);

/* Writes sequence seq's state into h_buf (host memory of buf_bytes bytes;
 * pinned memory copies fastest) with the n_tokens ids of h_tokens (host,
 * nullable when n_tokens = 0); *written = its size.  Waits for `stream`
 * first and returns when the copies are done.  K2_ERR_WORKSPACE if buf_bytes
 * is too small; K2_ERR_DEVICE_GUARD if the device guard is set (the cache may
 * not hold what the host expects). */
k2_status k2_kv_save(k2_ctx* ctx, int32_t seq, const int32_t* h_tokens, int32_t n_tokens, void* h_buf,
                     size_t buf_bytes, size_t* written, void* stream);

/* Checks a state in host memory against a config without a context: magic,
 * version, fingerprint and sizes.  K2_OK and *cached, *n_tokens (nullable) if
 * it could be loaded into a context of cfg's architecture and KV format;
 * K2_ERR_STATE otherwise (the reason is not kept: there is no context). */
k2_status k2_kv_peek(const k2_config* cfg, const void* h_buf, size_t buf_bytes, int32_t* cached, int32_t* n_tokens);

/* Restores a state into sequence seq (its previous rows are replaced), sets
 * its length to the saved row count, takes the first min(n_tokens, rows)
 * saved ids as the sequence's token history (what the repetition penalty
 * counts as seen), and copies the saved token ids into h_tokens (host,
 * max_tokens entries; nullable when max_tokens = 0).
 * Enqueued on `stream`, then waited for.  Before anything is changed:
 * K2_ERR_STATE for a state of another architecture or KV format or a damaged
 * one, K2_ERR_CONTEXT_FULL if its rows do not fit this context's
 * max_context, K2_ERR_ARG if max_tokens is smaller than the saved count. */
k2_status k2_kv_load(k2_ctx* ctx, int32_t seq, const void* h_buf, size_t buf_bytes, int32_t* h_tokens,
                     int32_t max_tokens, void* stream);

/* Device pointer of the fp32 residual stream of launch slot b ([hidden]); after
 * a decode step it holds the residual leaving the last layer for sequence b
 * (before the final norm). */
k2_status k2_hidden_view(k2_ctx* ctx, int32_t b, float** d_x);

/* ---- status, options, measurement ------------------------------------------- */

/* Waits for `stream` and reads the device guard word: K2_OK if clear,
 * K2_ERR_DEVICE_GUARD (with the reasons in k2_last_error) otherwise. */
k2_status k2_sync_status(k2_ctx* ctx, void* stream);

/* Clears the device guard word and re-reads every sequence's length from the
 * device (a step that failed on the device did not advance its sequences);
 * waits for `stream`. */
k2_status k2_clear_status(k2_ctx* ctx, void* stream);

typedef enum {
  K2_OPT_PDL = 0,         /* 1 (default): programmatic dependent launch between kernels */
  K2_OPT_GRAPH = 1,       /* 1: k2_decode_step records a CUDA graph per (batch, buffers,
                             stream) on first use and replays it (stream must not be NULL) */
  K2_OPT_ATTN_SPLITS = 2, /* > 0: force the number of attention key splits of the kernel chain (tests) */
  K2_OPT_PERSISTENT = 3,  /* 1 (default): batch-1 tokens run as one persistent cooperative kernel
                             (one CTA per SM, dataflow waits between the phases of a layer) when the
                             shape allows; 0: always the chain of per-step kernels */
  K2_OPT_TC_PREFILL = 4,  /* 1 (default): bf16, fp8 and int4 models prefill prompts of >= 8 tokens with
                             tensor-core GEMMs over blocks of up to 2048 tokens (int4: each layer's weights
                             dequantized into bf16 hi + lo halves first, three MMAs per K step); 0: one
                             decode step per token */
  K2_OPT_TC_DECODE = 5,   /* 1 (default): a bf16 decode step of batch >= 2 reads the weights once for
                             all sequences (tensor-core GEMMs, N = batch); 0: one token at a time */
  K2_OPT_WAIT_LIMIT_US = 6, /* how long (microseconds, 1 .. 1000000; default 1000000) a CTA of the
                             persistent step waits for words another CTA publishes before it gives up:
                             the step then ends early, raises the guard (K2_ERR_DEVICE_GUARD,
                             "bounded-wait-timeout"), writes no token and does not advance the
                             sequence.  Waits for the CTA's own copies keep their 1 s limit. */
  K2_OPT_STALL_PHASE = 7, /* test of that path: phase p (1 .. 5 * n_layers; layer l's phases are
                             5l + 0 QKV, 1 attention, 2 o_proj, 3 gate/up, 4 down, and 5 * n_layers
                             is the lm_head) of the persistent step waits for words that no phase
                             writes, so its waits run out; -1 (default) turns it off */
  K2_OPT_L2_AHEAD = 8,    /* persistent step: at the start of a phase, each warp fetches into L2 this many
                             of its next weight / K-V slots beyond those in flight (0 .. 64; default 2) */
  K2_OPT_L2_AHEAD_PHASES = 9, /* the phase kinds that do so, bit j for kind j (0 QKV, 1 attention, 2 o_proj,
                             3 gate/up, 4 down, 5 lm_head); default 0x18 (gate/up, down), 0 for fp8 and int4 weights */
  K2_OPT_TRACE = 10,      /* measurement: the device address (as an integer; 0 = off) of a caller's buffer of
                             (5 * n_layers + 2) * persistent_grid * 4 uint64 words; each persistent step then
                             writes, per phase q and CTA c, the SM's %clock64 at [(q * grid + c) * 4 + k]:
                             k = 0 phase start, 1 input ready, 2 slots consumed, 3 phase end; and at
                             [((5 * n_layers + 1) * grid + c) * 4 + {0, 1}] the %globaltimer ns and the
                             %clock64 of the CTA's start, which align the SMs' clocks */
  K2_OPT_PREFILL_ATTN = 11, /* prefill attention of fp16 caches (head_dim 64 / 128, 4 query heads per KV head):
                             1 (default) on the 5th-generation tensor cores (tcgen05, S and O in tensor
                             memory), 0 on mma.sync */
  K2_OPT_PREFILL_SPLIT = 12, /* tensor-core prefill of blocks over 16 tokens: 1 feeds the GEMMs each
                             fp32 activation as two bf16 halves (hi + lo, two MMAs: the decode step's
                             precision) and the tcgen05 attention its queries and probabilities as two
                             fp16 halves; 2 keeps the GEMMs' halves but gives the attention single fp16
                             queries and probabilities; 0 feeds single bf16 activations and single fp16
                             queries and probabilities (the model dtype; half the MMAs).  Decode steps and
                             blocks of up to 16 tokens always keep the halves; int4 weights keep the GEMMs'.
                             Measured on the 36-layer 3.7B shape (512-token prompt, 256 greedy steps, fp16
                             KV): 1 gives 100 % teacher-forced agreement, relative L2 4.3e-4 (4.5e-4 on the
                             prefill's logits); 2 gives 100 %, 5.1e-4 (1.4e-3); 0 gives 94.9-96.5 %,
                             1.1e-2 (2.1e-2), below the bf16 parity bars.  3 (bf16 weights, fp16
                             caches) runs every prefill contraction on single fp16 operands: each weight
                             matrix is converted to fp16 per layer (exact in fp16's normal range, values
                             beyond +-65504 raise the device guard), the activations enter as fp16 (11
                             significant bits, 3 more than bf16), one MMA per K step; elsewhere (fp8 / int4
                             weights, int8 or fp32 caches) 3 acts as 1.  3 is the default: on the same
                             model and test it gives 99.2-100 % agreement, relative L2 2.1e-3 (3.6e-3 on
                             the prefill's logits), and a 4096-token prompt takes 46.5 ms against 73.3 ms
                             with 1 and 66.3 ms with 2 (1 and 2 measured before the prefill kernels ran
                             under PDL). */
  K2_OPT_PREFILL_GEMM = 13 /* tensor-core prefill of blocks over 16 tokens, QKV and gate/up GEMMs: 1 (default)
                             one persistent CTA per SM over whole 128 x 128 tiles, two TMEM accumulators so
                             that a tile's epilogue (store, SwiGLU) overlaps the next tile's K steps; 0 one
                             CTA per tile (the epilogue after its own K steps) */
} k2_option;
k2_status k2_set_option(k2_ctx* ctx, int32_t option, int64_t value);

/* Kernel classes timed by k2_profile_decode. */
enum {
  K2_K_EMBED = 0, K2_K_QKV, K2_K_ATTN, K2_K_OPROJ, K2_K_GATEUP, K2_K_DOWN, K2_K_LMHEAD, K2_K_STEP, K2_K_SAMPLE,
  K2_K_COUNT
};
/* K2_K_STEP: a whole token run by the persistent kernel; K2_K_SAMPLE: the sampler */

/* One decode step (as k2_decode_step) launched without graph or PDL, with a
 * CUDA event pair around every kernel; all launches are queued first, then the
 * call waits for the last event and adds the device milliseconds of each
 * kernel class to ms[K2_K_COUNT] and the number of launches to
 * launches[K2_K_COUNT]. */
k2_status k2_profile_decode(k2_ctx* ctx, const int32_t* d_tokens, int32_t batch, int32_t* d_next, float* ms,
                            int32_t* launches, void* stream);

/* The fp8 quantization of K2_F8 weights, on its own: each of `rows` bf16 rows
 * of `cols` values at d_src (device, row-major) becomes d_scales[r] = max|w| /
 * 448 (448: the largest finite E4M3 value) and d_codes[r * cols + c] =
 * E4M3(w / scale), rounded to nearest with ties to even and saturating; a row
 * of zeros gets scale 0 and codes 0.  The model computes with E4M3(code) *
 * scale. */
k2_status k2_quantize_fp8(const void* d_src, int32_t rows, int32_t cols, uint8_t* d_codes, float* d_scales,
                          void* stream);

/* The int4 block quantization of K2_Q4 weights, on its own (k2-burn README,
 * "Quantization": int4 with block size 64; symmetric codes).  Each of `rows`
 * bf16 rows of `cols` values at d_src (device, row-major) is cut into blocks
 * of 64 consecutive values (the last block of a row may be shorter); block b
 * of row r gets d_scales[r * ceil(cols / 64) + b] = max|w| / 7 and each value
 * the code d_codes[r * cols + c] = w / scale rounded to the nearest integer,
 * ties to even, clamped to [-7, 7]; a block of zeros gets scale 0 and codes 0.
 * The model computes with code * scale.  All buffers are the caller's device
 * memory; K2_ERR_ARG for null pointers, rows < 0 or cols < 1. */
k2_status k2_quantize_q4(const void* d_src, int32_t rows, int32_t cols, int8_t* d_codes, float* d_scales,
                         void* stream);

/* ---- without a workspace ---------------------------------------------------- */

/* The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory -- code inside a host runtime that owns every
 * device buffer and offers no allocator (a plugin in a pre-planned memory
 * arena), or code that must not call cudaMalloc because it may synchronise
 * the device.
 *
 * It computes what the end of k2_decode_step computes for one hidden state:
 * logits = lm_head . GroupedRMSNorm(d_x; final_norm) and the first index of
 * their maximum, using cfg->hidden, vocab, norm_groups, eps and weight_dtype
 * (other config fields are ignored).  d_x [hidden] fp32, lm_head
 * [vocab, hidden] and final_norm [hidden] (weight_dtype, 16-byte aligned) are
 * device inputs; d_logits [vocab] (nullable) and d_token [1] are device
 * outputs.  No context is needed and nothing is allocated: the kernel's
 * scratch (one partial maximum per CTA) is a static device array of
 * K2_NOALLOC_MAX_CTAS entries that every device loading the library holds
 * until exit; K2_ERR_WORKSPACE if the launch would need more CTAs than that.
 * The first call on a device looks up that array's address and sets kernel
 * attributes; make it before any stream capture.  That look-up is kept for
 * the life of the process: do not call this across a cudaDeviceReset of the
 * device.  All calls share the array and each clears its counter and guard
 * bits before launching, so calls that overlap on the GPU race: serialise
 * them (one stream, one thread).
 *
 * Failure on the device: with no context there is no k2_sync_status to read,
 * so the token itself carries it.  If any logit is NaN, or a bounded wait in
 * the kernel ran out, *d_token is written as -1 (d_logits, when given, still
 * holds the logits computed); otherwise it is the first index of the largest
 * logit.  The return value covers only what the host can check (K2_OK,
 * K2_ERR_ARG, K2_ERR_SHAPE, K2_ERR_UNSUPPORTED, K2_ERR_WORKSPACE,
 * K2_ERR_CUDA). */
#define K2_NOALLOC_MAX_CTAS 1024
k2_status k2_greedy_head_noalloc(const k2_config* cfg, const void* lm_head, const void* final_norm, const float* d_x,
                                 float* d_logits, int32_t* d_token, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* K2_H */
