/*
 * tfl.h - C ABI of a GB300 (sm_103a) bf16 forward for dense Llama-family GQA
 * decoders of the Nanbeige4.3-33B shape (hidden 7168, 52 layers, 56 query and
 * 8 KV heads of 128, FFN 22016, vocabulary 166,912, NeoX RoPE theta 1.2e8).
 *
 * What is computed (source: pull request #1415 "llama: Nanbeige4.3-33B on
 * Metal, the bf16 release served as published", section "How"): HF
 * modeling_llama in bf16, rounding to bf16 exactly at its rounding points:
 *   residual      h = bf16(h + bf16(f(h)))
 *   RMSNorm       bf16(w * bf16(x * rsqrt(mean(x^2) + eps)))
 *   projections   fp32 sums rounded once to bf16 (weights read in place)
 *   RoPE          bf16(bf16(x c) + bf16(rotate_half(x) s)), c/s = bf16 cos/sin
 *                 of the fp32 angle pos * inv_freq, NeoX half-head pairs
 *   attention     causal GQA (q head h reads KV head h / (n_q / n_kv)) over
 *                 keys at absolute positions 0..pos, scale 1/sqrt(head_dim);
 *                 scores, softmax and P.V in fp32, output rounded once
 *   SwiGLU        bf16(bf16(silu(g)) * u)
 *   head          final RMSNorm, lm_head (untied), greedy argmax with ties to
 *                 the lower id (same pull request, teacher-forced misses reply)
 *
 * Memory ownership.  The caller owns every device buffer (weights, workspace,
 * KV buffers, ids, logits) and keeps it alive while the library uses it; the
 * library borrows device pointers and owns only small host metadata.  All
 * tensors are bf16 unless stated, row-major, weights in HF [out][in] layout.
 *
 * Streams.  Every call that takes `stream` (a cudaStream_t, NULL = legacy
 * default stream) only enqueues work on it and returns without synchronising,
 * except tfl_status.  Host-side bookkeeping (KV lengths) advances at enqueue
 * time.  A model or KV object must not be used from two host threads at once.
 *
 * Errors.  Every function returns TFL_OK (0) or a negative TFL_E_* code and
 * throws nothing.  Arguments are validated on the host before anything is
 * enqueued; on an error nothing is enqueued and no state changes.
 * tfl_last_error() gives a message for the calling thread's last error.
 */
#ifndef TFL_H
#define TFL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TFL_OK 0
#define TFL_E_GEOMETRY (-1)  /* not a qualified geometry (message names it) */
#define TFL_E_ARCH (-2)      /* the current device is not an sm_103 GPU */
#define TFL_E_CAPACITY (-3)  /* a position would reach the KV capacity */
#define TFL_E_ARG (-4)       /* bad pointer, size, count or alignment */
#define TFL_E_CUDA (-5)      /* a CUDA runtime call failed */
#define TFL_E_NONFINITE (-6) /* an argmax saw a NaN or +-Inf logit */
#define TFL_E_WORKSPACE (-7) /* workspace or KV buffer too small */
#define TFL_E_DEVICE (-8)    /* a kernel reported an internal error (bounded wait) */

typedef struct tfl_model tfl_model;
typedef struct tfl_kv tfl_kv;

typedef struct {
    int hidden;        /* H */
    int layers;        /* L */
    int n_q;           /* query heads */
    int n_kv;          /* key/value heads */
    int head_dim;      /* D, must be 128 */
    int ffn;           /* F */
    int vocab;         /* V */
    double rope_theta; /* unscaled NeoX RoPE base */
    float rms_eps;     /* RMSNorm epsilon */
    int max_rows;      /* rows of one tfl_prefill_chunk, 1..2048 */
    int max_decode_rows; /* total rows of one tfl_decode_step over all streams, 1..64 */
    int max_context;   /* largest max_positions of any KV buffer used with the model */
} tfl_config;

/*
 * Device pointers to the weights, bf16, HF layout.  Per-layer fields point to
 * host arrays of `layers` device pointers (the arrays are copied at tfl_init).
 * Every pointer must be 16-byte aligned.
 *   embed [V][H], final_norm [H], lm_head [V][H] (untied: may not equal embed),
 *   attn_norm [H], wq [n_q*D][H], wk [n_kv*D][H], wv [n_kv*D][H], wo [H][n_q*D],
 *   ffn_norm [H], wg [F][H], wu [F][H], wd [H][F].
 */
typedef struct {
    const void *embed, *final_norm, *lm_head;
    const void *const *attn_norm, *const *wq, *const *wk, *const *wv, *const *wo;
    const void *const *ffn_norm, *const *wg, *const *wu, *const *wd;
} tfl_weights;

/* ---- setup ---------------------------------------------------------------- */

/*
 * Host-only geometry check (no GPU needed).  Qualified geometries: the 33B
 * shape above with 1..52 layers (a truncated stack of the same model), and the
 * tiny test model (hidden 1024, 8 q / 1 KV head of 128, FFN 2816, vocab 4096,
 * 1..2 layers).  Also refuses head_dim != 128, non-positive sizes, and
 * max_rows / max_decode_rows / max_context outside their ranges.  This mirrors
 * the qualification gate of pull request #1415 (reply "Admission"): other
 * geometries are refused by name.  On refusal, writes a message into msg
 * (if msg_len > 0) and returns TFL_E_GEOMETRY or TFL_E_ARG.
 */
int tfl_qualify(const tfl_config* cfg, char* msg, size_t msg_len);

/*
 * The bf16 RoPE table tfl_init uploads, computed on the host (no GPU needed):
 * for position p < n_pos and pair i < 64 (head_dim 128),
 *   inv_freq[i] = fl32(1 / fl32(theta^(2i/128))),  a = fl32(p * inv_freq[i]),
 *   cos_out[p*64 + i] = bf16(cos(a)),  sin_out[p*64 + i] = bf16(sin(a))
 * with cos/sin evaluated in double and rounded once to bf16 (nearest, ties to
 * even).  "bf16 cos and sin of the fp32 angle": pull request #1415, "How".
 * Outputs are bf16 bit patterns in host arrays of n_pos*64 entries.
 */
void tfl_rope_table(double theta, int n_pos, uint16_t* cos_out, uint16_t* sin_out);

/* Bytes of device workspace tfl_init needs for cfg (0 if cfg is not qualified). */
size_t tfl_workspace_bytes(const tfl_config* cfg);

/*
 * Creates a model.  Checks cfg (tfl_qualify), that the current device is
 * sm_103 (TFL_E_ARCH otherwise, named in the message), pointer alignment and
 * ws_bytes >= tfl_workspace_bytes(cfg).  Builds the bf16 RoPE cos/sin table
 * for max_context positions on the host and uploads it into the workspace
 * (synchronously, on the legacy default stream).  The workspace (16-byte
 * aligned device memory) is owned by the caller and used exclusively by this
 * model until tfl_free.  The refusal of other devices by name follows the
 * pull request's refusal of GPUs without the tensor units its prompt path
 * needs, checked at load before anything is mapped (pull request #1415,
 * section "Checks", and the reply "No tensor units").
 */
int tfl_init(const tfl_config* cfg, const tfl_weights* weights, void* workspace, size_t ws_bytes,
             tfl_model** out);
void tfl_free(tfl_model* model);

/* Thread-local message for the last error returned to this thread ("" if none). */
const char* tfl_last_error(void);
const char* tfl_error_string(int code);

/* ---- KV cache ---------------------------------------------------------------- */

/*
 * Position-major paged bf16 cache.  A buffer of tfl_kv_bytes(cfg, P) bytes holds
 * a page table (int32 per page, logical page -> physical page, identity after
 * tfl_kv_alloc) followed by pages of TFL_KV_PAGE positions; within a page the
 * layout is [position][kv head][D] for keys and, separately, for values:
 *   K(layer, pos) at pages + (((layer*2 + 0)*n_pages + table[pos/PAGE])*PAGE + pos%PAGE)*n_kv*D
 *   V(layer, pos) at pages + (((layer*2 + 1)*n_pages + table[pos/PAGE])*PAGE + pos%PAGE)*n_kv*D
 * i.e. layers * 2 * n_kv * D * 2 bytes per position (212,992 B for the 33B
 * shape: the 208 KiB/token of the EXL3 model card's "Which rung" section).
 * Keys are stored after RoPE.
 */
#define TFL_KV_PAGE 128
size_t tfl_kv_bytes(const tfl_config* cfg, int max_positions);

/*
 * Creates a KV object over dev_buf (16-byte aligned, >= tfl_kv_bytes bytes,
 * owned by the caller).  1 <= max_positions <= cfg.max_context.  Writes the
 * identity page table (synchronously).  The length starts at 0.  The cache is
 * the position-major bf16 key/value cache of pull request #1415 ("How": prompt
 * attention "over a position-major cache"; "bf16 keys and values"), sized by
 * the caller as the served setup sizes it by --context.
 */
int tfl_kv_alloc(tfl_model* model, int max_positions, void* dev_buf, size_t bytes, tfl_kv** out);
void tfl_kv_free(tfl_kv* kv);

/*
 * Sets the length (number of valid positions) to keep, 0 <= keep <=
 * max_positions.  keep < length truncates to a kept prefix (resume: the next
 * call continues at position keep; "a turn resumed from a kept prompt state
 * equals the same request after a restart", pull request #1415, "Measured").  keep > length declares positions
 * [length, keep) valid; their contents must have been written by earlier calls
 * or by tfl_kv_write.  Host-only; enqueues nothing.
 */
int tfl_kv_reset(tfl_kv* kv, int keep);
int tfl_kv_length(const tfl_kv* kv);
int tfl_kv_capacity(const tfl_kv* kv);

/*
 * Copies n positions [pos0, pos0+n) of one layer between the cache and dense
 * device tensors k, v of shape [n][n_kv][D] (keys after RoPE).  write: dense ->
 * cache; read: cache -> dense.  Does not change the length.  Bounds: 0 <= layer
 * < layers, 0 <= pos0, pos0 + n <= max_positions.
 */
int tfl_kv_write(tfl_model* model, tfl_kv* kv, int layer, int pos0, int n, const void* k, const void* v,
                 void* stream);
int tfl_kv_read(tfl_model* model, const tfl_kv* kv, int layer, int pos0, int n, void* k, void* v,
                void* stream);

/* ---- prompt cache ------------------------------------------------------------ */

/*
 * Copies the keys and values of positions [0, n) of every layer from src to
 * dst (both of this model; n <= length(src), n <= capacity(dst)) and sets
 * length(dst) = n.  Prefilling the rest of a prompt into dst then gives the
 * same bits as prefilling the whole prompt fresh (a prompt resumed from a kept
 * prefix, pull request #1415: "resumed prompts equal to fresh ones").  One
 * 2-D device copy of the whole pages involved, enqueued on stream; src and dst
 * must not be written by other work meanwhile.
 */
int tfl_kv_copy_prefix(tfl_model* model, const tfl_kv* src, tfl_kv* dst, int n, void* stream);

/*
 * A host-side index of caches that hold prompt prefixes (the prompt cache of
 * the pages' served setup).  The caller owns the caches; the store keeps a copy
 * of each entry's tokens and a pointer to its cache, and never touches the
 * cache itself.  put registers `kv` under tokens[0, n) (host int32, n >= 1; the
 * caller keeps length(kv) >= n while the entry exists); TFL_E_CAPACITY when the
 * store holds max_entries entries.  match returns the entry with the longest
 * common token prefix with tokens[0, n) and that length (ties: the entry put
 * last; none: *kv = NULL, *matched = 0).  remove drops the entries of kv.
 * No counterpart API on the pages (they describe the behaviour, not an API).
 */
typedef struct tfl_prefix_store tfl_prefix_store;
int tfl_prefix_store_new(int max_entries, tfl_prefix_store** out);
void tfl_prefix_store_free(tfl_prefix_store* store);
int tfl_prefix_store_put(tfl_prefix_store* store, const int32_t* tokens, int n, tfl_kv* kv);
int tfl_prefix_store_match(tfl_prefix_store* store, const int32_t* tokens, int n, tfl_kv** kv, int* matched);
int tfl_prefix_store_remove(tfl_prefix_store* store, const tfl_kv* kv);
int tfl_prefix_store_size(const tfl_prefix_store* store);

/* ---- forward ------------------------------------------------------------------ */

/*
 * One decode step over n_streams streams (1..16) sharing the weight pass:
 * the decode rows of pull request #1415, section "How" (row projections with
 * fp32 sums rounded once, attention of each row over key blocks at absolute
 * positions; the lane host's shared rounds of several streams).
 * Stream s contributes rows_per_stream[s] (host array, 1..16) consecutive rows
 * of ids (device int32 [sum rows], stream-major), at positions length(s) ..
 * length(s) + rows - 1; a multi-row group is a causal window (each row sees
 * the earlier rows of the same stream).  Writes logits (device bf16 [sum
 * rows][V]) and appends the rows' keys and values; length(s) += rows.
 * The same kvs object may not appear twice.  TFL_E_CAPACITY if a stream would
 * pass its max_positions (nothing is enqueued then).  Results for each row are
 * bit-identical whatever the other rows and streams of the call are
 * (one-row steps == windows, solo == batched).
 */
int tfl_decode_step(tfl_model* model, tfl_kv* const* kvs, int n_streams, const int32_t* ids,
                    const int* rows_per_stream, void* logits, void* stream);

/*
 * A decode step of one or two rows in total runs, by default, as one
 * persistent cooperative launch (all layers and the head; one CTA per SM, grid
 * barriers between the operations) with the same arithmetic as the launch per
 * operation used for larger steps, so results are bit-identical either way.
 * enable = 0 makes every step use the launch per operation (for comparisons);
 * enable != 0 restores the default.  No counterpart on the pages (an execution
 * detail of this library).
 */
int tfl_set_persistent(tfl_model* model, int enable);

/*
 * Prompt chunk of n_rows (1..max_rows) ids (device int32) for one stream, at
 * positions length .. length + n_rows - 1 (causal over the cache and the
 * chunk): the prompt chunks of up to 2,048 rows of pull request #1415, section
 * "How" (projections as dense GEMMs, attention over the position-major cache).  logits: NULL for none; else device bf16 [1][V] for the last row
 * (all_rows == 0) or [n_rows][V] (all_rows != 0).  length += n_rows.
 * The row results do not depend on where chunk boundaries fall (a prompt
 * resumed from a kept prefix equals the same prompt prefilled fresh).
 */
int tfl_prefill_chunk(tfl_model* model, tfl_kv* kv, const int32_t* ids, int n_rows, void* logits,
                      int all_rows, void* stream);

/*
 * Greedy ids (device int32 [n_rows]) from logits (device bf16 [n_rows][V]),
 * ties to the lowest id.  A row holding NaN or +-Inf gets id -1 and raises the
 * model's device status word, read by tfl_status.
 */
int tfl_argmax(tfl_model* model, const void* logits, int n_rows, int32_t* ids, void* stream);

/*
 * Sampled ids (device int32 [n_rows], n_rows 1..max_decode_rows) from logits
 * (device bf16 [n_rows][V]) with temperature T > 0, top_k (0 = no cut) and
 * top_p (>= 1 = no cut); u: device float [n_rows], the caller's uniform draws in
 * [0, 1) (its seeded random numbers).  Per row: candidates = ids whose logit is
 * at least the top_k-th largest (ties included); weights exp((z - z_max)/T) in
 * double; nucleus = candidates at or above the first value (largest down) at
 * which the running mass of the values reaches top_p of the candidates' mass;
 * result = the smallest nucleus id whose running weight in id order exceeds
 * u x (nucleus mass).  The pages name a seeded GPU draw with temperature and
 * top-p beside argmax but fix no algorithm; this is the reading taken.  A row
 * holding NaN or +-Inf gets -1 and raises the device status word (tfl_status:
 * TFL_E_NONFINITE).  Deterministic.  Uses the model's workspace (serialise
 * calls on one model).
 */
int tfl_sample(tfl_model* model, const void* logits, int n_rows, float temperature, int top_k, float top_p,
               const float* u, int32_t* ids, void* stream);

/* ---- drafted greedy decode ---------------------------------------------- */

/*
 * Drafted greedy decode (the pages: a smaller Llama on the same tokenizer
 * drafting for the served model, "--drafter", with drafted greedy replies equal
 * to plain greedy ones; issue #1414, reply "Drafting", and pull request #1415,
 * section "How", whose lane host also makes "copy drafts").  Each round a
 * proposer guesses up to draft_len next tokens, the served model runs the
 * pending token and the guesses as one causal window, and the guesses that
 * equal the window's own greedy ids, up to the first that does not, are kept
 * together with the window's greedy id after them.  Because a window row is
 * bit-identical to a one-row step (tfl_decode_step), the ids produced are
 * exactly those of plain greedy decoding, whatever the proposer guesses.
 *
 * context: host int32 [n_context] (n_context >= 1), the tokens so far; the
 * last one is pending (not yet run): length(kv) must be n_context - 1.
 * Writes n_tokens >= 1 greedy ids to out_ids (host int32 [n_tokens]): out_ids[0]
 * is the served model's greedy id after the pending token, and so on, as n_tokens
 * plain one-row steps each fed the previous id would give.  On return
 * length(kv) = n_context - 1 + n_tokens (out_ids[n_tokens - 1] is pending).
 * kv's capacity must hold that length.
 *
 * Proposer: drafter != NULL: a model of the same vocabulary with its own cache
 * dkv, holding the first length(dkv) tokens of context, n_context - length(dkv)
 * in 1..min(16, drafter max_decode_rows); its greedy one-row steps propose the
 * guesses (a non-finite drafter row proposes id 0).  drafter == NULL (dkv
 * ignored): copy drafts, tfl_copy_draft over the tokens so far.  On return
 * dkv holds a prefix of the tokens (its contents only affect speed).
 *
 * draft_len: 1 .. min(16, target max_decode_rows) - 1.  workspace: device,
 * tfl_drafted_workspace_bytes(target, draft_len) bytes, 256-byte aligned,
 * caller-owned.  stats (NULL = none): rounds, guesses made, guesses kept, rows
 * run by the served model and by the drafter.
 *
 * Synchronous: each round reads the window's ids back to the host (one stream
 * synchronisation per round).  Errors: TFL_E_ARG / TFL_E_CAPACITY / TFL_E_WORKSPACE
 * before anything runs; TFL_E_NONFINITE when a served-model id is -1 (a NaN or
 * +-Inf logit): out_ids holds the ids up to and including that -1, the rest
 * are -1, and the caches hold the tokens before it.
 */
typedef struct {
    long long rounds;        /* windows run by the served model */
    long long drafted;       /* guesses proposed */
    long long accepted;      /* guesses kept */
    long long target_rows;   /* rows run by the served model */
    long long drafter_rows;  /* rows run by the drafter */
} tfl_draft_stats;

size_t tfl_drafted_workspace_bytes(const tfl_model* target, int draft_len);
int tfl_decode_drafted(tfl_model* target, tfl_kv* kv, tfl_model* drafter, tfl_kv* dkv, int draft_len,
                       const int32_t* context, int n_context, int n_tokens, int32_t* out_ids, void* workspace,
                       size_t ws_bytes, tfl_draft_stats* stats, void* stream);

/*
 * Copy drafts (host only): the longest suffix of tokens[0, n) of 1..3 tokens
 * that also occurs earlier, at its latest earlier occurrence, proposes the
 * tokens that followed that occurrence, continued periodically past the end
 * (a sequence that repeats with period P proposes its next tokens as the
 * repeat).  Writes up to max_draft ids to out and returns how many (0 when no
 * suffix recurs), or TFL_E_ARG.  The pages name copy drafts without a rule;
 * this is the reading taken.
 */
int tfl_copy_draft(const int32_t* tokens, int n, int max_draft, int32_t* out);

/*
 * Synchronises `stream`, reads and clears the device status word: returns
 * TFL_OK, TFL_E_NONFINITE (an argmax saw a non-finite logit) or TFL_E_DEVICE
 * (a kernel gave up a bounded wait), or TFL_E_CUDA if the stream had failed.
 * A non-finite row is refused rather than given an id, as the pages' checker
 * refuses a row holding NaN or +-Inf before choosing a token (pull request
 * #1415, the reply on non-finite rows of the teacher-forced checker).
 */
int tfl_status(tfl_model* model, void* stream);

/*
 * Test aid for the failure path of the device waits: runs one of the bounded
 * waits of the persistent decode step alone, on an event that never happens,
 * with a poll limit of spin_limit (1..2^20; the kernels' own limit is 2^24,
 * about a second):  which = 0: the grid-barrier wait (thread 0 of one CTA per
 * SM on a counter target no CTA reaches; the first to give up raises the abort
 * flag that ends the others' waits); which = 1: an mbarrier wait on a phase
 * that receives no arrival (no copy is in flight).  The wait gives up, sets the
 * device status word and the kernel returns, so the next tfl_status returns
 * TFL_E_DEVICE and the model stays usable (the grid-barrier words are reset at
 * every persistent step).  Enqueues on stream.  TFL_E_ARG for other values.
 * No counterpart on the pages, whose refusals are host-side ("rejected the
 * next token" past the cache, NInfer model card, "Validation"); this checks
 * that a device-side give-up is likewise an error status and not a hang.
 */
int tfl_wait_probe(tfl_model* model, int which, int spin_limit, void* stream);

/* ---- component entry points (the same kernels, for per-layer checks) ------- */

/*
 * The decoder layers only: like tfl_decode_step / tfl_prefill_chunk but the
 * rows are given as residual-stream rows h_in (device bf16 [rows][H], the
 * embedding output) and the result is the residual stream after the last
 * layer, h_out (device bf16 [rows][H]), before the final norm.  decode: the
 * decode kernels (n_streams, rows_per_stream as tfl_decode_step); prefill: the
 * prompt-chunk kernels for one stream.  KV lengths advance as in the full calls.
 */
int tfl_decode_hidden(tfl_model* model, tfl_kv* const* kvs, int n_streams, const int* rows_per_stream,
                      const void* h_in, void* h_out, void* stream);
int tfl_prefill_hidden(tfl_model* model, tfl_kv* kv, const void* h_in, int n_rows, void* h_out, void* stream);

/* Final RMSNorm + lm_head over rows of h (device bf16 [rows][H]) -> logits [rows][V]. */
int tfl_head(tfl_model* model, const void* h, int rows, void* logits, void* stream);

/*
 * One operation of the decode path, run by the same kernel a decode step uses,
 * on caller-given device inputs (so each kernel can be checked alone against
 * a reference fed the same bf16 inputs).  rows: 1..max_decode_rows, all of one
 * stream at positions pos0 .. pos0+rows-1 (kv and pos0 are used by QKV_ROPE
 * and ATTENTION only; other ops take kv = NULL).  Does not change KV lengths.
 *   TFL_OP_ATTN_NORM     in h [rows][H]           -> out bf16 RMSNorm with attn_norm[layer]
 *   TFL_OP_QKV_ROPE      in xn [rows][H]          -> out rotated q [rows][n_q*D]; rotated k and
 *                        v of the rows written into kv (layer) at their positions
 *   TFL_OP_ATTENTION     in rotated q [rows][n_q*D] -> out [rows][n_q*D]; row i attends
 *                        keys 0..pos0+i of kv (layer), which must already hold them
 *   TFL_OP_O_RESIDUAL    in attention out [rows][n_q*D]; out h [rows][H] updated in place:
 *                        h = bf16(h + bf16(Wo[layer] . in))
 *   TFL_OP_FFN_NORM      in h -> out RMSNorm with ffn_norm[layer]
 *   TFL_OP_GATE_UP       in xn [rows][H] -> out bf16(bf16(silu(Wg.xn)) * Wu.xn) [rows][F]
 *   TFL_OP_DOWN_RESIDUAL in act [rows][F]; out h updated: h = bf16(h + bf16(Wd[layer] . in))
 *   TFL_OP_FINAL_NORM    in h -> out RMSNorm with final_norm (layer ignored)
 *   TFL_OP_LM_HEAD       in xn [rows][H] -> out logits [rows][V] (layer ignored)
 *   TFL_OP_NORM_QKV_ROPE, TFL_OP_NORM_GATE_UP, TFL_OP_NORM_LM_HEAD: the norm and
 *                        the projection after it in one op, as a decode step
 *                        runs them: in is the residual stream h; the result is
 *                        bit-identical to the norm op followed by the projection op
 * Buffers are 16-byte aligned; in and out must not overlap.
 * op | TFL_OP_PROMPT runs the op with the prompt-chunk kernels instead (rows
 * 1..max_rows): the projections on the tensor-core GEMM, the norms always as a
 * separate kernel, attention by the one-pass causal prompt kernel.  Not for
 * TFL_OP_LM_HEAD / TFL_OP_NORM_LM_HEAD (a prompt chunk's logits come from the
 * decode head): TFL_E_ARG.
 */
#define TFL_OP_ATTN_NORM 0
#define TFL_OP_QKV_ROPE 1
#define TFL_OP_ATTENTION 2
#define TFL_OP_O_RESIDUAL 3
#define TFL_OP_FFN_NORM 4
#define TFL_OP_GATE_UP 5
#define TFL_OP_DOWN_RESIDUAL 6
#define TFL_OP_FINAL_NORM 7
#define TFL_OP_LM_HEAD 8
#define TFL_OP_NORM_QKV_ROPE 9
#define TFL_OP_NORM_GATE_UP 10
#define TFL_OP_NORM_LM_HEAD 11
#define TFL_OP_PROMPT 0x100
int tfl_layer_op(tfl_model* model, int op, int layer, tfl_kv* kv, int pos0, int rows, const void* in, void* out,
                 void* stream);

/*
 * Decode attention that allocates nothing and needs no workspace.  The pages
 * have no counterpart: this is a convenience for callers that cannot allocate
 * device memory where they run attention (a serving runtime whose memory
 * manager owns all of the GPU's memory, or code that must not call cudaMalloc
 * because it can synchronise the device or break a stream capture).
 * Same computation and kernels as TFL_OP_ATTENTION of tfl_layer_op: rows
 * (1..64) of rotated queries q (device bf16 [rows][n_q*D]) at positions pos0 ..
 * pos0+rows-1 attend keys 0..pos0+i of kv (layer); out is device bf16
 * [rows][n_q*D].  The softmax partials live in a fixed 16 MiB array inside the
 * library (held on every GPU that loads it until the process exits):
 * rows * n_q * ceil((pos0+rows)/512) must not exceed 32,263 (for the 33B shape:
 * one row up to 294,912 positions, 16 rows up to 18,432), else TFL_E_WORKSPACE
 * with a message.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the array: calls that overlap on
 * the GPU race, so serialise them (one stream, or events).  It needs no
 * clearing between calls.  Calls no cudaMalloc, cudaFree or allocating library
 * routine.
 */
int tfl_attention_decode_noalloc(tfl_kv* kv, int layer, int pos0, int rows, const void* q, void* out,
                                 void* stream);

/* ---- per-kernel timing ------------------------------------------------------------- */

/*
 * While enabled, every kernel launch of the model is bracketed by two CUDA
 * events recorded on the launch stream (this also serialises kernels that
 * would otherwise overlap through programmatic dependent launch, so profiled
 * steps run slightly slower than unprofiled ones).  Off after tfl_init.
 */
int tfl_profile(tfl_model* model, int enable);

/*
 * Synchronises the device and returns, per kernel family k < n_kinds, the
 * summed elapsed milliseconds ms[k] and the number of launches[k] recorded
 * since the last read (host arrays of n_kinds entries); then forgets them.
 * Family names: tfl_profile_kind(k) (NULL past the last family).
 */
int tfl_profile_read(tfl_model* model, int n_kinds, double* ms, long* launches);
const char* tfl_profile_kind(int kind);

/*
 * Phase times of the last persistent decode step run while profiling was on:
 * out[0..5] the mean per layer (microseconds, from the last CTA leaving the
 * previous grid barrier to the last CTA leaving this one) of the RMSNorm+QKV,
 * attention, merge, o projection, RMSNorm+gate/up and down phases; out[6] the
 * mean barrier latency (last arrival to first departure); out[7] the final
 * norm + lm_head phase; out[8] the whole kernel.  n >= 9.  Synchronises the
 * device.  TFL_E_ARG when no such step ran since the last call.  No
 * counterpart on the pages (a measurement aid).
 */
int tfl_step_phases(tfl_model* model, double* out, int n);

#ifdef __cplusplus
}
#endif
#endif /* TFL_H */
