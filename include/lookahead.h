/*
 * lookahead.h -- C ABI of liblookahead.so: one combined Lookahead Decoding
 * step on one GB300 (sm_103a).
 *
 * Method: Fu, Bailis, Stoica, Zhang 2024, "Break the Sequential Dependency of
 * LLM Inference Using Lookahead Decoding" (summary page, "Summary" and "Key
 * points").  Each decode step runs ONE forward pass of a Llama-style decoder
 * over 1 + W(N-1) lookahead-branch rows plus G(N-1) verification-branch rows
 * under a combined attention mask against the KV cache, then greedily
 * verifies the candidate n-grams, harvests new n-grams from the 2D window into
 * the n-gram pool, and commits the accepted tokens' keys/values.  The output
 * equals plain greedy decoding token for token.
 *
 * Conventions (all entry points):
 *  - Return LA_OK (0) or a negative LA_ERR_* code; no exception crosses the
 *    ABI.  la_last_error() gives a message for the last failure on a context.
 *  - A context is single-threaded; all device work is issued on desc.stream
 *    (NULL = the legacy default stream).
 *  - "host" pointers are caller-owned host memory; "device" pointers are
 *    caller-owned device memory that must stay valid until la_destroy.
 *  - Matrices are row-major [out][in] (PyTorch nn.Linear layout).
 *  - Compiled limits: rows per step T = 1 + (W+G)(N-1) <= 128 (batched:
 *    batch x T <= 128), N <= 8, head_dim in {64, 128},
 *    n_heads % n_kv_heads == 0, d_model % 64 == 0.
 */
#ifndef LOOKAHEAD_H
#define LOOKAHEAD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LA_API __attribute__((visibility("default")))
#else
#define LA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define LA_OK 0
#define LA_ERR_ARG (-1)         /* invalid argument or unsupported shape        */
#define LA_ERR_OOM (-2)         /* device or pinned-host allocation failed      */
#define LA_ERR_CAPACITY (-3)    /* KV cache (max_seq) or pool capacity exceeded */
#define LA_ERR_CUDA (-4)        /* a CUDA runtime call failed                   */
#define LA_ERR_TIMEOUT (-5)     /* a bounded device-side wait gave up           */
#define LA_ERR_STATE (-6)       /* call out of order (e.g. step before prefill) */

#define LA_FP32 0 /* fp32 weights/activations: SIMT debug path               */
#define LA_BF16 1 /* bf16 weights/activations: tcgen05 GEMMs, MMA attention  */

#define LA_PRESEED_PROMPT 1 /* insert the prompt's n-grams into the pool at prefill */
#define LA_DEBUG_LOGITS 2   /* keep the last step's fp32 logits for la_debug_logits */
#define LA_NO_GRAPH 4       /* launch kernels directly instead of a CUDA graph      */
#define LA_SIMT 8           /* bf16 model on the SIMT kernels (debug)               */
#define LA_PROFILE 16       /* time kernel classes with CUDA events (la_get_profile) */
#define LA_ATTN_TC 32       /* bf16: the step's attention on tcgen05 + TMA (needs      \
                               W + N - 2 <= 31 and max_seq <= 4096; see la_create)   */
#define LA_MASK_DIAG 64     /* lookahead branch as diagonal levels (see la_create)     */

typedef struct la_ctx la_ctx;

/* Decoder description.  Weight pointers are DEVICE pointers of `dtype`
 * elements, borrowed until la_destroy (the bf16 tensor-core path also packs
 * a copy of the matrices at la_create, see there).
 *   emb        [vocab][d_model]
 *   layer_w    n_layers*9 pointers, per layer in this order:
 *              attn_norm [d_model], wq [H*hd][d_model], wk [Hkv*hd][d_model],
 *              wv [Hkv*hd][d_model], wo [d_model][H*hd], ffn_norm [d_model],
 *              wg [ffn][d_model], wu [ffn][d_model], wd [d_model][ffn]
 *              (the array itself is host memory, copied by la_create)
 *   final_norm [d_model]
 *   lm_head    [vocab][d_model]  (untied)
 * Model: h = x + Wo Attn(RMSNorm(x)); y = h + Wd(silu(Wg n) * Wu n),
 * n = RMSNorm(h); rotate-half RoPE with angle pos*rope_theta^(-2i/hd). */
typedef struct la_model_desc {
    int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab, max_seq;
    float rms_eps;    /* e.g. 1e-5  */
    float rope_theta; /* e.g. 1e4   */
    int dtype;        /* LA_FP32 or LA_BF16 */
    const void* emb;
    const void* const* layer_w;
    const void* final_norm;
    const void* lm_head;
    void* stream; /* cudaStream_t */
} la_model_desc;

typedef struct la_stats {
    long long steps;          /* la_step calls since the last prefill        */
    long long emitted;        /* tokens emitted since the last prefill       */
    long long prefill_tokens; /* prompt tokens written to the cache          */
    long long accept_hist[9]; /* steps by tokens emitted (1..N)              */
    int P;                    /* tokens whose KV is cached                   */
    int rows;                 /* rows per step: T (batched: batch x T)       */
    float last_step_ms;       /* device time of the last step (CUDA events)  */
    int kernels_per_step;     /* kernel launches in one captured step        */
} la_stats;

/* Per-kernel-class timing (LA_PROFILE): CUDA events recorded on the launching
 * stream around every launch of the class, summed over the steps so far.
 * bytes / flops are the ALGORITHMIC traffic and work of those launches
 * (weights once, the rows' activations in and out once; attention: the KV
 * cache once plus the rows' q, k, v and output). */
typedef struct la_prof_entry {
    char name[24];
    long long launches;
    double total_ms;
    double bytes;
    double flops;
} la_prof_entry;

/* Bytes of device workspace la_create needs for this model and (W,N,G):
 * KV cache, per-layer step K/V, activations, row tables, window and pool.
 * Returns 0 for unsupported arguments.
 * No counterpart on the pages: sizing of this library's device memory. */
LA_API size_t la_workspace_bytes(const la_model_desc* desc, int W, int N, int G);

/* Pages: summary page, "Key points" (the knobs: window size W, n-gram size N,
 * verification candidates G; G = W in the pages' settings).
 * Create a decoding context.  W >= 0 lookahead columns, N >= 2 n-gram size,
 * G >= 0 verification candidates per step; W = G = 0 is plain greedy.
 * workspace: DEVICE buffer of ws_bytes >= la_workspace_bytes(), borrowed; or
 * NULL, and the library allocates (and frees) its own.  seed initialises the
 * lookahead window (splitmix64 stream).  flags: LA_PRESEED_PROMPT |
 * LA_DEBUG_LOGITS | LA_NO_GRAPH | LA_SIMT | LA_PROFILE | LA_ATTN_TC |
 * LA_MASK_DIAG.  On success *out owns the context.
 * LA_MASK_DIAG reads the pages' 2D window the other way their text allows:
 * each of the N-1 levels is one Jacobi iterate over positions P+1..P+W and
 * its rows see only their own level (row (l,j) sees c and (l,0..j)); the new
 * last level is the Jacobi update of the last one (argmax of row 0, then of
 * row (N-2, j-1) at column j); the n-grams run along diagonals (key
 * win[0][j], value win[1][j+1], ..., win[N-2][j+N-2], argmax of row
 * (N-2, j+N-2)).  The row count and the verification branch are unchanged;
 * the default is the column reading (row (l,j) at P+1+j+l sees level 0 up to
 * column j and column j up to level l).  LA_ATTN_TC (bf16 tensor-core path) runs the
 * step's attention on a second kernel pair: each row's keys older than its
 * 31..46 most recent positions in splits of 128 positions on tcgen05 (TMA-fed,
 * accumulators in tensor memory), the recent window per row group on
 * mma.sync, merged per row; LA_ERR_ARG when W + N - 2 > 31 or max_seq > 4096.
 * Its arithmetic differs from the default kernel's, so a greedy context
 * compared token for token with a lookahead context must use the same flag.
 * On the bf16 tensor-core path la_create also makes, and the context owns, a
 * tile-packed copy of every projection, MLP and LM-head matrix (their size
 * again, in device memory outside the workspace); later changes to those
 * caller buffers are not seen.  LA_ERR_CUDA if that allocation fails.
 * Fault injection for tests of callers' error handling, from the host only:
 * the environment variable LA_FAULT, read here, = "alloc" (la_create returns
 * LA_ERR_OOM) | "badarg" (LA_ERR_ARG) | "timeout@K" (the K-th la_step after
 * a prefill returns LA_ERR_TIMEOUT: the host sets the device status word a
 * bounded device wait sets when it gives up) | "capacity@K" (the K-th
 * la_step returns LA_ERR_CAPACITY); each fires once per context. */
LA_API int la_create(const la_model_desc* desc, int W, int N, int G, void* workspace, size_t ws_bytes,
              uint64_t seed, int flags, la_ctx** out);

/* Pages: "Summary" (the lookahead branch's 2D window of W columns x N-1
 * levels, set up here) and "Key points" (prompt n-grams added to the pool:
 * LA_PRESEED_PROMPT).
 * Prefill: write the KV of prompt[0..len-2] into the cache, reset the window
 * and the pool (optionally seed it with the prompt's n-grams) and make
 * prompt[len-1] the current token.  prompt: HOST int32[len], len >= 1,
 * len + W + N <= max_seq.  Blocks until done. */
LA_API int la_prefill(la_ctx* ctx, const int32_t* prompt, int len);

/* Pages: "Summary" (one forward pass holds the lookahead branch over the 2D
 * window and the verification branch over pool candidates; new n-grams go to
 * the pool; the output stays exactly the greedy output).
 * One combined lookahead decode step.  Writes the 1..N emitted tokens to the
 * HOST buffer out (cap >= N entries) and their count to *n_out.  Blocks until
 * the tokens are on the host.  LA_ERR_CAPACITY if the cache cannot hold the
 * step (P + W + N > max_seq); LA_ERR_STATE before la_prefill.  After an error
 * raised on the device (LA_ERR_TIMEOUT, or a full pool: LA_ERR_CAPACITY) the
 * context returns LA_ERR_STATE until the next la_prefill. */
LA_API int la_step(la_ctx* ctx, int32_t* out, int cap, int* n_out);

/* Pages: "Summary" (the method supports sampling and keeps the output
 * distribution; the pages give no rule, so the rule below is this library's).
 * Sampling verification (temperature sampling, lossless in distribution;
 * the method's summary page says sampling is supported and the output
 * distribution kept, without giving the rule).  temperature > 0: every
 * emitted token is drawn from softmax(logits / temperature) of its row.  At
 * each candidate level the distinct candidate tokens v are tried in
 * candidate order, v accepted with probability p(v) / (1 - mass of the
 * values already rejected at that level).  If none is accepted, the token
 * is drawn from p without the rejected values.  After the last level a bonus
 * token is drawn.  The uniforms are the top 24 bits of a splitmix64 stream
 * seeded with `seed`, one per candidate try and one per drawn token.
 * temperature <= 0 restores greedy verification.  The lookahead branch
 * keeps using argmaxes either way.  Takes effect at the next la_step (the
 * step is captured again); la_prefill keeps the stream's position.  Costs
 * the logits of the step in device memory (already in the workspace) and a
 * row-statistics kernel per step.  LA_ERR_ARG for a NULL context or a
 * non-finite temperature; LA_ERR_CUDA if the stream state cannot be
 * written. */
LA_API int la_set_sampling(la_ctx* ctx, float temperature, uint64_t seed);

/* Pages: "Summary" (several sampling schemes are supported; the pages give
 * none of them, so this restriction is this library's).
 * Top-k for sampling verification: with top_k in 1..vocab-1, every row's
 * distribution (the temperature softmax of la_set_sampling, as integer
 * weights) is restricted to its top_k tokens by weight, equal weights lower
 * token index first, and renormalised; the verification rule is unchanged,
 * so each emitted token follows the restricted distribution of its row.
 * 0 (the default) or >= vocab keeps every token; no effect under greedy
 * verification.  Takes effect at the next step (the step is captured
 * again).  Costs a radix select over each sampled row's vocabulary per step.
 * LA_ERR_ARG for top_k < 0. */
LA_API int la_set_top_k(la_ctx* ctx, int top_k);

/* Pages: "Summary" (several sampling schemes are supported; the pages give
 * none of them, so this restriction is this library's).
 * Top-p (nucleus) for sampling verification: after the top-k restriction,
 * every row's distribution is restricted to the smallest leading set of its
 * tokens, in the top-k order (larger weight first, equal weights lower token
 * index first), whose weight A reaches A 2^24 >= floor(top_p 2^24) S (S the
 * weight left by top-k), and renormalised; the verification rule is
 * unchanged, so each emitted token follows the restricted distribution of
 * its row.  1 (the default) keeps every token; no effect under greedy
 * verification.  Takes effect at the next step (the step is captured
 * again).  Costs a weighted radix select over each sampled row's
 * vocabulary per step.  LA_ERR_ARG for a NULL context or top_p outside
 * (0, 1] (NaN included). */
LA_API int la_set_top_p(la_ctx* ctx, float top_p);

/* Pages: "Summary" (decoding that emits what plain greedy decoding emits,
 * several tokens per step).
 * la_prefill, then la_step until max_new tokens; out: HOST int32[max_new]
 * receives exactly min(max_new, emitted) tokens, count in *n_out. */
LA_API int la_generate(la_ctx* ctx, const int32_t* prompt, int len, int max_new, int32_t* out, int* n_out);

/* ---- batched decoding: several sequences in one forward pass per step ----
 * Pages: "Key points" (main limitation: the per-step FLOPs the lookahead and
 * verification rows add make the method gain less when the GPU serves large
 * batches, since the step is then no longer bandwidth bound).  A batched
 * context decodes B independent sequences with the same model and the same
 * (W, N, G): each step's forward pass holds every sequence's 1 + (W+G)(N-1)
 * rows (sequence b's are rows b*T .. b*T+T-1), so the weights stream once for
 * all of them; attention, verification, harvest, window and KV commit run per
 * sequence on its own cache, window and pool.  Every sequence's output is the
 * output of a batch-1 context with the same seed (bit for bit: no row's
 * arithmetic depends on the other rows).  B * (1 + (W+G)(N-1)) <= 128.
 * Not with LA_ATTN_TC (LA_ERR_ARG).  la_prefill, la_step and la_generate
 * return LA_ERR_STATE on a batched context. */

/* No counterpart on the pages: sizing of this library's device memory.
 * Workspace of a batched context (la_workspace_bytes is batch = 1): the KV
 * cache, window, pool and decode state once per sequence, the rest shared.
 * 0 for unsupported arguments. */
LA_API size_t la_workspace_bytes_batch(const la_model_desc* desc, int W, int N, int G, int batch);
/* Pages: "Key points" (main limitation, serving batches; the knobs W, N, G).
 * la_create for `batch` sequences (la_create is batch = 1); same arguments
 * and ownership.  LA_ERR_ARG when batch < 1, batch * T > 128 or LA_ATTN_TC
 * is asked for with batch > 1. */
LA_API int la_create_batch(const la_model_desc* desc, int W, int N, int G, int batch, void* workspace,
                           size_t ws_bytes, uint64_t seed, int flags, la_ctx** out);
/* Pages: "Summary" (the 2D window set up from the prompt), per sequence.
 * la_prefill of sequence seq (0 <= seq < batch) alone; its window is drawn
 * from `seed` as in la_prefill.  Every sequence must be prefilled before
 * la_step_batch; prefilling sequence 0 starts new la_get_stats counters. */
LA_API int la_prefill_seq(la_ctx* ctx, int seq, const int32_t* prompt, int len);
/* Pages: "Summary" (one forward pass holds both branches; output equal to
 * greedy decoding) and "Key points" (main limitation: batches).
 * One combined step of every sequence.  out: HOST int32[batch][cap]
 * (cap >= N): sequence b's 1..N tokens at out[b*cap ..], their count in
 * n_out[b] (HOST int32[batch]).  Errors as la_step, for any sequence (a
 * device error makes every sequence need its prefill again).  Sampling
 * verification (la_set_sampling) gives sequence b the stream seeded with
 * seed + b. */
LA_API int la_step_batch(la_ctx* ctx, int32_t* out, int cap, int* n_out);

/* Pages: "Summary" (output equal to greedy decoding) and "Key points" (main
 * limitation: batches).
 * Batched la_generate: prefill every sequence (prompts: HOST int32, the
 * sequences' prompts back to back, lens: HOST int32[batch], each >= 1), then
 * step the batch until every sequence has max_new tokens.  out: HOST
 * int32[batch][max_new]; n_out: HOST int32[batch], each min(max_new,
 * emitted).  A sequence that has its tokens keeps stepping with the others;
 * its further tokens are dropped.  Errors as la_prefill_seq and
 * la_step_batch (LA_ERR_CAPACITY when a sequence's cache fills first). */
LA_API int la_generate_batch(la_ctx* ctx, const int32_t* prompts, const int* lens, int max_new, int32_t* out,
                             int* n_out);

/* Pages: "Key points" (steps taken against tokens emitted: the step count
 * the scaling law is about).  Counters since the last la_prefill (batched:
 * since sequence 0's; emitted and accept_hist count every sequence, steps
 * count batched steps, P is sequence 0's, rows = batch * T). */
LA_API int la_get_stats(la_ctx* ctx, la_stats* out);
/* No counterpart on the pages: this library's kernel timing.
 * Copy up to cap entries (one per kernel class seen); *n_out = entries written.
 * LA_ERR_STATE unless the context was made with LA_PROFILE. */
LA_API int la_get_profile(la_ctx* ctx, la_prof_entry* out, int cap, int* n_out);

/* ---- debug accessors (host copies of device state, after a step) ---- */

/* No counterpart on the pages (a parity accessor).
 * Last step's logits, fp32 [T][vocab]; needs LA_DEBUG_LOGITS; n >= T*vocab. */
LA_API int la_debug_logits(la_ctx* ctx, float* host, size_t n);
/* Pages: "Summary" (greedy verification compares candidates with the model's
 * own choices).  Last step's per-row argmax, int32[T]; *T_out = T. */
LA_API int la_debug_argmax(la_ctx* ctx, int32_t* host, int cap, int* T_out);
/* Pages: "Summary" (the step's lookahead-branch and verification-branch rows).
 * Last step's row table: tokens and positions int32[T]; *ncand = candidates
 * found in the pool (rows of missing candidates are padding). */
LA_API int la_debug_rows(la_ctx* ctx, int32_t* tok, int32_t* pos, int cap, int* T_out, int* ncand);
/* Pages: "Summary" (n-grams cached in a pool).
 * Pool entries of key, oldest first: int32[count][N-1] into host (cap ints). */
LA_API int la_debug_pool(la_ctx* ctx, int32_t key, int32_t* host, int cap, int* count);
/* Pages: "Summary" (the 2D window of Jacobi iteration history).
 * Lookahead window, int32[N-1][W] into host (cap ints). */
LA_API int la_debug_window(la_ctx* ctx, int32_t* host, int cap);
/* No counterpart on the pages (a parity accessor of batched decoding).
 * Make the debug accessors above and below read sequence seq of a batched
 * context (0 at creation).  LA_ERR_ARG for seq outside 0..batch-1. */
LA_API int la_debug_select(la_ctx* ctx, int seq);
/* No counterpart on the pages (a parity accessor for the controller).
 * Replace the model's argmaxes seen by verification, harvest and window
 * update with host[0..n) (one token per step row, n = T) for every following
 * la_step until called with host = NULL.  The forward still runs; only the
 * integer controller reads the override, so that a test can drive it through
 * any acceptance pattern.  LA_ERR_ARG for n != T or a token outside the
 * vocabulary.  Synchronises the context's stream. */
LA_API int la_debug_set_argmax_override(la_ctx* ctx, const int32_t* host, int n);

/* No counterpart on the pages: message of the last failure on ctx. */
LA_API const char* la_last_error(la_ctx* ctx);
/* No counterpart on the pages: frees the context (and its own workspace). */
LA_API void la_destroy(la_ctx* ctx);

/* ---- standalone attention (one layer of the combined step, bf16) ----
 * Pages: "Summary" (both branches share one forward pass; the method works
 * with FlashAttention-style attention).
 * The masked attention la_step runs in every layer, on its own: the T =
 * 1 + (W+G)(N-1) rows of a step (current token, W x (N-1) lookahead-window
 * rows, G full candidates x (N-1) verification rows, in that order) at
 * positions P + offset attend to the cache [0,P) and to the in-step rows the
 * combined 2D-window + verification mask lets them see (the lookahead
 * branch and verification branch of the summary page's "Summary").
 *   q       DEVICE bf16 [T][n_heads][head_dim]  (rotary embedding applied)
 *   k_cache DEVICE bf16 [n_kv_heads][max_seq][head_dim], v_cache likewise;
 *           positions [0,P) are read
 *   k_step  DEVICE bf16 [T][n_kv_heads][head_dim], v_step likewise
 *   out     DEVICE bf16 [T][n_heads * head_dim]
 * head_dim 64 or 128; P + W + N - 1 <= max_seq (else LA_ERR_CAPACITY).
 * Allocates its scratch with cudaMallocAsync on stream and synchronises the
 * stream before returning. */
LA_API int la_attention(const void* q, const void* k_cache, const void* v_cache, const void* k_step,
                        const void* v_step, void* out, int n_heads, int n_kv_heads, int head_dim, int max_seq, int P,
                        int W, int N, int G, void* stream);

/* la_attention without allocating device memory.  No counterpart in the
 * paper.  It is for callers that cannot call cudaMalloc: runtimes that carve
 * all device memory out of one pool at start-up and forbid further device
 * allocation, and latency-bound callers for which the allocator's implicit
 * device-wide synchronisation or its failure modes are not acceptable.  Same
 * arguments and result as la_attention.  Scratch (the step's row tables, the
 * decode-state word and the attention's split partials) lives in one fixed
 * 16 MiB device array inside this library, which every GPU that loads the
 * library holds until the process exits.  The call needs
 *   ceil256((5*128 + 1 + g * o) * 4) + ceil256(sizeof decode state)
 *   + n_heads * ceil(max_seq / 256) * 128 * (head_dim + 4) * 4   bytes,
 * g = max(1, W + G) row groups, o = 1 + the largest position offset of a
 * step row (W + N - 2 with a window, N - 1 with candidates only, 0 for plain
 * greedy); more than the array holds
 * returns LA_ERR_CAPACITY with a message on stderr.  The first call on a
 * device, with that device current, looks up the array's device address and
 * sets the kernels' shared-memory limit (thread-safe, once per device).
 * Every call shares the array: calls that overlap on the GPU race.  Nothing
 * in it needs to start at zero (each call rewrites what it reads).  The
 * tables are uploaded from host memory and the call synchronises the stream
 * before returning. */
LA_API int la_attention_noalloc(const void* q, const void* k_cache, const void* v_cache, const void* k_step,
                                const void* v_step, void* out, int n_heads, int n_kv_heads, int head_dim, int max_seq,
                                int P, int W, int N, int G, void* stream);

/* ---- standalone n-gram pool (the pool the step uses, exposed for bulk work) ----
 * Pages: "Summary" (the n-grams the lookahead branch produces are cached in a
 * pool and checked by the verification branch).
 * A GPU hash table keyed on a token, each key holding up to G (N-1)-grams in
 * insertion order with first-in-first-out eviction; an insert of an n-gram
 * already held is a no-op.  Open addressing with warp-cooperative probing.
 * capacity: number of key slots (rounded up to a power of two, >= 64). */
typedef struct la_pool la_pool;
/* Pages: "Summary" (the pool).  Keys are tokens, >= 0. */
LA_API int la_pool_create(int capacity, int N, int G, void* stream, la_pool** out);
/* Pages: "Summary" (n-grams cached in the pool).
 * Insert n (key, (N-1)-gram) pairs in index order (equal keys keep their
 * order; distinct keys are inserted in parallel).  keys: DEVICE int32[n],
 * grams: DEVICE int32[n][N-1].  LA_ERR_CAPACITY when the table is full;
 * LA_ERR_ARG when a key is negative (that insert is skipped, the others are
 * made).  Synchronises the pool's stream. */
LA_API int la_pool_insert(la_pool* pool, const int32_t* keys, const int32_t* grams, int n);
/* Pages: "Summary" (candidates for verification come from the pool).
 * Look up n keys.  out: DEVICE int32[n][G][N-1] (oldest first, unused slots
 * -1), counts: DEVICE int32[n] (0 for absent or negative keys).
 * Asynchronous on the pool's stream. */
LA_API int la_pool_lookup(la_pool* pool, const int32_t* keys, int n, int32_t* out, int32_t* counts);
/* Pages: "Summary" (the pool).  Number of keys held (synchronises the stream). */
LA_API int la_pool_size(la_pool* pool, int* n_keys);
/* No counterpart on the pages: frees the pool. */
LA_API void la_pool_destroy(la_pool* pool);

#ifdef __cplusplus
}
#endif
#endif /* LOOKAHEAD_H */
