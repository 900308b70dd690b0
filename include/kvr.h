/*
 * kvr.h -- prefix-reused (suffix) prefill against a resident GPU KV slot.
 *
 * One process, one GB300 (sm_103a).  The library keeps a table of KV-cache
 * slots, one conversation each, and runs only the un-cached suffix of a
 * prompt (or the m = k+1 rows of a speculative verify) through a decoder
 * stack whose K/V for the cached prefix already sit in the slot.
 *
 * Sources (page title, section):
 *   goinfer "Turn nine in under half a second":
 *     "What goinfer does"  -- recent conversations keep their K and V rows
 *                             (one key and one value row per token and
 *                             layer); a prompt runs only past the part a
 *                             conversation already holds.
 *     "How it works"       -- the slot with the longest common token prefix
 *                             wins, provided that prefix exceeds the longest
 *                             prefix this slot has in common with any other
 *                             slot; the slot is truncated to the common
 *                             length; on a GPU model --kv-sessions slots,
 *                             an empty one first, else the least recently
 *                             used; usage.prefill_reused_tokens.
 *     "Use it"             -- --kv-sessions N (0 turns reuse off); the memory
 *                             check may grant fewer slots than asked for.
 *     "What we got wrong"  -- the one-token-short cache after speculation.
 *   thinkspread "The economics of speculative decoding", cost model -- the
 *     m = k+1 verify rows run as one batched pass that reads each weight once.
 *   OpenJev "Latency", What changed / Repeated state -- several questions
 *     resume from one checkpoint placed exactly at the end of a shared state;
 *     Next -- continuous batching across requests.
 *   Tempo9 docs: "KV cache spills to disk, by default" (slot spill/restore
 *     with a configuration hash) and "Models and quantizations" (Q4_K: 256
 *     weights in 144 bytes).
 *
 * ---------------------------------------------------------------------------
 * Ownership.  The caller allocates every device buffer (the KV arena, the
 * scratch area, weights, inputs, outputs) and owns the CUDA stream.  The
 * library makes no device allocation; it owns host state (the slot token
 * lists, lengths, LRU stamps, cached TMA descriptors) and, on each GPU that
 * loads it, the fixed staging array of kvr_slot_match_static.  All calls that take a
 * stream are asynchronous on it, except kvr_slot_match (it waits for the
 * stream to read back the match lengths), kvr_verify_accept (it returns the
 * decision to the host) and kvr_sync_status.
 *
 * Errors.  Every int-returning call returns KVR_OK (0) or a negative code;
 * kvr_last_error() says why.  A call refused by its checks launches nothing
 * and leaves every slot's length and tokens unchanged (validation precedes
 * any launch); what a call leaves after a failure past that point is stated
 * with the call.
 *
 * Threads.  A context is not thread-safe; serialise calls on one context.
 * ---------------------------------------------------------------------------
 */
#ifndef KVR_H
#define KVR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVR_OK 0
#define KVR_ERR_ARG (-1)         /* null pointer, bad slot, n <= 0, m <= 0, bad config   */
#define KVR_ERR_CAPACITY (-2)    /* len + m > capacity, m > max_rows, small arena/scratch */
#define KVR_ERR_CUDA (-3)        /* a CUDA runtime / driver call failed                   */
#define KVR_ERR_TIMEOUT (-4)     /* a device-side wait gave up (status word set)          */
#define KVR_ERR_FAULT (-5)       /* injected through the KVR_FAULT environment variable   */
#define KVR_ERR_UNSUPPORTED (-6) /* a shape the kernels do not handle (see kvr_config)    */
#define KVR_ERR_MISMATCH (-7)    /* a spilled slot from another model or KV layout        */

#define KVR_WEIGHTS_BF16 0
#define KVR_WEIGHTS_INT4_G32 1
#define KVR_WEIGHTS_Q4K 2

#define KVR_MAX_SLOTS 16
#define KVR_MAX_BRANCHES 16

/*
 * Model and table configuration.
 *   n_slots        requested KV slots (--kv-sessions).  0 = reuse off: one
 *                  working slot, every kvr_slot_match returns slot 0 with
 *                  reused = 0.  At most KVR_MAX_SLOTS.
 *   capacity       tokens per slot; a multiple of 64.
 *   n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn
 *                  decoder shape.  head_dim is 64 or 128; n_q_heads is a
 *                  multiple of n_kv_heads (grouped-query attention: query head
 *                  h reads KV head h / (n_q_heads / n_kv_heads)).
 *   weight_format  KVR_WEIGHTS_BF16, KVR_WEIGHTS_INT4_G32 or KVR_WEIGHTS_Q4K
 *                  (layouts below).
 *                  For int4 every projection's input width K must be a
 *                  multiple of 256.
 *   attn_only      1: a layer is out = Attn(x) Wo^T (no norms, no FFN, no
 *                  residual).  0: the pre-norm decoder layer
 *                    a = RMSNorm(h); h += Attn(a) Wo^T;
 *                    b = RMSNorm(h); h += (silu(b Wg^T) * (b Wu^T)) Wd^T.
 *   match_threshold 1 (default): the anti-theft rule of kvr_slot_match.
 *   max_rows       largest m of one prefill / verify / branches call; sizes
 *                  the scratch area.
 *   rope_theta     rotate-half RoPE base; rows sit at absolute slot positions.
 *   rms_eps        RMSNorm epsilon.
 *   vocab          largest output-head vocabulary (kvr_verify_accept); 0 for
 *                  none.  Sizes the scratch area; at most KVR_MAX_VOCAB.
 */
#define KVR_MAX_VOCAB 262144

typedef struct kvr_config {
  int n_slots;
  int capacity;
  int n_layers;
  int hidden;
  int n_q_heads;
  int n_kv_heads;
  int head_dim;
  int ffn;
  int weight_format;
  int attn_only;
  int match_threshold;
  int max_rows;
  float rope_theta;
  float rms_eps;
  int vocab;
} kvr_config;

/*
 * Weights of one layer: device pointers owned by the caller, stable while a
 * call that uses them is in flight.  Matrices are in the torch Linear
 * orientation [N][K] (output row n, input k):
 *   wq [Hq*d][H], wk [Hkv*d][H], wv [Hkv*d][H], wo [H][Hq*d],
 *   wg [F][H], wu [F][H], wd [H][F]   (wg/wu/wd unused when attn_only).
 * KVR_WEIGHTS_BF16: w* are bf16 [N][K] row-major; s* unused.
 * KVR_WEIGHTS_INT4_G32 (symmetric int4, one fp16 scale per 32 inputs):
 *   w* are uint8 [N][K/2]: row n is K/2 bytes.  Group g of row n (inputs
 *   32g .. 32g+31) is the 16 bytes at row offset 16g, read as four
 *   little-endian 32-bit words.  Input k' = k - 32g (0..31) is held in word
 *   (k' mod 8) div 2, in the 4-bit field number (k' div 8) + 4*(k' mod 2)
 *   counted from the least significant bits.  A field holds code + 8 with
 *   code in [-8, 7].
 *   s* are fp16 [N][K/32] row-major; weight(n, k) = code(n, k) * s[n][k/32].
 *   Any positive finite fp16 scale is accepted (no requirement on its
 *   significant bits).  Precision of the arithmetic: calls with up to 32 rows
 *   (the GEMV) use code * scale exactly (fp32 sums of code * x per group,
 *   scaled in fp32).  Calls with more rows (the tcgen05 GEMM, fp16 operands)
 *   keep the Q, K and V projections exact too (each weight as two fp16
 *   terms, two MMAs) and round each O, gate, up and down weight once to fp16
 *   (relative error at most 2^-12); their activations are the model's bf16
 *   values, which fp16 holds exactly for magnitudes 2^-14 .. 65504, so an
 *   activation above 65504 (not produced by these random-weight workloads,
 *   and unusual for real ones) would overflow that path.
 *   (The field order lets one 32-bit shared-memory load give a tensor-core
 *   fragment its eight inputs of one group.)
 * KVR_WEIGHTS_Q4K (K-quant 4-bit superblocks; Tempo9 docs, "Models and
 * quantizations": Q4_K keeps 256 weights in 144 bytes; the byte layout
 * inside is this library's, the pages give only the size):
 *   w* hold codes q in [0, 15] in the int4 layout above (a field holds q,
 *   no offset).  s* are uint8 [N][K/256][16]: for row n and superblock s
 *   (inputs 256s .. 256s+255) fp16 d (bytes 0-1), fp16 dmin (bytes 2-3) and
 *   a little-endian 96-bit string (bytes 4-15) of sixteen 6-bit fields,
 *   field f at bits 6f: fields 0-7 the scales sc_j, fields 8-15 the mins mn_j
 *   of sub-block j (inputs 256s + 32j .. +31).
 *   weight(n, k) = d*sc_j*q - dmin*mn_j.  The small-m GEMV applies d*sc_j
 *   and dmin*mn_j to fp32 sums; the tcgen05 GEMM forms each weight in fp32
 *   and, as for int4, keeps it as two fp16 terms for Q, K and V and rounds
 *   it once to fp16 for the other projections.
 *   Every projection input width must be a multiple of 256 (as for int4).
 * norm_attn, norm_ffn: bf16 [H] RMSNorm gains (unused when attn_only).
 * Every pointer must be 16-byte aligned.
 */
typedef struct kvr_layer_weights {
  const void *wq, *wk, *wv, *wo, *wg, *wu, *wd;
  const void *sq, *sk, *sv, *so, *sg, *su, *sd;
  const void *norm_attn, *norm_ffn;
} kvr_layer_weights;

typedef struct kvr_ctx kvr_ctx;

/*
 * Device bytes the caller must provide.
 * KV arena (slot-major; a slot's region is contiguous), bf16:
 *   K of slot s, layer l, KV head j, position p, element e at
 *     ((((s*L + l)*2 + 0)*Hkv + j)*capacity + p)*head_dim + e   ([capacity][head_dim] per head);
 *   V is stored transposed, element e of position p at
 *     ((((s*L + l)*2 + 1)*Hkv + j)*head_dim + e)*capacity + p   ([head_dim][capacity] per head),
 *   so that both tensor-core operands of P.V are K-major tiles;
 *   followed by the device token mirror int32 [n_slots][capacity].
 *   kvr_ctx_create zeroes the K/V part once.  Attention reads whole 64-key
 *   blocks, so positions past a slot's length (weighted by zero) must hold
 *   finite values: everything the library writes is finite, and K/V a caller
 *   writes itself (kvr_slot_assign) must be finite too.
 *   kvr_arena_bytes(cfg, n) is the size for n slots (n = cfg->n_slots, or 1
 *   when n_slots is 0).
 * Scratch: activations, partial sums, RoPE tables, the match buffers and the
 *   device status word; its contents do not outlive a call.
 * Both return 0 for an invalid configuration.
 */
size_t kvr_arena_bytes(const kvr_config* cfg, int n_slots);
size_t kvr_scratch_bytes(const kvr_config* cfg);

/*
 * Create a context over caller-allocated device memory (256-byte aligned).
 * If arena_bytes holds fewer slots than cfg->n_slots (but at least one) the
 * context grants that many and kvr_ctx_info reports both numbers ("Use it":
 * the memory check may allow fewer slots than asked for).  Fails with
 * KVR_ERR_CAPACITY if not even one slot or the scratch area fits.  Must be
 * called with the device that owns the buffers current.
 */
int kvr_ctx_create(const kvr_config* cfg, void* kv_arena, size_t arena_bytes, void* scratch,
                   size_t scratch_bytes, kvr_ctx** out);
int kvr_ctx_info(const kvr_ctx* ctx, int* slots_granted, int* slots_requested, int* capacity);
int kvr_ctx_destroy(kvr_ctx* ctx);

/*
 * Choose the slot for a prompt (tokens: host int32[n], n >= 1) and cut it
 * back to the shared point.  Prefix lengths are computed on the device by the
 * prefix-match kernel on `stream`; the call then synchronises on the stream
 * and applies the policy on the host:
 *   l(s) = longest common token prefix of slot s and the prompt;
 *   o(s) = longest common prefix of slot s and any other occupied slot;
 *   s* = the occupied slot with the largest l (lowest index on ties).
 *   With match_threshold = 1, s* is accepted iff l(s*) > 0, l(s*) > o(s*), and
 *   it would not cut s* back (l(s*) < len(s*)) while another slot is empty.
 *   With match_threshold = 0, s* is accepted iff l(s*) > 0.
 *   Accepted: reused = min(l(s*), n-1); the slot is truncated to reused.
 *   Otherwise the lowest-index empty slot, else the least recently used slot,
 *   restarts empty: reused = 0.
 * *slot receives the slot, *reused the count to report as
 * usage.prefill_reused_tokens.  The caller then prefills tokens[reused:].
 */
int kvr_slot_match(kvr_ctx* ctx, const int32_t* tokens, int n, int* slot, int* reused,
                   void* stream);
/*
 * kvr_slot_match_static -- kvr_slot_match for callers that cannot allocate
 * device memory for it.  (The pages have no counterpart: this is a property
 * of the library, not of the method.)
 *
 * kvr_slot_match stages the prompt and its match lengths in the scratch area
 * handed to kvr_ctx_create.  Some callers have no device memory to hand over
 * when they match: a request router or scheduler thread whose process leaves
 * every device byte to another component's caching allocator (calling
 * cudaMalloc behind that allocator's back breaks its accounting and can fail
 * when it holds the whole device), or code that must not allocate while
 * another stream is being captured into a CUDA graph.  This call computes the
 * same (slot, reused) with the same policy, but stages everything in a fixed
 * array inside the library: KVR_STATIC_MATCH_MAX_TOKENS prompt tokens plus
 * the slot and match lengths (about 66 KB), held by every GPU that loads the
 * library until the process exits.  It calls no cudaMalloc/cudaFree.
 *
 * Limits and rules:
 *  - n > KVR_STATIC_MATCH_MAX_TOKENS (or > capacity) fails with
 *    KVR_ERR_CAPACITY and a message saying so; nothing is launched.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture on the device.  The address is cached per
 *    device for the life of the process: it does not survive a
 *    cudaDeviceReset or any other teardown of the device's primary context.
 *    After one, the next call returns a stale address; do not call this
 *    entry point again in that process.
 *  - Every call, from every context on the device, shares the one array and
 *    leaves its contents behind.  Each call writes every word it reads
 *    before reading it, so nothing needs clearing; but calls that overlap on
 *    the GPU (different streams or threads without ordering) race on the
 *    array and may return wrong results.  Serialise them.
 */
#define KVR_STATIC_MATCH_MAX_TOKENS 16384
int kvr_slot_match_static(kvr_ctx* ctx, const int32_t* tokens, int n, int* slot, int* reused,
                          void* stream);

/* Cut a slot back to new_len <= len (a host length update; K/V beyond it are
 * simply ignored from then on).  Used after a verify to keep p0+1+accepted. */
int kvr_slot_truncate(kvr_ctx* ctx, int slot, int new_len);
int kvr_slot_len(const kvr_ctx* ctx, int slot, int* len);
/* Copy of the first min(n, len) tokens of a slot into host tokens[]. */
int kvr_slot_tokens(const kvr_ctx* ctx, int slot, int32_t* tokens, int n);
/* Declare that slot `slot` holds tokens[0..n) whose K/V the caller has
 * written into the arena (restoring a saved slot, or synthetic K/V).  Uploads
 * the token mirror on `stream`. */
int kvr_slot_assign(kvr_ctx* ctx, int slot, const int32_t* tokens, int n, void* stream);
/* Device addresses of a slot's K and V for one layer: K is [Hkv][capacity][head_dim] bf16,
 * V is [Hkv][head_dim][capacity] bf16 (transposed, see the arena layout). */
int kvr_slot_kv(const kvr_ctx* ctx, int slot, int layer, void** k, void** v);

/*
 * Slot spill and restore through host memory (Tempo9 docs, "KV cache spills
 * to disk, by default": reusable prefixes leave device memory and come back
 * later; a record made under a different model, number format or KV layout
 * is detected through a configuration hash and discarded, never reused).
 * Files, the size cap and eviction of records are the caller's.
 *
 * kvr_config_hash: FNV-1a (64-bit) over the fields that fix what a slot's K/V
 * hold -- n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn,
 * weight_format, attn_only, rope_theta, rms_eps (as little-endian 32-bit
 * words, in that order) -- followed by the caller's 64-bit model_tag (which
 * names the weights).  n_slots, capacity, match_threshold, max_rows and vocab
 * do not enter: a record restores into any context whose capacity holds it.
 *
 * Record (host bytes, written by kvr_slot_spill, 16-byte aligned sections):
 *   64-byte header: magic "KVRSLOT1", the hash, len, n_layers, n_kv_heads,
 *     head_dim, the byte size of the record;
 *   tokens int32[len], padded to 16 bytes;
 *   per layer l: K as [Hkv][len][head_dim] bf16, then V^T as
 *     [Hkv][head_dim][len] bf16 (the arena's layout with capacity cut to len).
 * kvr_slot_spill_bytes gives the record size of a slot's current length.
 *
 * kvr_slot_spill copies the slot into host (caller-owned, `bytes` long) on
 * `stream`; the record is complete once the stream reaches that point (pinned
 * host memory makes the copies asynchronous).  KVR_ERR_CAPACITY if bytes is
 * too small.  The slot is unchanged.
 * kvr_slot_restore checks the header (KVR_ERR_MISMATCH for another hash,
 * KVR_ERR_ARG for a damaged header, KVR_ERR_CAPACITY if len > capacity), then
 * copies the K/V into `slot` on `stream`, sets its tokens and refreshes its
 * LRU stamp.  The host record must stay valid until the stream reaches the
 * copies.  A refused record leaves the slot unchanged; a copy that fails
 * leaves it empty (length 0).
 */
uint64_t kvr_config_hash(const kvr_config* cfg, uint64_t model_tag);
size_t kvr_slot_spill_bytes(const kvr_ctx* ctx, int slot);
int kvr_slot_spill(kvr_ctx* ctx, int slot, uint64_t model_tag, void* host, size_t bytes, void* stream);
int kvr_slot_restore(kvr_ctx* ctx, int slot, uint64_t model_tag, const void* host, size_t bytes,
                     void* stream);

/*
 * Suffix prefill: run m rows (tokens: host int32[m]; hidden: device bf16
 * [m][hidden], the rows' input hidden states) at positions p0 .. p0+m-1 of
 * slot `slot`, p0 = the slot's length.  Each row attends causally to the
 * slot's cached K/V [0, p0) and to the new rows up to itself; the new rows'
 * K/V are appended.  w: host array of n_layers kvr_layer_weights.  out:
 * device bf16 [m][hidden], the last layer's output (the residual stream for a
 * full layer, Attn(x) Wo^T for attn_only).  On success the slot's length is
 * p0+m and its tokens gain tokens[0..m).
 * KVR_ERR_CAPACITY if p0+m > capacity or m > max_rows.
 */
int kvr_prefill_suffix(kvr_ctx* ctx, int slot, const int32_t* tokens, int m, const void* hidden,
                       const kvr_layer_weights* w, void* out, void* stream);

/* Speculative verify: the same computation for the m = k+1 rows (the last
 * accepted token plus k drafts).  The rows are appended; the caller then calls
 * kvr_slot_truncate(slot, p0 + 1 + accepted) so the cache holds exactly the
 * committed tokens (the "one token short" fix).  1 <= m <= 64. */
int kvr_verify(kvr_ctx* ctx, int slot, const int32_t* tokens, int m, const void* hidden,
               const kvr_layer_weights* w, void* out, void* stream);

/*
 * Several questions resuming from one checkpoint in one batch.  The slot's
 * length P is the checkpoint.  Branch b has lens[b] rows (rows are
 * concatenated in branch order: tokens host int32[sum], hidden device bf16
 * [sum][hidden]).  Row i of branch b sits at position P+i, as if it were the
 * only question, and attends to [0, P) plus its own branch's rows up to
 * itself.  The branches' K/V are written after position P (in branch order)
 * but are not committed: the slot keeps length P and its tokens.
 * 1 <= n_branch <= KVR_MAX_BRANCHES; P + sum(lens) <= capacity.
 */
int kvr_prefill_branches(kvr_ctx* ctx, int slot, int n_branch, const int* lens,
                         const int32_t* tokens, const void* hidden, const kvr_layer_weights* w,
                         void* out, void* stream);

/*
 * Several conversations in one call (continuous batching across requests:
 * OpenJev "Next"; goinfer "What was measured", several clients each keeping
 * their own history; the Tempo9 agents article, "concurrency").  Conversation
 * j appends lens[j] rows to slot slots[j] after that slot's len_j cached
 * tokens, with the same result as kvr_prefill_suffix(slots[j], ...) alone;
 * the projections read each weight once for the rows of every conversation,
 * and attention runs per conversation over its own slot.
 *   n_seq          1 .. KVR_MAX_BRANCHES; slots[] distinct and granted.
 *   lens           host [n_seq], each >= 1; sum <= max_rows and
 *                  len_j + lens[j] <= capacity.
 *   tokens         host int32 [sum lens], conversation-major.
 *   hidden, out    device bf16 [sum lens][hidden] in the same order.
 * A verify of several conversations is this call followed by one
 * kvr_slot_truncate per slot.  Errors as kvr_prefill_suffix; on error no
 * slot's length changes.
 */
int kvr_prefill_batch(kvr_ctx* ctx, int n_seq, const int* slots, const int* lens, const int32_t* tokens,
                      const void* hidden, const kvr_layer_weights* weights, void* out, void* stream);

/* Wait for `stream` and check the device status word that kernels set when a
 * bounded device-side wait gives up.  Returns KVR_ERR_TIMEOUT (and clears the
 * word and the kernels' arrival counters, so the next call starts clean) if
 * one did; the outputs of the call that timed out are not to be used.
 * While the word is set, every kernel the library launches leaves at entry
 * and every pending wait gives up within microseconds: the calls issued after
 * a timeout and before this check compute nothing (their outputs, and the
 * K/V rows they were to append, are not to be used either). */
int kvr_sync_status(kvr_ctx* ctx, void* stream);

/* Per-layer trace for checking a long stack one layer at a time.  While a
 * buffer is set (dev: device float32 [n_layers + 1][max_rows][hidden],
 * bytes >= that size; NULL clears it), every prefill / verify / branches call
 * of a full-layer model (attn_only = 0) copies the float32 residual stream of
 * its m rows into it on the call's stream: entry 0 after the first RMSNorm's
 * input load, entry l+1 after layer l (row i of entry e at
 * (e*max_rows + i)*hidden).  Returns KVR_ERR_CAPACITY if bytes is too small. */
int kvr_trace_set(kvr_ctx* ctx, void* dev, size_t bytes);

/* The output head for greedy verification: the final RMSNorm gain and the
 * LM head in the layer weights' int4 group-32 layout (device pointers, caller-
 * owned, 16-byte aligned). */
typedef struct {
  const void* norm;  /* bf16 [hidden]                              */
  const void* w;     /* int4 bytes [vocab][hidden/2]               */
  const void* s;     /* fp16 group scales [vocab][hidden/32]       */
  int vocab;         /* 1 .. the context's configured vocab        */
} kvr_head_weights;

/* Speculative verify with the greedy decision (goinfer "What we got wrong":
 * a speculative step checks the guessed tokens and must give the same words
 * as plain decoding; thinkspread, cost model: the m = k+1 rows run as one
 * batched pass).  tokens (host, m <= 64) are [t0, d1 .. dk]: t0 the last
 * committed token, d the drafts; rows sit at p0 .. p0+m-1, p0 = the slot's
 * length.  Runs kvr_verify, then logits = RMSNorm(h) * lm^T per row (the
 * normed rows rounded to bf16), next_tokens[i] = argmax of row i (lowest
 * index on ties), *accepted = the number of leading drafts with
 * d_(j+1) == next_tokens[j].  The slot is cut back to p0 + 1 + accepted (the
 * next token, next_tokens[accepted], is not in the cache).  out (device bf16
 * [m][hidden]) receives the rows' outputs as kvr_verify's, or may be null.
 * next_tokens (host, m entries) and accepted are written after the call has
 * synchronised the stream.  int4 weights only (KVR_ERR_UNSUPPORTED otherwise).
 * On error the slot keeps its length before the call. */
int kvr_verify_accept(kvr_ctx* ctx, int slot, const int32_t* tokens, int m, const void* hidden,
                      const kvr_layer_weights* weights, const kvr_head_weights* head, void* out,
                      int32_t* next_tokens, int* accepted, void* stream);

/* Greedy verification of several conversations in one call: the rows of
 * conversation j ([t0, d1 .. dk] of slot slots[j], lens[j] of them, in the
 * order and layout of kvr_prefill_batch, at most 64 rows in all) run as one
 * batch, then the output head decides every row.  next_tokens (host, sum of
 * lens) receives every row's argmax and accepted (host, n_seq) each
 * conversation's count of accepted drafts; slot slots[j] is cut back to its
 * length before the call + 1 + accepted[j].  Conversation j's results equal
 * kvr_verify_accept on its slot alone.  Synchronises the stream.  On an error
 * after the rows ran every slot keeps its length before the call. */
int kvr_verify_accept_batch(kvr_ctx* ctx, int n_seq, const int* slots, const int* lens,
                            const int32_t* tokens, const void* hidden, const kvr_layer_weights* weights,
                            const kvr_head_weights* head, void* out, int32_t* next_tokens, int* accepted,
                            void* stream);

/* Self-test of the failure path, without a GPU fault: launches one device
 * wait on an mbarrier that nothing completes.  Like every wait in the
 * library's kernels it gives up after 1 s and records the timeout in the
 * status word; the next kvr_sync_status returns KVR_ERR_TIMEOUT, clears the
 * word and the arrival counters (projection tiles and attention splits), and
 * the context stays usable. */
int kvr_selftest_wait(kvr_ctx* ctx, void* stream);

/* Per-kernel-class timing with CUDA events recorded on the launch stream.
 * While enabled, every launch is bracketed by an event pair; kvr_profile_read
 * synchronises and returns milliseconds summed since the last read for
 * classes: 0 projections (GEMV/GEMM), 1 attention (incl. split merge),
 * 2 epilogues / norms / RoPE tables, 3 prefix match; and launch counts. */
int kvr_profile_enable(kvr_ctx* ctx, int on);
int kvr_profile_read(kvr_ctx* ctx, float ms[4], int launches[4]);

/* The launches recorded since the last kvr_profile_read, in launch order:
 * cls[i] (as above) and ms[i], the time between the event pair around launch
 * i (the kernel plus any wait for the host to issue it).  Synchronises; fills
 * at most max_n entries and sets *n to the number recorded.  Does not reset:
 * kvr_profile_read still returns (and clears) the sums. */
int kvr_profile_launches(kvr_ctx* ctx, int* cls, float* ms, int max_n, int* n);

const char* kvr_last_error(const kvr_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* KVR_H */
