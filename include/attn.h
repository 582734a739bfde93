/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * The library computes scaled-dot-product attention forward,
 *
 *     S = scale * Q K^T  (+ causal mask),   P = softmax(S),   O = P V,
 *     lse = m + ln(l)    (per query row: m = max_j S, l = sum_j exp(S - m)),
 *
 * as defined by the standard attention chain of "GPU 学习日报 Day 24：Operator
 * Fusion" (Operator Fusion, GPU learning diary day 24), §3.4 "Attention Fusion:
 * FlashAttention", computed by the tiled online-softmax recurrence of the same
 * section's second listing (running row max m, running row sum l, rescaled O
 * accumulator, one normalisation at the end), so that the Lq x Lkv score matrix
 * never reaches HBM.  The log-sum-exp output is not on that page; it is the
 * natural-log normaliser built from the m and l that listing carries.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never frees or retains them.  Every pointer must be 16-byte aligned.
 *  - Element types: q, k, v, kcache, vcache are bf16 (raw 16-bit words, passed
 *    as void*).  out is bf16 unless an *_ex call asks for fp32.  lse is fp32.
 *  - Arithmetic: fp32 accumulation everywhere; on the tensor-core paths
 *    (prefill, multi-token decode) P is rounded to bf16 before the P V
 *    product, single-token decode keeps P in fp32.
 *  - Causal masking is aligned to the bottom-right corner: key j is visible to
 *    query i iff j <= i + (Lkv - Lq).  For Lq == Lkv this is the lower
 *    triangle.  A query row that sees no key gets O = 0 and lse = -inf.
 *  - Grouped-query attention: Hq must be a multiple of Hkv; query head h reads
 *    key/value head h / (Hq / Hkv) (contiguous groups).
 *  - D (head dimension) must be 64 or 128.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous with respect to the host: they enqueue kernels and return.
 *  - Errors the host can see (NULL pointer, bad size, misalignment, wrong GPU)
 *    are returned synchronously before anything is enqueued.  A CUDA launch
 *    failure returns ATTN_ERR_CUDA.  Problems only the device can see (a
 *    kv_len outside [0, Lmax], a pipeline wait that timed out) are recorded in
 *    a per-device status word read by attn_get_device_status(); the kernels
 *    never trap.
 *  - There is no CPU fallback: without an sm_103 device every compute call
 *    returns ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,     /* NULL pointer, non-positive size, Hq % Hkv != 0, ... */
  ATTN_ERR_UNSUPPORTED = 2,     /* D not in {64,128}, device is not sm_103, ...        */
  ATTN_ERR_ALIGNMENT = 3,       /* a pointer is not 16-byte aligned                    */
  ATTN_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed                */
  ATTN_ERR_DEVICE_TIMEOUT = 5,  /* device status: a bounded pipeline wait expired      */
  ATTN_ERR_DEVICE_BOUNDS = 6,   /* device status: a kv_len was outside [0, Lmax]       */
  ATTN_ERR_SCRATCH_TOO_SMALL = 7 /* attn_decode_noalloc: partials exceed its fixed buffer */
} attn_status;

typedef enum attn_dtype { ATTN_DTYPE_BF16 = 0, ATTN_DTYPE_F32 = 1 } attn_dtype;

/*
 * attn_rope -- rotary position embedding (RoPE) applied inside the kernels,
 * as "Что такое kernel fusion и как он применяется в LLM serving?" §3.5 and
 * Operator Fusion's exercise 1 (RoPE fused into the attention kernel)
 * describe; the pages give no formula, so the standard rotary embedding is
 * used: pair i of a row at position p, (a, b), becomes
 *     (a * cos[p][i] - b * sin[p][i],  b * cos[p][i] + a * sin[p][i]),
 * the pairs being dims (i, i + D/2) for ATTN_ROPE_HALF and (2i, 2i + 1) for
 * ATTN_ROPE_INTERLEAVED.
 *
 *   cos, sin  DEVICE fp32 [max_pos, D/2] tables (row p: position p), 16-byte
 *             aligned; read-only.
 *   max_pos   rows of both tables.
 *   style     ATTN_ROPE_NONE (or cos == NULL): no rotation.
 *
 * Positions follow the causal alignment.  Prefill: key j of a sequence sits
 * at j and query i at Lkv - Lq + i (a dense call with Lq > Lkv returns
 * ATTN_ERR_INVALID_ARG; a packed sequence with more queries than keys is
 * flagged ATTN_ERR_DEVICE_BOUNDS).  The keys are rotated once per call by a
 * pass of their own into k_out (or the library workspace, grown like the
 * decode workspace and shared with it), the queries by a second pass into the
 * workspace, then the attention kernel streams the rotated copies.  Such a
 * call needs 256 KiB + (k_out ? 0 : rows of k * D * 2) + rows of q * D * 2
 * bytes of workspace; during CUDA graph capture it is never grown (make one
 * uncaptured call with the largest sizes first), and calls that can overlap
 * on the GPU race on it, as decode calls do.  Decode:
 * only the query is rotated, to kv_len - 1 (token t of attn_decode_multi to
 * kv_len - Lq + t); cached keys must be stored already rotated.  Every
 * position must be below max_pos: calls whose Lkv (prefill) or Lmax (decode)
 * exceeds max_pos return ATTN_ERR_INVALID_ARG.
 */
typedef enum attn_rope_style { ATTN_ROPE_NONE = 0, ATTN_ROPE_HALF = 1, ATTN_ROPE_INTERLEAVED = 2 } attn_rope_style;

typedef struct attn_rope {
  const float* cos;
  const float* sin;
  int max_pos;
  int style;
  void* k_out;  /* prefill only, optional: DEVICE bf16 buffer shaped like k (16-byte aligned) that receives the
                   rotated keys -- e.g. to append them to a KV cache; NULL = the library's workspace holds them */
} attn_rope;

/*
 * attn_fwd -- prefill attention over dense [batch, heads, seq_len, head_dim]
 * tensors (the Q/K/V shape of "Что такое kernel fusion и как он применяется в
 * LLM serving?", §2, and the chain of Operator Fusion §3.4).
 *
 *   q    bf16 [B, Hq,  Lq,  D]  contiguous
 *   k    bf16 [B, Hkv, Lkv, D]  contiguous
 *   v    bf16 [B, Hkv, Lkv, D]  contiguous
 *   out  bf16 [B, Hq,  Lq,  D]  written
 *   lse  fp32 [B, Hq,  Lq]      written; may be NULL (then not written)
 *   scale   multiplies the logits (pass 1/sqrt(D) for the standard chain), before
 *           the mask is added; any finite value, zero (uniform weights over the
 *           visible keys) and negative values included (NaN or +-inf:
 *           ATTN_ERR_INVALID_ARG).  Every entry point treats scale this way.
 *   causal  0 = no mask, 1 = bottom-right-aligned causal mask
 *
 * Runs on the tensor cores (tcgen05 MMAs with TMEM accumulators, TMA-fed
 * shared-memory tiles).  Returns an attn_status.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
             int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale, int causal,
             void* stream);

/*
 * attn_fwd_params / attn_fwd_ex -- prefill with every option.
 *
 * Dense layout (cu_seqlens_q == NULL): as attn_fwd; Lq/Lkv are the lengths.
 *
 * Packed variable-length layout (cu_seqlens_q != NULL and cu_seqlens_k != NULL):
 *   q    bf16 [total_q, Hq,  D]   (token-major, heads, head_dim)
 *   k/v  bf16 [total_k, Hkv, D]
 *   out       [total_q, Hq,  D]
 *   lse  fp32 [total_q, Hq]       may be NULL
 *   cu_seqlens_q/k  DEVICE int32 [B + 1], non-decreasing, cu[0] = 0,
 *                   cu_q[B] == total_q, cu_k[B] == total_k; sequence s owns
 *                   rows cu[s] .. cu[s+1]-1 and is an independent problem.
 *   Lq, Lkv   upper bounds of the per-sequence query / key lengths.
 *   B         number of sequences.
 *
 * out_dtype selects bf16 (ATTN_DTYPE_BF16) or fp32 (ATTN_DTYPE_F32) output.
 */
typedef struct attn_fwd_params {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  int B, Hq, Hkv, Lq, Lkv, D;
  float scale;
  int causal;
  int out_dtype;
  const int* cu_seqlens_q;
  const int* cu_seqlens_k;
  int total_q, total_k;
  void* stream;
  attn_rope rope;  /* optional; zero-initialised = no rotation */
} attn_fwd_params;

int attn_fwd_ex(const attn_fwd_params* p);

/*
 * attn_decode -- single-token decode over a KV cache ("Оптимизация Decoder
 * Attention для LLM на GPU", section on the structure of attention in decoding
 * mode: the new token's query against all cached keys, softmax, times V),
 * split along the KV sequence (Flash-Decoding, Operator Fusion FAQ Q4) and
 * merged by a log-sum-exp combine.
 *
 *   q        bf16 [B, Hq, D]
 *   kcache   bf16 [B, Hkv, Lmax, D]
 *   vcache   bf16 [B, Hkv, Lmax, D]
 *   kv_lens  DEVICE int32 [B]; sequence b attends to cache rows 0..kv_lens[b]-1.
 *            A value outside [0, Lmax] is clamped into it and flagged as
 *            ATTN_ERR_DEVICE_BOUNDS in the device status word.  kv_len == 0
 *            gives O = 0, lse = -inf.
 *   out      bf16 [B, Hq, D]
 *   lse      fp32 [B, Hq]  may be NULL
 *
 * Uses a library-owned split-KV workspace on the current device, grown on
 * demand with cudaMalloc (see attn_release_workspace); during CUDA graph
 * capture it is never grown (a call that would need a larger one returns
 * ATTN_ERR_INVALID_ARG: make one uncaptured call with the largest sizes
 * first).  Decode calls on one device share that workspace, so calls that can
 * overlap on the GPU (different streams with no ordering) race on it.
 * One kernel is enqueued: persistent CTAs (three per SM when a CTA serves up
 * to 4 query heads, two with 8) each stream an equal slice of the flattened
 * key space of all rows (every row also charged a fixed cost for its
 * piece-end work), and the CTA that lands a row's last partial merges that
 * row's partials.
 */
int attn_decode(const void* q, const void* kcache, const void* vcache, const int* kv_lens,
                void* out, float* lse, int B, int Hq, int Hkv, int Lmax, int D, float scale,
                void* stream);

/*
 * attn_decode_params / attn_decode_ex -- decode with every option.
 *   out_dtype     ATTN_DTYPE_BF16 or ATTN_DTYPE_F32
 *   chunk         0 = default; otherwise the smallest number of keys one CTA's
 *                 slice of the key space may hold (default 64), in
 *                 [1, 1048576]: smaller values spread short problems over more
 *                 CTAs and split rows into more partials.  The slices never
 *                 number fewer than the rows that have keys (while CTAs
 *                 last), so a short problem still runs a row per CTA.
 * Rows: B * Hkv * (Hq / Hkv / g) must stay at or below 65534, g being the
 * number of query heads one CTA serves (the largest of 8, 4, 2, 1 dividing
 * Hq / Hkv); otherwise ATTN_ERR_UNSUPPORTED.
 */
typedef struct attn_decode_params {
  const void* q;
  const void* kcache;
  const void* vcache;
  const int* kv_lens;
  void* out;
  float* lse;
  int B, Hq, Hkv, Lmax, D;
  float scale;
  int out_dtype;
  int chunk;
  void* stream;
  attn_rope rope;  /* optional; zero-initialised = no rotation */
} attn_decode_params;

int attn_decode_ex(const attn_decode_params* p);

/*
 * attn_decode_paged_params / attn_decode_paged -- decode over a paged KV cache
 * (the serving form of the cache: fixed-size pages from a shared pool, listed
 * per sequence in a block table, as in PagedAttention, which "Что такое kernel
 * fusion и как он применяется в LLM serving?" §6 names).  Same computation
 * and results as attn_decode_ex on the cache the pages describe.
 *
 *   kpages, vpages  bf16 [num_pages, Hkv, page_size, D]: page g of kv head h
 *                   holds page_size consecutive key (value) rows
 *   block_table     DEVICE int32 [B, max_pages]: entry (b, i) is the pool page
 *                   holding keys i*page_size .. (i+1)*page_size-1 of sequence b
 *   kv_lens         DEVICE int32 [B], at most max_pages * page_size (clamped
 *                   and flagged otherwise, as in attn_decode)
 *   page_size       keys per page, 8 .. 65536 (any value, not only powers of 2)
 *   max_pages       columns of block_table; num_pages rows of the pool.  Only
 *                   the entries of pages that hold keys of a sequence (the
 *                   first ceil(kv_len / page_size)) are read; the rest may hold
 *                   anything (e.g. -1 padding).  A page id read outside
 *                   [0, num_pages) is flagged ATTN_ERR_DEVICE_BOUNDS in the
 *                   device status word and page 0 is read instead.
 *   other fields    as attn_decode_params (q, out, lse, B, Hq, Hkv, D, scale,
 *                   out_dtype, chunk, stream); same workspace as attn_decode_ex.
 */
typedef struct attn_decode_paged_params {
  const void* q;
  const void* kpages;
  const void* vpages;
  const int* block_table;
  const int* kv_lens;
  void* out;
  float* lse;
  int B, Hq, Hkv, D;
  int page_size, max_pages, num_pages;
  float scale;
  int out_dtype;
  int chunk;
  void* stream;
  attn_rope rope;  /* optional; zero-initialised = no rotation */
} attn_decode_paged_params;

int attn_decode_paged(const attn_decode_paged_params* p);

/*
 * attn_decode_multi_params / attn_decode_multi -- decode of several new tokens
 * per sequence at once (multi-token or speculative decode), on the tensor
 * cores.  The decoder page ("Оптимизация Decoder Attention для LLM на GPU",
 * "Техника выжимания производительности", item 1: token-level parallelism)
 * processes several query tokens of a step together so that each K/V block is
 * loaded once for all of them and the tensor cores have work.
 *
 *   q        bf16 [B, Hq, Lq, D]   the Lq new tokens of every sequence
 *   kcache   bf16 [B, Hkv, Lmax, D]
 *   vcache   bf16 [B, Hkv, Lmax, D]
 *   kv_lens  DEVICE int32 [B]: the number of cached keys of sequence b,
 *            INCLUDING the Lq new tokens, whose keys and values must already
 *            be in rows kv_len-Lq .. kv_len-1.  New token t (0-based) sits at
 *            position kv_len - Lq + t and attends to keys 0 .. kv_len - Lq + t
 *            (the bottom-right causal mask of attn_fwd with Lkv = kv_len).
 *            Rows at or past kv_len are never read.  A value outside
 *            [0, Lmax] is clamped and flagged ATTN_ERR_DEVICE_BOUNDS; a token
 *            that sees no key (kv_len < Lq) gets O = 0, lse = -inf.
 *   out      [B, Hq, Lq, D]  bf16, or fp32 when out_dtype = ATTN_DTYPE_F32
 *   lse      fp32 [B, Hq, Lq]  may be NULL
 *   Lq       1 .. 128 / (Hq / Hkv): every query row of one kv head (the heads
 *            of its group times the tokens) forms one 128-row MMA tile;
 *            larger products return ATTN_ERR_UNSUPPORTED.
 * B * Hkv must stay at or below 65534 and B * Hq * Lq below 2^31
 * (ATTN_ERR_UNSUPPORTED otherwise).  Uses the split-KV workspace of
 * attn_decode (same growth, capture and concurrency rules).  One kernel is
 * enqueued: persistent CTAs (one per SM) each stream an equal share of all
 * sequences' 128-key tiles, and the CTA that lands an item's last partial
 * merges its partials.
 */
typedef struct attn_decode_multi_params {
  const void* q;
  const void* kcache;
  const void* vcache;
  const int* kv_lens;
  void* out;
  float* lse;
  int B, Hq, Hkv, Lq, Lmax, D;
  float scale;
  int out_dtype;
  void* stream;
  attn_rope rope;  /* optional; zero-initialised = no rotation */
} attn_decode_multi_params;

int attn_decode_multi(const attn_decode_multi_params* p);

/*
 * attn_decode_workspace_bytes -- bytes of split-KV workspace a decode call
 * with these sizes needs (0 on invalid sizes).  It depends on Hq / Hkv, D and
 * the current device's SM count (148 assumed when no device is visible), not
 * on B, Lmax or chunk: 256 KiB of counters plus two partials per CTA.
 */
unsigned long long attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int D, int chunk);

/*
 * attn_get_device_status -- synchronises `stream`, then returns and clears the
 * current device's status word (ATTN_OK if no kernel flagged a problem since
 * the last read).  Returns ATTN_ERR_CUDA if the synchronisation fails.
 */
int attn_get_device_status(void* stream);

/* attn_status_string -- static, NUL-terminated name of a status code. */
const char* attn_status_string(int status);

/*
 * attn_release_workspace -- frees the current device's split-KV workspace.
 * The caller must ensure no decode call using it is still in flight (for
 * example by synchronising the streams it was used on).
 */
void attn_release_workspace(void);

/*
 * attn_decode_noalloc -- attn_decode_ex for callers that must not allocate
 * device memory.  (The source pages have no counterpart: this entry point is
 * an integration aid, not part of the attention method.)
 *
 * Who needs it: code that runs while a CUDA graph is being captured (where a
 * cudaMalloc is not allowed), serving engines that reserve nearly all of HBM
 * up front for KV caches and route every allocation through their own pool,
 * and latency-critical paths that cannot afford the device-wide
 * synchronisation cudaMalloc/cudaFree can cause.  attn_decode_ex may grow its
 * workspace with cudaMalloc on the first call with a larger problem; this
 * call never does.
 *
 * Same arguments, layouts and results as attn_decode_ex.  Its scratch is a
 * fixed 4 MiB buffer compiled into the library (a file-scope __device__
 * array): every GPU on which the library's kernels are loaded holds that
 * buffer until the process exits, whether or not this call is used.  The
 * buffer holds 256 KiB of work counters followed by the split-KV partials,
 * two per CTA of the persistent launch (2.5 MiB at most on a 152-SM GB300).
 * A problem that does not fit -- more than 65534 (b, kv head, head group)
 * rows, or partials beyond the buffer on a device with more SMs -- returns
 * ATTN_ERR_SCRATCH_TOO_SMALL before anything is enqueued.
 *
 * No call allocates: no cudaMalloc, no cudaFree, no allocating library
 * routine.  The first call on a device looks up the buffer's device address
 * (cudaGetSymbolAddress, once per device, with that device current) and
 * zeroes the counter area (cudaMemset, then a device synchronise); make that
 * first call outside any stream capture (a first call on a capturing stream
 * returns ATTN_ERR_INVALID_ARG and leaves the capture untouched).  The kernel leaves the counters at
 * zero after every call, and every partial is written before it is read in
 * the same call.  All calls share the one buffer and it keeps the last call's
 * contents: two calls that can overlap on the GPU (different streams with no
 * ordering between them) race on it and may return wrong results.  Order such
 * calls on one stream.
 */
int attn_decode_noalloc(const attn_decode_params* p);

/*
 * attn_selftest_wait_timeout -- exercises the failure detection every kernel
 * carries, without a GPU fault.  (The pages have no counterpart; it exists so
 * that the device-timeout path can be tested.)  Enqueues a one-thread kernel
 * that waits on an mbarrier nothing arrives on, using the same bounded wait
 * as every pipeline stage but a limit of limit_us microseconds (1 .. 1000000);
 * when it expires the kernel records ATTN_ERR_DEVICE_TIMEOUT in the device
 * status word, exactly as a stalled pipeline would, and returns.  The context
 * stays usable; attn_get_device_status() then reports and clears the status.
 * Returns ATTN_ERR_INVALID_ARG for a limit out of range.
 */
int attn_selftest_wait_timeout(unsigned int limit_us, void* stream);

/* attn_version -- library version as major*10000 + minor*100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
