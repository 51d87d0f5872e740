/*
 * csa.h -- C ABI of the compressed-sparse-attention (CSA) decode hot path for
 * GB300 (sm_103a): FP4 paged cache append, FP4 indexer score, exact top-512,
 * and sparse MQA attention over the selected FP4 entries plus an FP8 window.
 *
 * Sources (web pages, cited by title and section):
 *  [SGL]  "DeepSeek-V4.1 Flash on SGLang: from 35 to 873 tokens/s"
 *         - "Architecture changes and KV cache compression": global KV caches
 *           store FP4 entries of 288 B (main KV) and 68 B (indexer K); three
 *           caches pool every two tokens into one entry, one keeps one entry
 *           per token; only the top 512 global positions take part in
 *           attention; 890 B per token is the logical size and the allocated
 *           layout may differ.
 *         - "Small-operator fusion and GEMV": pooling, FP4 quantisation and the
 *           cache write are fused; per-step request indices are built once and
 *           shared across layers.
 *         - "DSpark adaptation and optimization": up to 6 verify rows per
 *           request; the valid-length check is fused with candidate handling;
 *           post-top-k score check, invalid-position filtering and KV page
 *           address translation are one step; pair pooling, quantisation and
 *           the main-KV write are one kernel, the first row reading the saved
 *           previous token.
 *  [VLLM] "DeepSeek-V4.1-Flash runs 5.3x faster on vLLM after three weeks of
 *         optimization" - "SWA bounded replay...": the local window is
 *         uncompressed FP8 over the most recent 128 positions; "CUDA graphs and
 *         the new kernels": decode steps are captured in CUDA graphs.
 *
 * FORMAT (this library's byte layout; the pages fix only the entry sizes)
 *  - e2m1 codes: bit 3 sign, magnitude 0..7 = {0,.5,1,1.5,2,3,4,6}; element
 *    2j in the low nibble of byte j.  E4M3 = OCP FP8 "fn" (max 448);
 *    E8M0 = 2^(code-127).
 *  - Main-KV entry (288 B): 512 e2m1 + one E4M3 scale per 16 values (NVFP4:
 *    s = E4M3(amax/6), codes = RNE(x/s)).
 *  - Indexer-K entry (68 B): 128 e2m1 + one E8M0 scale per 32 values (MXFP4,
 *    OCP MX rule: scale 2^(floor(log2 amax) - 2)).
 *  - Pages of 64 entries:
 *      main-KV page 18432 B: entry e data at 256*e, scales at 16384 + 32*e
 *      indexer page  4352 B: 8 groups of 544 B, group g = entries 8g..8g+7;
 *        data byte k (0..63) of entry 8g+r at 544*g + 128*(k/16) + 16*r + k%16
 *        (16-byte core matrices of 8 entries, the tensor-core operand order),
 *        scale byte b (0..3) of entry 8g+r at 544*g + 512 + 4*r + b.
 *    A whole indexer page is therefore one contiguous copy that lands in
 *    shared memory as an MMA operand (8-entry groups 544 B apart).
 *    page_table[b*max_pages_per_req + j] = physical page of request b's j-th
 *    logical page; the same id indexes both pools.
 *  - Entry e of a request pools tokens P*e .. P*e+P-1 (P = pool_ratio, 2 or 1):
 *    x = (t0 + t1) * 0.5 in fp32.  A row at position t sees entries
 *    e < floor((t+1)/P) and window positions max(0,t-127)..t.
 *  - FP8 window ring: token at position p of request b lives in slot
 *    b*capacity + p % capacity: 512 E4M3 codes + one fp32 scale (amax/448).
 *
 * CONVENTIONS
 *  - All pointers are device pointers unless marked "host".  The caller owns
 *    and frees every buffer; the library never allocates, frees or
 *    synchronises (except csa_check_device_status).  All work is enqueued on
 *    `stream`, so calls can be captured in a CUDA graph.
 *  - bf16 tensors are passed as void* (IEEE bfloat16 bit patterns).
 *  - Pools, pages, q, out and the window must be 16-byte aligned; the pools
 *    128-byte aligned.
 *  - Host-detectable errors return before any launch.  Faults only the device
 *    can see (page id out of range, a row seeing more entries than its pages
 *    hold, rows not grouped by request, a top-k index outside the row's
 *    visible range, a bounded wait that ran out) never trap: the unit is
 *    skipped (outputs zero / -1) and a flag is OR-ed into the status word at
 *    the head of the workspace; read it with csa_check_device_status().
 *  - Calls that run concurrently need distinct workspaces.
 *  - Stream order: a call's first kernel is an ordinary launch, so it starts
 *    after all work enqueued before it on `stream` has completed; inputs may
 *    come from any earlier work on the stream.  The later kernels of the same
 *    call (csa_index_score, csa_decode, csa_step) use programmatic dependent
 *    launch: each may start while the call's previous kernel finishes and
 *    waits for it before reading anything that kernel wrote.
 */
#ifndef CSA_H
#define CSA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CSA_API __attribute__((visibility("default")))
#else
#define CSA_API
#endif

#define CSA_D                 512   /* main latent width                        */
#define CSA_DI                128   /* indexer key width                        */
#define CSA_TOPK              512   /* selected global positions per row        */
#define CSA_WINDOW            128   /* FP8 window positions per row             */
#define CSA_PAGE_ENTRIES      64
#define CSA_KV_ENTRY_BYTES    288
#define CSA_IDX_ENTRY_BYTES   68
#define CSA_KV_PAGE_BYTES     18432
#define CSA_IDX_PAGE_BYTES    4352
#define CSA_MAX_HEADS         64    /* attention heads per row: 16, 32 or 64;
                                       other counts return CSA_ERR_UNSUPPORTED  */
#define CSA_MAX_IDX_HEADS     128   /* indexer heads per row                    */
#define CSA_MAX_ROW_GROUP_COLS 128  /* rows-per-request x indexer heads scored
                                       together; larger groups are split        */

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARGUMENT = 1,    /* NULL / misaligned pointer, bad size       */
  CSA_ERR_UNSUPPORTED = 2,         /* shape outside the compiled limits         */
  CSA_ERR_WORKSPACE_TOO_SMALL = 3,
  CSA_ERR_CUDA = 4,                /* a launch or runtime call failed           */
  CSA_ERR_DEVICE_FAULT = 5,        /* device status word has a fault flag       */
  CSA_ERR_TIMEOUT = 6              /* device status word has the timeout flag   */
} csa_status_t;

/* Device status flags (csa_check_device_status). */
#define CSA_FLAG_PAGE_OOB    0x1u   /* page id or logical page out of range     */
#define CSA_FLAG_ROW_INVALID 0x2u   /* bad row_req / rows not grouped / n > cap  */
#define CSA_FLAG_TOPK_OOB    0x4u   /* selected index outside the visible range */
#define CSA_FLAG_TIMEOUT     0x8u   /* a bounded device wait ran out             */
#define CSA_FLAG_APPEND      0x10u  /* token offsets inconsistent with total    */

/* Paged FP4 cache (caller-owned device memory). */
typedef struct {
  void*          kv_pool;          /* num_pages * 18432 B, 128-B aligned          */
  void*          idx_pool;         /* num_pages *  4352 B, 128-B aligned          */
  const int32_t* page_table;       /* [num_requests, max_pages_per_req]           */
  int32_t        num_pages;
  int32_t        num_requests;
  int32_t        max_pages_per_req;
  int32_t        pool_ratio;       /* 2 (pair pooled) or 1 (one entry per token)  */
} csa_cache_t;

/* FP8 local window ring. */
typedef struct {
  uint8_t* e4m3;                   /* [num_requests, capacity, 512]               */
  float*   scale;                  /* [num_requests, capacity]                    */
  int32_t  capacity;               /* >= 128 + (rows per request) - 1             */
} csa_window_t;

/* Query rows of one decode step, built once per step and shared by every
 * layer that reads the same cache ([SGL] "Small-operator fusion and GEMV"). */
typedef struct {
  int32_t        num_rows;         /* R                                           */
  const int32_t* row_req;          /* [R] request of each row, non-decreasing      */
  const int32_t* row_pos;          /* [R] token position of each row              */
  int32_t        max_entries;      /* host bound: max over rows of (pos+1)/P      */
  int32_t        max_rows_per_req; /* host bound on rows sharing one request      */
} csa_rows_t;

/* Workspace sizing: op = one of the CSA_OP_* values; bytes for num_rows rows
 * of at most max_entries entries each and n_heads attention heads.  For
 * CSA_OP_SPARSE_ATTN and CSA_OP_DECODE the size also depends on the current
 * device's SM count: with more rows than SMs, the rows of the last wave of one
 * CTA per SM are split over several CTAs that merge through the workspace
 * (see csa_sparse_attn); a workspace without that room (at least the size
 * computed for a device with num_rows or more SMs) runs every row whole.
 * A workspace is zero-filled before its first use (its status word starts at
 * zero); the tail split's arrival counters are zeroed by each call that uses
 * them, so a workspace can serve calls of different shapes.  0 = bad op. */
enum { CSA_OP_APPEND = 0, CSA_OP_INDEX_SCORE = 1, CSA_OP_TOPK = 2,
       CSA_OP_SPARSE_ATTN = 3, CSA_OP_DECODE = 4 };
CSA_API size_t csa_workspace_size(int32_t op, int32_t num_rows, int32_t max_entries, int32_t n_heads);

/* csa_append -- pool, quantise and write new tokens ([SGL] "DSpark adaptation
 * and optimization": fused pair pooling + quantisation + main-KV write, reused
 * for index-K; [SGL] "Architecture changes...": 2:1 pooling or 1:1).
 *  pos0      [B]   position of each request's first new token
 *  tok_off   [B+1] request b's new tokens are rows tok_off[b]..tok_off[b+1]-1
 *  total_tokens    host copy of tok_off[B] (grid size)
 *  kv_in     bf16 [total_tokens, 512]; idx_in bf16 [total_tokens, 128]
 *  pending   bf16 [B, 640] in/out: the unpaired last token of each request
 *            (512 latent then 128 key).  Read when pos0 is odd (P = 2),
 *            written when the last new token is left unpaired.
 *  window    nullable; when given, the new tokens are also written to the FP8
 *            ring (of a call's tokens for one request only the last `capacity`
 *            land there, which is the ring's content after the call).
 *  Entries are complete when their last token arrives; a row must only see
 *  complete entries.  ws may be NULL (ws_bytes 0): faults are then not
 *  reported. */
CSA_API csa_status_t csa_append(const csa_cache_t* cache, const csa_window_t* window,
                        const int32_t* pos0, const int32_t* tok_off, int32_t total_tokens,
                        const void* kv_in, const void* idx_in, void* pending,
                        void* ws, size_t ws_bytes, cudaStream_t stream);

/* csa_index_score -- score[r,i] = sum_h w[r,h] * relu(qhat[r,h] . khat[i]) for
 * i < n(r), with qhat = MXFP4(q_idx) and khat the cached MXFP4 indexer keys,
 * as a block-scaled FP4 tensor-core product ([SGL] "Architecture changes...":
 * the indexer decides which 512 global positions attend).
 *  q_idx bf16 [R, Hi, 128]; w fp32 [R, Hi]; scores fp32 [R, ld], ld >= max_entries,
 *  entries i >= n(r) are left untouched.  Hi <= 128. */
CSA_API csa_status_t csa_index_score(const csa_cache_t* cache, const csa_rows_t* rows,
                             int32_t n_idx_heads, const void* q_idx, const float* w,
                             float* scores, int32_t ld, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* csa_topk -- exact top-512 of scores[r, 0..n_valid[r]) by (score desc, index
 * asc), written in ascending index order and padded with -1 ([SGL]
 * "Architecture changes...": top 512 global positions; "DSpark adaptation and
 * optimization": invalid-position filtering).  k must be 512. max_n is a host
 * bound on n_valid.  -0.0 and +0.0 compare equal; NaN scores are unsupported. */
CSA_API csa_status_t csa_topk(int32_t num_rows, const float* scores, int32_t ld,
                      const int32_t* n_valid, int32_t max_n, int32_t k, int32_t* out_idx,
                      void* ws, size_t ws_bytes, cudaStream_t stream);

/* csa_sparse_attn -- for each row and head: softmax attention of q over the
 * dequantised FP4 main-KV entries listed in topk_idx (ascending, -1 skipped;
 * page translation done here, [SGL] "DSpark adaptation and optimization") and
 * the FP8 window positions max(0,t-127)..t ([VLLM] "SWA bounded replay").
 * K = V = the shared 512-d latent (MQA).  With fewer rows than SMs a row is
 * split over key blocks; its CTAs form one thread-block cluster and merge by
 * log-sum-exp in shared memory.  With more rows than SMs, when the last wave
 * of one CTA per SM holds at most half the SMs' worth of rows, each of those
 * rows is split over up to five CTAs that leave their partials in ws and the
 * row's last CTA to finish merges them (same weights).  ws:
 * csa_workspace_size(CSA_OP_SPARSE_ATTN, R, max_entries, n_heads) bytes,
 * 256-byte aligned, at least 256.
 *  q bf16 [R, H, 512]; out bf16 [R, H, 512]; lse fp32 [R, H] (nullable). */
CSA_API csa_status_t csa_sparse_attn(const csa_cache_t* cache, const csa_window_t* window,
                             const csa_rows_t* rows, const int32_t* topk_idx,
                             int32_t n_heads, const void* q, float softmax_scale,
                             void* out, float* lse, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* csa_decode -- one decode step of one CSA layer for every query row: the
 * indexer scores every visible entry, the exact top 512 are kept, and the
 * rows attend to those entries plus their FP8 window ([SGL] "Architecture
 * changes and KV cache compression": the indexer selects the top 512 global
 * positions that take part in attention; "DSpark adaptation and
 * optimization": the post-top-k filter and page translation in one step;
 * [VLLM] "SWA bounded replay": the 128-position FP8 window).  Arguments are
 * those of csa_index_score and csa_sparse_attn; everything is enqueued on
 * `stream` (csa_index_score -> csa_topk -> csa_sparse_attn).
 *  topk_out [R, 512] (nullable): the selected indices, ascending, -1 padded.
 *  ws: csa_workspace_size(CSA_OP_DECODE, R, max_entries, n_heads) bytes,
 *  256-byte aligned.  n_heads must be 16, 32 or 64 and n_idx_heads 1..128;
 *  every argument is checked before the first launch. */
CSA_API csa_status_t csa_decode(const csa_cache_t* cache, const csa_window_t* window,
                        const csa_rows_t* rows, int32_t n_idx_heads, const void* q_idx,
                        const float* w, int32_t n_heads, const void* q, float softmax_scale,
                        void* out, float* lse, int32_t* topk_out,
                        void* ws, size_t ws_bytes, cudaStream_t stream);

/* Options of the selection and attention steps (csa_sparse_attn_ex,
 * csa_decode_ex, csa_step_ex); NULL = none of them.
 *  candidate_blocks  0: the exact top-512 over every visible entry.  B in
 *            [1, 128] (csa_decode_ex / csa_step_ex): the two-level candidate
 *            filter of csa_topk_two_level instead ([SGL] "Architecture changes
 *            and KV cache compression": CSA2 narrows the indexer's search).
 *  plan_out  [R, 512] int32 (nullable): the resolved cache entry of every
 *            selected index, page * 64 + slot (-1: none), as the attention
 *            step looked it up -- the plan that further layers reading the
 *            same cache reuse ([SGL] "Small-operator fusion and GEMV": per-step
 *            indices built once and shared across layers).
 *  plan_in   [R, 512] int32 (nullable; csa_sparse_attn_ex only, then topk_idx
 *            may be NULL): a plan written by an earlier call for the same rows
 *            and cache, read instead of topk_idx: no page-table lookup.  Its
 *            entries are trusted apart from the pool bound (page >= num_pages
 *            raises CSA_FLAG_PAGE_OOB and the entry is skipped).
 *  rope_cos, rope_sin  [rope_rows, 32] fp32 (both or neither): the query's last
 *            64 dims are rotated with table row t (the row's position) and each
 *            window token's with row p (its position), as key and as value,
 *            by the rotate-half rule of csa_append_compress; global entries are
 *            used as stored (rotated when appended) ([SGL] "DSpark adaptation
 *            and optimization": Q RoPE merged into the attention-buffer write).
 *            A row with t >= rope_rows raises CSA_FLAG_ROW_INVALID and gets a
 *            zero output and lse -inf. */
typedef struct {
  const int32_t* plan_in;
  int32_t*       plan_out;
  const float*   rope_cos;
  const float*   rope_sin;
  int32_t        rope_rows;
  int32_t        candidate_blocks;
} csa_opts_t;

/* csa_topk_two_level -- the two-level candidate filter (NEXT f-2), a variant of
 * csa_topk, not its replacement ([SGL] "Architecture changes and KV cache
 * compression": CSA2 narrows the indexer's search before the top 512;
 * "DSpark adaptation and optimization": chosen candidate blocks expand
 * straight into a token mask).  The pages give no block size or block score;
 * this library's reading: a block is 64 consecutive entries (a page),
 * scored by its largest score; the first `blocks` blocks by (block score
 * descending, block index ascending) are kept; the exact top-512 among their
 * entries by (score descending, index ascending) is written in ascending
 * order, padded with -1.  With blocks >= ceil(n/64) or blocks >= 512 the
 * result equals csa_topk's.  blocks in [1, 128] (CSA_ERR_UNSUPPORTED
 * otherwise); max_n <= 262144; scores 16-byte aligned, ld a multiple of 4.
 * Other arguments as csa_topk. */
CSA_API csa_status_t csa_topk_two_level(int32_t num_rows, const float* scores, int32_t ld,
                                        const int32_t* n_valid, int32_t max_n, int32_t blocks,
                                        int32_t* out_idx, void* ws, size_t ws_bytes, cudaStream_t stream);

/* csa_sparse_attn with options; arguments and errors otherwise as
 * csa_sparse_attn.  CSA_ERR_INVALID_ARGUMENT for a misaligned option pointer,
 * one rotary table without the other, rope_rows < 1, or both plan_in and
 * plan_out. */
CSA_API csa_status_t csa_sparse_attn_ex(const csa_cache_t* cache, const csa_window_t* window,
                                        const csa_rows_t* rows, const int32_t* topk_idx,
                                        int32_t n_heads, const void* q, float softmax_scale,
                                        void* out, float* lse, const csa_opts_t* opts,
                                        void* ws, size_t ws_bytes, cudaStream_t stream);

/* csa_decode with options for its attention step (plan_in not allowed: the
 * decode makes its own selection; plan_out receives that selection resolved). */
CSA_API csa_status_t csa_decode_ex(const csa_cache_t* cache, const csa_window_t* window,
                                   const csa_rows_t* rows, int32_t n_idx_heads, const void* q_idx,
                                   const float* w, int32_t n_heads, const void* q, float softmax_scale,
                                   void* out, float* lse, int32_t* topk_out, const csa_opts_t* opts,
                                   void* ws, size_t ws_bytes, cudaStream_t stream);

/* csa_index_score_noalloc -- the same scores as csa_index_score, without a
 * workspace argument.  The pages have no counterpart to this entry point; it
 * exists for callers that cannot call cudaMalloc: a serving loop that reserves
 * all of its device memory at start-up and may not allocate while it decodes
 * (an allocation can synchronise the device and stall the other streams), or
 * a plain C host that embeds this library and has no device allocator of its
 * own.  Its scratch is a fixed array of CSA_NOALLOC_SCRATCH_BYTES inside this
 * library, present on every GPU that loads the library until the process
 * exits; nothing is allocated or freed.
 *  - The first call on each device looks up the array's device address with
 *    that device current; make that first call before any stream capture.  A
 *    lookup that fails returns CSA_ERR_CUDA and is tried again next call.
 *  - Every call shares the one array and leaves its contents behind (the
 *    status word is cleared at the start of each call, the rest is rewritten
 *    before it is read).  Calls that overlap on the GPU -- other streams, or
 *    other host threads without ordering between them -- race on the array.
 *  - Scratch need is about num_rows x 8*ceil(n_idx_heads/8) x 68 B; a call
 *    that needs more than the array returns CSA_ERR_WORKSPACE_TOO_SMALL before
 *    any launch.  Device-detected faults land in the array's status word:
 *    csa_check_device_status(NULL, stream, &flags) reads and clears it.
 *  Arguments are those of csa_index_score without ws / ws_bytes. */
#define CSA_NOALLOC_SCRATCH_BYTES (4u << 20)
CSA_API csa_status_t csa_index_score_noalloc(const csa_cache_t* cache, const csa_rows_t* rows,
                                             int32_t n_idx_heads, const void* q_idx, const float* w,
                                             float* scores, int32_t ld, cudaStream_t stream);

/* csa_append_compress -- csa_append with the compressor's normalisation and
 * rotary steps applied to every new pooled entry (main latent and indexer
 * key) after pooling and before quantisation ([SGL] "DSpark adaptation and
 * optimization": pair pooling, RMSNorm, RoPE, quantisation and the main-KV
 * write fused in one kernel, reused for index-K).  The pages give neither the
 * weights nor a rotary convention; this library's reading:
 *  - RMSNorm: v_i = (v_i * r) * gamma_i, r = 1 / sqrt(ss / dim + eps), every
 *    step rounded to fp32 (no fused multiply-add); ss = sum of squares taken
 *    as 32 contiguous parts of dim/32 values summed left to right, the part
 *    sums then combined pairwise at distance 16, 8, 4, 2, 1.
 *  - RoPE: rotate-half on the last 64 dims of each vector: for j < 32,
 *    a = v[dim-64+j], b = v[dim-32+j]: a' = a*c_j - b*s_j, b' = b*c_j + a*s_j,
 *    with (c, s) = rope_cos/rope_sin row p, p = the position of the entry's
 *    last token (p = P*e + P - 1 for entry e).
 *  - The FP8 window tokens and the pending token stay raw (unnormalised).
 * compress (host pointer, required): any of its device pointers may be NULL
 * to skip that step.  kv_gamma fp32 [512], idx_gamma fp32 [128]; rope_cos /
 * rope_sin fp32 [rope_rows, 32], 4-byte aligned.  An entry whose position is
 * >= rope_rows is not written and raises CSA_FLAG_APPEND.  Other arguments,
 * layouts and errors as csa_append. */
typedef struct {
  const float* kv_gamma;
  const float* idx_gamma;
  float        eps;
  const float* rope_cos;
  const float* rope_sin;
  int32_t      rope_rows;
} csa_compress_t;

CSA_API csa_status_t csa_append_compress(const csa_cache_t* cache, const csa_window_t* window,
                                         const int32_t* pos0, const int32_t* tok_off, int32_t total_tokens,
                                         const void* kv_in, const void* idx_in, void* pending,
                                         const csa_compress_t* compress, void* ws, size_t ws_bytes,
                                         cudaStream_t stream);

/* csa_step -- one decode step of a layer in one call: csa_append_compress of
 * the step's new tokens (compress nullable: plain csa_append), then
 * csa_decode of its query rows, on `stream`.  Arguments and results are those
 * of the two calls made back to back, except that ws is csa_decode's
 * workspace and also takes the append's device-side faults.  In one call the
 * score step's preparation (indexer-q quantisation, segment table) runs beside
 * the append kernel: it reads only the step's inputs and writes only the score
 * workspace, which the append does not touch.  ([SGL] "Small-operator fusion
 * and GEMV": a decode step is a chain of short kernels; "mHC: reduction fusion
 * and overlap": the compressor's and the indexer's work overlapped.)
 * All arguments are checked before the first launch. */
CSA_API csa_status_t csa_step(const csa_cache_t* cache, const csa_window_t* window,
                      const int32_t* pos0, const int32_t* tok_off, int32_t total_tokens,
                      const void* kv_in, const void* idx_in, void* pending,
                      const csa_compress_t* compress, const csa_rows_t* rows,
                      int32_t n_idx_heads, const void* q_idx, const float* w,
                      int32_t n_heads, const void* q, float softmax_scale,
                      void* out, float* lse, int32_t* topk_out,
                      void* ws, size_t ws_bytes, cudaStream_t stream);

/* csa_step with options for its attention step (as csa_decode_ex).  With the
 * compressor's rotary tables passed again in opts, the keys rotated at append,
 * the query and the window tokens share one rotation. */
CSA_API csa_status_t csa_step_ex(const csa_cache_t* cache, const csa_window_t* window,
                                 const int32_t* pos0, const int32_t* tok_off, int32_t total_tokens,
                                 const void* kv_in, const void* idx_in, void* pending,
                                 const csa_compress_t* compress, const csa_rows_t* rows,
                                 int32_t n_idx_heads, const void* q_idx, const float* w,
                                 int32_t n_heads, const void* q, float softmax_scale,
                                 void* out, float* lse, int32_t* topk_out, const csa_opts_t* opts,
                                 void* ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronises `stream`, returns the status word's flags in *flags_out (host)
 * and clears it.  Returns CSA_OK, CSA_ERR_TIMEOUT or CSA_ERR_DEVICE_FAULT.
 * ws == NULL reads the status word of csa_index_score_noalloc's fixed scratch
 * array on the current device. */
CSA_API csa_status_t csa_check_device_status(void* ws, cudaStream_t stream, uint32_t* flags_out);

/* csa_set_wait_budget -- failure detection (no counterpart in the pages).
 * Every wait of the index score's pipeline (a copy landing, an MMA
 * completing, a buffer coming free) is bounded by this many SM clocks; a wait
 * that runs out stops the kernel, which raises CSA_FLAG_TIMEOUT in the status
 * word, waits for the copies and tensor-core work it already issued, frees
 * its tensor memory and returns.  Process-wide; takes effect at the next
 * call's launch.  sm_clocks <= 0 restores the default (3e9 clocks, about 1.5
 * s).  A small budget is a way to exercise the time-out path without a
 * fault; scores are incomplete after a time-out. */
CSA_API csa_status_t csa_set_wait_budget(int64_t sm_clocks);

CSA_API const char* csa_status_string(csa_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H */
