// The C ABI (include/csa.h): argument validation, workspace carving and
// kernel launches.  No allocation, no host sync except in
// csa_check_device_status (and the no-workspace entry point's one-time
// scratch lookup).
#include <cstdint>
#include <atomic>
#include <mutex>

#include "csa_device.cuh"
#include "csa_internal.h"

using namespace csa;

namespace {

// Budget of the index score's pipeline waits (csa_set_wait_budget).
std::atomic<long long> g_wait_budget{kWaitBudget};

// Device address of csa_index_score_noalloc's scratch array (end of file).
cudaError_t noalloc_scratch(void** out);

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) & ~(a - 1); }
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

csa_status_t check_cache(const csa_cache_t* c) {
  if (!c || !c->kv_pool || !c->idx_pool || !c->page_table) return CSA_ERR_INVALID_ARGUMENT;
  if (!aligned(c->kv_pool, 128) || !aligned(c->idx_pool, 128) || !aligned(c->page_table, 4))
    return CSA_ERR_INVALID_ARGUMENT;
  if (c->num_pages <= 0 || c->num_requests <= 0 || c->max_pages_per_req <= 0) return CSA_ERR_INVALID_ARGUMENT;
  if (c->pool_ratio != 1 && c->pool_ratio != 2) return CSA_ERR_INVALID_ARGUMENT;
  return CSA_OK;
}

csa_status_t check_window(const csa_window_t* w, int32_t rows_per_req) {
  if (!w) return CSA_OK;
  if (!w->e4m3 || !w->scale || !aligned(w->e4m3, 16) || !aligned(w->scale, 4)) return CSA_ERR_INVALID_ARGUMENT;
  if (w->capacity < CSA_WINDOW + (rows_per_req > 0 ? rows_per_req : 1) - 1) return CSA_ERR_INVALID_ARGUMENT;
  return CSA_OK;
}

csa_status_t check_rows(const csa_rows_t* r, const csa_cache_t* c) {
  if (!r || r->num_rows < 0) return CSA_ERR_INVALID_ARGUMENT;
  if (r->num_rows > 0 && (!r->row_req || !r->row_pos)) return CSA_ERR_INVALID_ARGUMENT;
  if (r->max_entries < 0 || r->max_rows_per_req < 1) return CSA_ERR_INVALID_ARGUMENT;
  if ((int64_t)r->max_entries > (int64_t)c->max_pages_per_req * CSA_PAGE_ENTRIES) return CSA_ERR_INVALID_ARGUMENT;
  return CSA_OK;
}

size_t scores_ld(int32_t max_entries) { return align_up((size_t)(max_entries > 0 ? max_entries : 1), 64); }

// Head count the attention workspace is sized for: the call's, or the largest.
int32_t ws_heads(int32_t n_heads) { return n_heads > 0 && n_heads <= CSA_MAX_HEADS ? n_heads : CSA_MAX_HEADS; }

struct DecodeLayout {
  size_t scores, topk, tail, end;
};
DecodeLayout decode_layout(int32_t R, int32_t max_entries, int32_t n_heads) {
  DecodeLayout L;
  L.scores = align_up(score_ws_bytes(R, CSA_MAX_IDX_HEADS));
  L.topk = align_up(L.scores + sizeof(float) * (size_t)R * scores_ld(max_entries));
  L.tail = align_up(L.topk + sizeof(int32_t) * (size_t)R * CSA_TOPK);
  L.end = align_up(L.tail + attn_tail_ws_bytes(R, ws_heads(n_heads), num_sms()));
  return L;
}

// Attention options: pointers aligned, a plan read only where no selection is
// computed, rotary tables with at least one row.
csa_status_t check_attn_opts(const csa_opts_t* o, bool plan_in_allowed) {
  if (!o) return CSA_OK;
  if (o->plan_in && (!plan_in_allowed || !aligned(o->plan_in, 4))) return CSA_ERR_INVALID_ARGUMENT;
  if (o->plan_out && !aligned(o->plan_out, 4)) return CSA_ERR_INVALID_ARGUMENT;
  if (o->plan_in && o->plan_out) return CSA_ERR_INVALID_ARGUMENT;
  if ((o->rope_cos == nullptr) != (o->rope_sin == nullptr)) return CSA_ERR_INVALID_ARGUMENT;
  if (o->rope_cos && (o->rope_rows < 1 || !aligned(o->rope_cos, 4) || !aligned(o->rope_sin, 4)))
    return CSA_ERR_INVALID_ARGUMENT;
  if (o->candidate_blocks < 0 || o->candidate_blocks > kTwoLevelMaxBlocks) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

// The attention kernel is compiled for these head counts only.
bool attn_heads_supported(int32_t H) { return H == 16 || H == 32 || H == 64; }

csa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

csa_status_t run_score(const csa_cache_t* cache, const csa_rows_t* rows, int32_t Hi, const void* q_idx,
                       const float* w, float* scores, int64_t ld, void* ws, Order prep_order,
                       cudaStream_t stream) {
  ScoreArgs a;
  a.idx_pool = cache->idx_pool;
  a.page_table = cache->page_table;
  a.num_pages = cache->num_pages;
  a.num_requests = cache->num_requests;
  a.max_pages = cache->max_pages_per_req;
  a.P = cache->pool_ratio;
  a.row_req = rows->row_req;
  a.row_pos = rows->row_pos;
  a.num_rows = rows->num_rows;
  a.Hi = Hi;
  a.group_rows = score_group_rows(Hi, rows->max_rows_per_req);   // rows of a request scored by one MMA
  a.wait_budget = g_wait_budget.load(std::memory_order_relaxed);
  a.max_entries = rows->max_entries;
  a.q_idx = static_cast<const uint16_t*>(q_idx);
  a.w = w;
  a.scores = scores;
  a.ld = ld;
  a.status = static_cast<uint32_t*>(ws);
  return from_cuda(launch_index_score(a, num_sms(), prep_order, stream));
}

// The attention's tail split for these rows (tail_splits 1: none): the bytes
// of ws from tail_off on hold its counters and partials when they fit.
AttnArgs tail_args(const csa_rows_t* rows, int32_t H, void* ws, size_t tail_off, size_t ws_bytes, int sms) {
  AttnArgs t{};
  t.num_rows = rows->num_rows;
  t.H = H;
  t.splits = attn_choose_splits(rows->num_rows, sms);
  attn_tail_setup(t, ws_bytes > tail_off ? static_cast<uint8_t*>(ws) + tail_off : nullptr,
                  ws_bytes > tail_off ? ws_bytes - tail_off : 0, sms);
  return t;
}

// Zeroes the tail split's arrival counters, if the call will split a tail;
// enqueued before the call's first kernel.  Their place in the workspace
// depends on the call's shapes, so a workspace reused with other shapes may
// hold anything there.
csa_status_t zero_tail_counters(const csa_rows_t* rows, int32_t H, void* ws, size_t tail_off, size_t ws_bytes,
                                cudaStream_t stream) {
  const AttnArgs t = tail_args(rows, H, ws, tail_off, ws_bytes, num_sms());
  if (t.tail_splits < 2) return CSA_OK;
  return from_cuda(cudaMemsetAsync(t.row_done, 0, sizeof(uint32_t) * (size_t)(t.num_rows - t.tail_row0), stream));
}

// ws_bytes: the workspace's size; the bytes from tail_off on hold the tail
// split's counters and partials when they fit (otherwise the rows run unsplit).
csa_status_t run_attn(const csa_cache_t* cache, const csa_window_t* window, const csa_rows_t* rows,
                      const int32_t* topk, int32_t H, const void* q, float softmax_scale, void* out, float* lse,
                      const csa_opts_t* opts, void* ws, size_t tail_off, size_t ws_bytes, Order order,
                      cudaStream_t stream) {
  AttnArgs a;
  a.plan_in = opts ? opts->plan_in : nullptr;
  a.plan_out = opts ? opts->plan_out : nullptr;
  const bool rope = opts && opts->rope_cos && opts->rope_sin;
  a.rope_cos = rope ? opts->rope_cos : nullptr;
  a.rope_sin = rope ? opts->rope_sin : nullptr;
  a.rope_rows = rope ? opts->rope_rows : 0;
  a.kv_pool = static_cast<const uint8_t*>(cache->kv_pool);
  a.page_table = cache->page_table;
  a.num_pages = cache->num_pages;
  a.num_requests = cache->num_requests;
  a.max_pages = cache->max_pages_per_req;
  a.P = cache->pool_ratio;
  a.win_codes = window ? window->e4m3 : nullptr;
  a.win_scale = window ? window->scale : nullptr;
  a.win_cap = window ? window->capacity : 0;
  a.row_req = rows->row_req;
  a.row_pos = rows->row_pos;
  a.num_rows = rows->num_rows;
  a.H = H;
  a.topk = topk;
  a.q = static_cast<const uint16_t*>(q);
  a.softmax_scale = softmax_scale;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.status = static_cast<uint32_t*>(ws);
  const AttnArgs t = tail_args(rows, H, ws, tail_off, ws_bytes, num_sms());
  a.splits = t.splits;
  a.tail_row0 = t.tail_row0;
  a.tail_splits = t.tail_splits;
  a.part = t.part;
  a.row_done = t.row_done;
  return from_cuda(launch_sparse_attn(a, order, stream));
}

// Validates csa_append's arguments and fills the kernel's; no launch.
csa_status_t append_args(const csa_cache_t* cache, const csa_window_t* window, const int32_t* pos0,
                         const int32_t* tok_off, int32_t total_tokens, const void* kv_in, const void* idx_in,
                         void* pending, const csa_compress_t* compress, void* ws, size_t ws_bytes,
                         AppendArgs* out) {
  csa_status_t s = check_cache(cache);
  if (s != CSA_OK) return s;
  if ((s = check_window(window, 1)) != CSA_OK) return s;
  if (total_tokens < 0 || !pos0 || !tok_off) return CSA_ERR_INVALID_ARGUMENT;
  if (total_tokens > 0 && (!kv_in || !idx_in || !aligned(kv_in, 16) || !aligned(idx_in, 16)))
    return CSA_ERR_INVALID_ARGUMENT;
  if (cache->pool_ratio == 2 && (!pending || !aligned(pending, 16))) return CSA_ERR_INVALID_ARGUMENT;
  if (ws && ws_bytes < kStatusBytes) return CSA_ERR_WORKSPACE_TOO_SMALL;
  AppendArgs a;
  a.kv_pool = static_cast<uint8_t*>(cache->kv_pool);
  a.idx_pool = static_cast<uint8_t*>(cache->idx_pool);
  a.page_table = cache->page_table;
  a.num_pages = cache->num_pages;
  a.num_requests = cache->num_requests;
  a.max_pages = cache->max_pages_per_req;
  a.P = cache->pool_ratio;
  a.win_codes = window ? window->e4m3 : nullptr;
  a.win_scale = window ? window->scale : nullptr;
  a.win_cap = window ? window->capacity : 1;
  a.pos0 = pos0;
  a.tok_off = tok_off;
  a.total_tokens = total_tokens;
  a.kv_in = static_cast<const uint16_t*>(kv_in);
  a.idx_in = static_cast<const uint16_t*>(idx_in);
  a.pending = static_cast<uint16_t*>(pending);
  a.status = static_cast<uint32_t*>(ws);
  a.kv_gamma = compress ? compress->kv_gamma : nullptr;
  a.idx_gamma = compress ? compress->idx_gamma : nullptr;
  a.eps = compress ? compress->eps : 0.0f;
  const bool rope = compress && compress->rope_cos && compress->rope_sin;
  a.rope_cos = rope ? compress->rope_cos : nullptr;
  a.rope_sin = rope ? compress->rope_sin : nullptr;
  a.rope_rows = rope ? compress->rope_rows : 0;
  if (compress) {
    if (!aligned(compress->kv_gamma, 4) || !aligned(compress->idx_gamma, 4)) return CSA_ERR_INVALID_ARGUMENT;
    if (rope && (compress->rope_rows < 0 || !aligned(compress->rope_cos, 4) || !aligned(compress->rope_sin, 4)))
      return CSA_ERR_INVALID_ARGUMENT;
    if (!(compress->eps >= 0.0f)) return CSA_ERR_INVALID_ARGUMENT;
  }
  *out = a;
  return CSA_OK;
}

csa_status_t check_decode(const csa_cache_t* cache, const csa_window_t* window, const csa_rows_t* rows,
                          int32_t n_idx_heads, const void* q_idx, const float* w, int32_t n_heads, const void* q,
                          const void* out, const void* ws, size_t ws_bytes) {
  csa_status_t s = check_cache(cache);
  if (s != CSA_OK) return s;
  if ((s = check_rows(rows, cache)) != CSA_OK) return s;
  if ((s = check_window(window, rows->max_rows_per_req)) != CSA_OK) return s;
  if (n_idx_heads < 1 || n_idx_heads > CSA_MAX_IDX_HEADS || !attn_heads_supported(n_heads))
    return CSA_ERR_UNSUPPORTED;
  if (rows->num_rows == 0) return CSA_OK;
  if (!q_idx || !w || !q || !out || !aligned(q_idx, 16) || !aligned(q, 16) || !aligned(out, 16))
    return CSA_ERR_INVALID_ARGUMENT;
  // the attention's tail-split partials (past L.tail) are used when they fit
  const DecodeLayout L = decode_layout(rows->num_rows, rows->max_entries, n_heads);
  if (!ws || ws_bytes < L.tail || !aligned(ws, 256)) return CSA_ERR_WORKSPACE_TOO_SMALL;
  return CSA_OK;
}

// index score -> top-512 -> attention, arguments already checked; `first` is
// the order of the score prep, the first of these kernels.
csa_status_t run_decode(const csa_cache_t* cache, const csa_window_t* window, const csa_rows_t* rows,
                        int32_t n_idx_heads, const void* q_idx, const float* w, int32_t n_heads, const void* q,
                        float softmax_scale, void* out, float* lse, int32_t* topk_out,
                        const csa_opts_t* opts, void* ws, size_t ws_bytes, Order first, cudaStream_t stream) {
  const DecodeLayout L = decode_layout(rows->num_rows, rows->max_entries, n_heads);
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* scores = reinterpret_cast<float*>(base + L.scores);
  int32_t* topk = topk_out ? topk_out : reinterpret_cast<int32_t*>(base + L.topk);
  const int64_t ld = (int64_t)scores_ld(rows->max_entries);
  csa_status_t s;
  if ((s = run_score(cache, rows, n_idx_heads, q_idx, w, scores, ld, ws, first, stream)) != CSA_OK) return s;
  TopkArgs t;
  t.scores = scores;
  t.ld = ld;
  t.num_rows = rows->num_rows;
  t.n_valid = nullptr;
  t.row_pos = rows->row_pos;
  t.P = cache->pool_ratio;
  t.max_n = rows->max_entries;
  t.out = topk;
  t.status = static_cast<uint32_t*>(ws);
  const int32_t blocks = opts ? opts->candidate_blocks : 0;
  if ((s = from_cuda(blocks > 0 ? launch_topk_two_level(t, blocks, Order::kChained, stream)
                                : launch_topk(t, Order::kChained, stream))) != CSA_OK)
    return s;
  return run_attn(cache, window, rows, topk, n_heads, q, softmax_scale, out, lse, opts, ws, L.tail, ws_bytes,
                  Order::kChained, stream);
}

}  // namespace

extern "C" {

size_t csa_workspace_size(int32_t op, int32_t num_rows, int32_t max_entries, int32_t n_heads) {
  if (num_rows < 0 || max_entries < 0) return 0;
  switch (op) {
    case CSA_OP_APPEND:
    case CSA_OP_TOPK:
      return kStatusBytes;
    case CSA_OP_INDEX_SCORE:
      return align_up(score_ws_bytes(num_rows, CSA_MAX_IDX_HEADS));
    case CSA_OP_SPARSE_ATTN:
      return kStatusBytes + attn_tail_ws_bytes(num_rows, ws_heads(n_heads), num_sms());
    case CSA_OP_DECODE:
      return decode_layout(num_rows, max_entries, n_heads).end;
    default:
      return 0;
  }
}

csa_status_t csa_append(const csa_cache_t* cache, const csa_window_t* window, const int32_t* pos0,
                        const int32_t* tok_off, int32_t total_tokens, const void* kv_in, const void* idx_in,
                        void* pending, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return csa_append_compress(cache, window, pos0, tok_off, total_tokens, kv_in, idx_in, pending, nullptr, ws,
                             ws_bytes, stream);
}

csa_status_t csa_append_compress(const csa_cache_t* cache, const csa_window_t* window, const int32_t* pos0,
                                 const int32_t* tok_off, int32_t total_tokens, const void* kv_in,
                                 const void* idx_in, void* pending, const csa_compress_t* compress, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  AppendArgs a;
  const csa_status_t s =
      append_args(cache, window, pos0, tok_off, total_tokens, kv_in, idx_in, pending, compress, ws, ws_bytes, &a);
  if (s != CSA_OK) return s;
  return from_cuda(launch_append(a, stream));
}

csa_status_t csa_index_score(const csa_cache_t* cache, const csa_rows_t* rows, int32_t n_idx_heads,
                             const void* q_idx, const float* w, float* scores, int32_t ld, void* ws,
                             size_t ws_bytes, cudaStream_t stream) {
  csa_status_t s = check_cache(cache);
  if (s != CSA_OK) return s;
  if ((s = check_rows(rows, cache)) != CSA_OK) return s;
  if (n_idx_heads < 1 || n_idx_heads > CSA_MAX_IDX_HEADS) return CSA_ERR_UNSUPPORTED;
  if (rows->num_rows == 0) return CSA_OK;
  if (!q_idx || !w || !scores || !aligned(q_idx, 16) || !aligned(w, 4) || !aligned(scores, 4))
    return CSA_ERR_INVALID_ARGUMENT;
  if (ld < rows->max_entries || ld < 1) return CSA_ERR_INVALID_ARGUMENT;
  if (!ws || ws_bytes < score_ws_bytes(rows->num_rows, CSA_MAX_IDX_HEADS) || !aligned(ws, 256))
    return CSA_ERR_WORKSPACE_TOO_SMALL;
  return run_score(cache, rows, n_idx_heads, q_idx, w, scores, ld, ws, Order::kStream, stream);
}

csa_status_t csa_topk(int32_t num_rows, const float* scores, int32_t ld, const int32_t* n_valid, int32_t max_n,
                      int32_t k, int32_t* out_idx, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (k != CSA_TOPK) return CSA_ERR_UNSUPPORTED;
  if (num_rows < 0 || max_n < 0 || ld < max_n || ld < 1) return CSA_ERR_INVALID_ARGUMENT;
  if (num_rows == 0) return CSA_OK;
  if (!scores || !n_valid || !out_idx || !aligned(scores, 16) || (ld % 4) != 0) return CSA_ERR_INVALID_ARGUMENT;
  if (ws && ws_bytes < kStatusBytes) return CSA_ERR_WORKSPACE_TOO_SMALL;
  TopkArgs a;
  a.scores = scores;
  a.ld = ld;
  a.num_rows = num_rows;
  a.n_valid = n_valid;
  a.row_pos = nullptr;
  a.P = 1;
  a.max_n = max_n;
  a.out = out_idx;
  a.status = static_cast<uint32_t*>(ws);
  return from_cuda(launch_topk(a, Order::kStream, stream));
}

csa_status_t csa_topk_two_level(int32_t num_rows, const float* scores, int32_t ld, const int32_t* n_valid,
                                int32_t max_n, int32_t blocks, int32_t* out_idx, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  if (blocks < 1 || blocks > kTwoLevelMaxBlocks || max_n > kTwoLevelMaxEntries) return CSA_ERR_UNSUPPORTED;
  if (num_rows < 0 || max_n < 0 || ld < max_n || ld < 1) return CSA_ERR_INVALID_ARGUMENT;
  if (num_rows == 0) return CSA_OK;
  if (!scores || !n_valid || !out_idx || !aligned(scores, 16) || (ld % 4) != 0) return CSA_ERR_INVALID_ARGUMENT;
  if (ws && ws_bytes < kStatusBytes) return CSA_ERR_WORKSPACE_TOO_SMALL;
  TopkArgs a;
  a.scores = scores;
  a.ld = ld;
  a.num_rows = num_rows;
  a.n_valid = n_valid;
  a.row_pos = nullptr;
  a.P = 1;
  a.max_n = max_n;
  a.out = out_idx;
  a.status = static_cast<uint32_t*>(ws);
  return from_cuda(launch_topk_two_level(a, blocks, Order::kStream, stream));
}

csa_status_t csa_sparse_attn(const csa_cache_t* cache, const csa_window_t* window, const csa_rows_t* rows,
                             const int32_t* topk_idx, int32_t n_heads, const void* q, float softmax_scale,
                             void* out, float* lse, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return csa_sparse_attn_ex(cache, window, rows, topk_idx, n_heads, q, softmax_scale, out, lse, nullptr, ws,
                            ws_bytes, stream);
}

csa_status_t csa_sparse_attn_ex(const csa_cache_t* cache, const csa_window_t* window, const csa_rows_t* rows,
                                const int32_t* topk_idx, int32_t n_heads, const void* q, float softmax_scale,
                                void* out, float* lse, const csa_opts_t* opts, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  csa_status_t s = check_cache(cache);
  if (s != CSA_OK) return s;
  if ((s = check_rows(rows, cache)) != CSA_OK) return s;
  if ((s = check_window(window, rows->max_rows_per_req)) != CSA_OK) return s;
  if (!attn_heads_supported(n_heads)) return CSA_ERR_UNSUPPORTED;
  if ((s = check_attn_opts(opts, true)) != CSA_OK) return s;
  if (rows->num_rows == 0) return CSA_OK;
  const bool planned = opts && opts->plan_in;
  if ((!topk_idx && !planned) || !q || !out || !aligned(q, 16) || !aligned(out, 16)) return CSA_ERR_INVALID_ARGUMENT;
  if (!ws || ws_bytes < kStatusBytes || !aligned(ws, 256)) return CSA_ERR_WORKSPACE_TOO_SMALL;
  if ((s = zero_tail_counters(rows, n_heads, ws, kStatusBytes, ws_bytes, stream)) != CSA_OK) return s;
  return run_attn(cache, window, rows, topk_idx, n_heads, q, softmax_scale, out, lse, opts, ws, kStatusBytes, ws_bytes,
                  Order::kStream,
                  stream);
}

csa_status_t csa_decode(const csa_cache_t* cache, const csa_window_t* window, const csa_rows_t* rows,
                        int32_t n_idx_heads, const void* q_idx, const float* w, int32_t n_heads, const void* q,
                        float softmax_scale, void* out, float* lse, int32_t* topk_out, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  return csa_decode_ex(cache, window, rows, n_idx_heads, q_idx, w, n_heads, q, softmax_scale, out, lse, topk_out,
                       nullptr, ws, ws_bytes, stream);
}

csa_status_t csa_decode_ex(const csa_cache_t* cache, const csa_window_t* window, const csa_rows_t* rows,
                           int32_t n_idx_heads, const void* q_idx, const float* w, int32_t n_heads, const void* q,
                           float softmax_scale, void* out, float* lse, int32_t* topk_out,
                           const csa_opts_t* opts, void* ws, size_t ws_bytes, cudaStream_t stream) {
  csa_status_t s = check_decode(cache, window, rows, n_idx_heads, q_idx, w, n_heads, q, out, ws, ws_bytes);
  if (s != CSA_OK) return s;
  if ((s = check_attn_opts(opts, false)) != CSA_OK) return s;
  if (opts && opts->candidate_blocks > 0 && rows->max_entries > kTwoLevelMaxEntries) return CSA_ERR_UNSUPPORTED;
  if (rows->num_rows == 0) return s;
  if ((s = zero_tail_counters(rows, n_heads, ws, decode_layout(rows->num_rows, rows->max_entries, n_heads).tail,
                              ws_bytes, stream)) != CSA_OK)
    return s;
  return run_decode(cache, window, rows, n_idx_heads, q_idx, w, n_heads, q, softmax_scale, out, lse, topk_out, opts,
                    ws, ws_bytes, Order::kStream, stream);
}

csa_status_t csa_step(const csa_cache_t* cache, const csa_window_t* window, const int32_t* pos0,
                      const int32_t* tok_off, int32_t total_tokens, const void* kv_in, const void* idx_in,
                      void* pending, const csa_compress_t* compress, const csa_rows_t* rows, int32_t n_idx_heads,
                      const void* q_idx, const float* w, int32_t n_heads, const void* q, float softmax_scale,
                      void* out, float* lse, int32_t* topk_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return csa_step_ex(cache, window, pos0, tok_off, total_tokens, kv_in, idx_in, pending, compress, rows,
                     n_idx_heads, q_idx, w, n_heads, q, softmax_scale, out, lse, topk_out, nullptr, ws, ws_bytes,
                     stream);
}

csa_status_t csa_step_ex(const csa_cache_t* cache, const csa_window_t* window, const int32_t* pos0,
                         const int32_t* tok_off, int32_t total_tokens, const void* kv_in, const void* idx_in,
                         void* pending, const csa_compress_t* compress, const csa_rows_t* rows,
                         int32_t n_idx_heads, const void* q_idx, const float* w, int32_t n_heads, const void* q,
                         float softmax_scale, void* out, float* lse, int32_t* topk_out,
                         const csa_opts_t* opts, void* ws, size_t ws_bytes, cudaStream_t stream) {
  AppendArgs a;
  csa_status_t s =
      append_args(cache, window, pos0, tok_off, total_tokens, kv_in, idx_in, pending, compress, ws, ws_bytes, &a);
  if (s != CSA_OK) return s;
  if ((s = check_decode(cache, window, rows, n_idx_heads, q_idx, w, n_heads, q, out, ws, ws_bytes)) != CSA_OK)
    return s;
  if ((s = check_attn_opts(opts, false)) != CSA_OK) return s;
  if (opts && opts->candidate_blocks > 0 && rows->max_entries > kTwoLevelMaxEntries) return CSA_ERR_UNSUPPORTED;
  if (rows->num_rows > 0 &&
      (s = zero_tail_counters(rows, n_heads, ws, decode_layout(rows->num_rows, rows->max_entries, n_heads).tail,
                              ws_bytes, stream)) != CSA_OK)
    return s;
  if ((s = from_cuda(launch_append(a, stream))) != CSA_OK) return s;
  if (rows->num_rows == 0) return CSA_OK;
  // With an append kernel in flight, the score prep is chained to it: it reads
  // only the step's inputs and the score workspace, which the append does not
  // touch, and it waits for the append before it exits.  Without one it is the
  // call's first kernel.
  return run_decode(cache, window, rows, n_idx_heads, q_idx, w, n_heads, q, softmax_scale, out, lse, topk_out, opts,
                    ws, ws_bytes, total_tokens > 0 ? Order::kChained : Order::kStream, stream);
}

csa_status_t csa_check_device_status(void* ws, cudaStream_t stream, uint32_t* flags_out) {
  if (!flags_out) return CSA_ERR_INVALID_ARGUMENT;
  if (!ws && noalloc_scratch(&ws) != cudaSuccess) return CSA_ERR_CUDA;   // the fixed scratch array's word
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CSA_ERR_CUDA;
  uint32_t f = 0;
  if (cudaMemcpy(&f, ws, sizeof(f), cudaMemcpyDeviceToHost) != cudaSuccess) return CSA_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(f), stream) != cudaSuccess) return CSA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CSA_ERR_CUDA;
  *flags_out = f;
  if (f & CSA_FLAG_TIMEOUT) return CSA_ERR_TIMEOUT;
  return f ? CSA_ERR_DEVICE_FAULT : CSA_OK;
}

csa_status_t csa_set_wait_budget(int64_t sm_clocks) {
  g_wait_budget.store(sm_clocks > 0 ? (long long)sm_clocks : kWaitBudget, std::memory_order_relaxed);
  return CSA_OK;
}

const char* csa_status_string(csa_status_t s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported shape";
    case CSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case CSA_ERR_CUDA: return "CUDA launch or runtime error";
    case CSA_ERR_DEVICE_FAULT: return "device-detected fault (see status flags)";
    case CSA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"

// ---------------------------------------------------------------------------
// csa_index_score_noalloc: the index score with its scratch in a fixed device
// array owned by this library, for callers that cannot allocate (see csa.h).
namespace {

constexpr size_t kNoAllocScratchBytes = CSA_NOALLOC_SCRATCH_BYTES;
// One copy per GPU that loads the library, alive until the process exits.
// Host code must not use this name as an address: the device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up with
// that device current on its first successful call and kept from then on.  A
// lookup that fails (for example inside a stream capture) is not remembered:
// the next call tries again.
cudaError_t noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return e;
      }
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" csa_status_t csa_index_score_noalloc(const csa_cache_t* cache, const csa_rows_t* rows,
                                                int32_t n_idx_heads, const void* q_idx, const float* w,
                                                float* scores, int32_t ld, cudaStream_t stream) {
  csa_status_t s = check_cache(cache);
  if (s != CSA_OK) return s;
  if ((s = check_rows(rows, cache)) != CSA_OK) return s;
  if (n_idx_heads < 1 || n_idx_heads > CSA_MAX_IDX_HEADS) return CSA_ERR_UNSUPPORTED;
  if (rows->num_rows == 0) return CSA_OK;
  if (!q_idx || !w || !scores || !aligned(q_idx, 16) || !aligned(w, 4) || !aligned(scores, 4))
    return CSA_ERR_INVALID_ARGUMENT;
  if (ld < rows->max_entries || ld < 1) return CSA_ERR_INVALID_ARGUMENT;
  if (score_ws_bytes(rows->num_rows, n_idx_heads) > kNoAllocScratchBytes) return CSA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  if (noalloc_scratch(&ws) != cudaSuccess) return CSA_ERR_CUDA;
  // every call starts with a clear status word; the rest of the scratch is
  // fully rewritten by the score step before it is read
  if (cudaMemsetAsync(ws, 0, kStatusBytes, stream) != cudaSuccess) return CSA_ERR_CUDA;
  return run_score(cache, rows, n_idx_heads, q_idx, w, scores, ld, ws, Order::kStream, stream);
}
