// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/csa.h"

namespace csa {

// How a kernel is ordered after the work before it in its stream.
//  kStream   plain stream order: the kernel starts once everything enqueued
//            before it has completed.  The first kernel of every public call
//            is launched so; from then on the call's inputs are complete and
//            no earlier call still reads the workspace.
//  kChained  programmatic dependent launch, for the later kernels of a call:
//            the kernel may start while the previous kernel of the same call is
//            still running; it runs its prologue (and may read the call's
//            inputs), then griddepcontrol.wait (pdl_wait) blocks until that
//            kernel has completed and its memory is visible, before anything
//            it produced is read.  (griddepcontrol.wait returns at once in a
//            kStream launch.)
enum class Order { kStream, kChained };

// Adds the launch attribute for `order` at attr[0]; returns how many it added.
inline unsigned order_attr(Order order, cudaLaunchAttribute* attr) {
  if (order != Order::kChained) return 0;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  return 1;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(Order order, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = order_attr(order, attr);
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

struct AppendArgs {
  uint8_t* kv_pool;
  uint8_t* idx_pool;
  const int32_t* page_table;
  int32_t num_pages, num_requests, max_pages, P;
  uint8_t* win_codes;
  float* win_scale;
  int32_t win_cap;
  const int32_t* pos0;
  const int32_t* tok_off;
  int32_t total_tokens;
  const uint16_t* kv_in;
  const uint16_t* idx_in;
  uint16_t* pending;
  uint32_t* status;
  // compressor steps (NULL: skipped); see csa_append_compress
  const float* kv_gamma;
  const float* idx_gamma;
  float eps;
  const float* rope_cos;
  const float* rope_sin;
  int32_t rope_rows;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);

// Indexer score: k_score_prep + the persistent tcgen05 score kernel.
struct ScoreArgs {
  const void* idx_pool;
  const int32_t* page_table;
  int32_t num_pages, num_requests, max_pages, P;
  const int32_t* row_req;
  const int32_t* row_pos;
  int32_t num_rows, Hi, group_rows;   // rows scored together per MMA
  int32_t max_entries;                 // host bound on entries per row
  const uint16_t* q_idx;               // bf16 [R, Hi, 128]
  const float* w;                      // [R, Hi]
  float* scores;                       // [R, ld]
  int64_t ld;
  uint32_t* status;                    // head of the workspace
  int32_t grid;                        // score CTAs (set by the launcher)
  long long wait_budget;               // SM clocks a pipeline wait may take
};
// prep_order: the score prep's order (kStream when it is its call's first kernel)
cudaError_t launch_index_score(const ScoreArgs& a, int num_sms, Order prep_order, cudaStream_t stream);
size_t score_ws_bytes(int32_t R, int32_t Hi);
int score_group_rows(int32_t Hi, int32_t max_rows_per_req);

struct TopkArgs {
  const float* scores;
  int64_t ld;
  int32_t num_rows;
  const int32_t* n_valid;  // [R] or null (then n(r) comes from row_pos / P)
  const int32_t* row_pos;
  int32_t P;
  int32_t max_n;
  int32_t* out;            // [R, 512]
  uint32_t* status;
};
cudaError_t launch_topk(const TopkArgs& a, Order order, cudaStream_t stream);
// Two-level candidate filter: blocks in [1, 128], rows up to 262144 entries.
cudaError_t launch_topk_two_level(const TopkArgs& a, int32_t blocks, Order order, cudaStream_t stream);
constexpr int32_t kTwoLevelMaxBlocks = 128;
constexpr int32_t kTwoLevelMaxEntries = 262144;

struct AttnArgs {
  const uint8_t* kv_pool;
  const int32_t* page_table;
  int32_t num_pages, num_requests, max_pages, P;
  const uint8_t* win_codes;
  const float* win_scale;
  int32_t win_cap;
  const int32_t* row_req;
  const int32_t* row_pos;
  int32_t num_rows, H;
  const int32_t* topk;      // [R, 512]
  const uint16_t* q;        // bf16 [R, H, 512]
  float softmax_scale;
  uint16_t* out;            // bf16 [R, H, 512]
  float* lse;               // [R, H] or null
  int32_t splits;
  uint32_t* status;
  const int32_t* plan_in;   // [R, 512] resolved entries (page * 64 + slot, -1 none) read instead of topk
  int32_t* plan_out;        // [R, 512] or null: the resolved entries written here
  const float* rope_cos;    // [rope_rows, 32] or null: query and window tokens rotated
  const float* rope_sin;
  int32_t rope_rows;
  // Tail split (splits == 1 only): rows from tail_row0 on take tail_splits CTAs
  // each and merge through the workspace; tail_splits == 1: none.
  int32_t tail_row0, tail_splits;
  float* part;              // [tail CTAs][H][512] unnormalised O, then [tail CTAs][2][H] (m, l)
  uint32_t* row_done;       // [num_rows - tail_row0] CTAs of a tail row that finished; zeroed by the call
};
cudaError_t launch_sparse_attn(const AttnArgs& a, Order order, cudaStream_t stream);
int32_t attn_choose_splits(int32_t num_rows, int num_sms);
// The last wave's rows when the rows fill more than one wave of one CTA per SM
// and the last wave at most half: they are split into tail_splits CTAs each.
// Returns tail_splits (1: no tail split) and sets *tail_row0.
int32_t attn_tail_plan(int32_t num_rows, int num_sms, int32_t* tail_row0);
// Workspace bytes of the tail split's partials and arrival counters (0: none).
size_t attn_tail_ws_bytes(int32_t num_rows, int32_t H, int num_sms);
// Sets a's tail split (tail_row0, tail_splits, row_done, part: the counters
// first) when the rows have a tail and `bytes` at `base` hold it; otherwise no
// tail split.  The counters are zeroed before the call's first kernel.
void attn_tail_setup(AttnArgs& a, void* base, size_t bytes, int num_sms);

}  // namespace csa
