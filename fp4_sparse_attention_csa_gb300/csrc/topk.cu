// csa_topk: exact top-512 per row by (score descending, index ascending),
// output in ascending index order, padded with -1.
//
// [SGL] "DeepSeek-V4.1 Flash on SGLang: from 35 to 873 tokens/s",
//   "Architecture changes and KV cache compression": only the top 512 global
//   positions take part in attention; "DSpark adaptation and optimization":
//   invalid-position filtering is fused with the selection (rows with n <= 512
//   return every visible index, the rest of the row is -1).
//
// One thread-block cluster of C CTAs per row; CTA k owns a contiguous slice of
// the row and stages its keys in shared memory.  Keys are the order-preserving
// uint32 image of the fp32 scores (-0 folded onto +0).  Three radix passes
// (11, 11 and 10 bits) find the exact 512th-largest key T: each CTA builds a
// histogram of the keys that match the prefix so far (warp-aggregated shared
// atomics), the cluster sums the C histograms through distributed shared
// memory, and every CTA walks the summed histogram from the top.  A final
// index-ordered ballot compaction writes every key > T and the lowest-index
// keys == T until 512 are taken.  Cluster barriers are hardware barriers, so
// there is no spin-wait here.
#include <cooperative_groups.h>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kStageMax = 32768;   // keys staged per CTA (128 KB)
constexpr int kMaxCluster = 8;

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Pass {
  int shift;      // bit position of this digit
  int bits;       // digit width
};
__constant__ Pass kPasses[3] = {{21, 11}, {10, 11}, {0, 10}};

__global__ void __launch_bounds__(kThreads, 1) k_topk(TopkArgs a, int C, int slice_cap, int staged) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);                 // [kBins]
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + kBins * 4);     // [slice_cap] when staged
  __shared__ uint32_t s_warp[kWarps][2];
  __shared__ uint32_t s_cta_counts[2];      // this CTA's (gt, eq) for the final pass
  __shared__ uint32_t s_sel[4];             // prefix, remaining, threshold state

  const int r = blockIdx.y;
  const int k = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  const float* row = a.scores + (size_t)r * a.ld;
  int32_t* out = a.out + (size_t)r * TOPK;

  int n = a.n_valid ? __ldg(a.n_valid + r) : (__ldg(a.row_pos + r) + 1) / a.P;
  if (n < 0 || n > a.max_n) {
    if (tid == 0 && k == 0) raise_flag(a.status, CSA_FLAG_ROW_INVALID);
    n = n < 0 ? 0 : a.max_n;
  }
  if (n <= TOPK) {                 // every visible index, then padding
    if (k == 0)
      for (int i = tid; i < TOPK; i += kThreads) out[i] = i < n ? i : -1;
    return;                        // uniform across the cluster: no cluster barrier below is reached
  }
  const int per = (n + C - 1) / C;
  const int lo = min(n, k * per), hi = min(n, lo + per);
  const int len = hi - lo;
  if (staged) {
    for (int i = tid; i < len; i += kThreads) keys[i] = score_key(__ldg(row + lo + i));
  }
  auto key_at = [&](int i) -> uint32_t { return staged ? keys[i] : score_key(__ldg(row + lo + i)); };

  uint32_t prefix = 0, prefix_mask = 0;
  int remaining = TOPK;            // how many still to take at or below the prefix
  for (int p = 0; p < 3; ++p) {
    const int shift = kPasses[p].shift, bits = kPasses[p].bits, nb = 1 << bits;
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0u;
    __syncthreads();
    for (int base = 0; base < len; base += kThreads) {
      const int i = base + tid;
      bool take = false;
      uint32_t bin = 0;
      if (i < len) {
        const uint32_t key = key_at(i);
        take = (key & prefix_mask) == prefix;
        bin = (key >> shift) & (uint32_t)(nb - 1);
      }
      const uint32_t active = __ballot_sync(0xFFFFFFFFu, take);
      if (take) {
        const uint32_t peers = __match_any_sync(active, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
      }
    }
    cluster.sync();                // every CTA's histogram is complete
    // Sum the cluster's histograms and find the bin holding the remaining-th
    // largest key: thread t owns bins [4t, 4t+4) (nb <= 2048 = 4 * 512).
    uint32_t c4[4] = {0u, 0u, 0u, 0u};
    for (int j = 0; j < 4; ++j) {
      const int bin = 4 * tid + j;
      if (bin < nb) {
        for (int q = 0; q < C; ++q) c4[j] += *cluster.map_shared_rank(hist + bin, q);
      }
    }
    // exclusive count of keys in bins above this thread's bins
    uint32_t mine = c4[0] + c4[1] + c4[2] + c4[3];
    uint32_t incl = mine;          // suffix sum over threads > tid, via reversed scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, incl, o);
      if (lane + o < 32) incl += y;
    }
    if (lane == 0) s_warp[warp][0] = incl;
    __syncthreads();
    uint32_t above = incl - mine;  // later lanes of this warp
    for (int w2 = warp + 1; w2 < kWarps; ++w2) above += s_warp[w2][0];
    // bins 4t+3 .. 4t from the top
    uint32_t acc = above;
    for (int j = 3; j >= 0; --j) {
      const int bin = 4 * tid + j;
      if (bin < nb && acc < (uint32_t)remaining && acc + c4[j] >= (uint32_t)remaining) {
        s_sel[0] = (uint32_t)bin;
        s_sel[1] = (uint32_t)remaining - acc;
      }
      acc += c4[j];
    }
    cluster.sync();                // all remote reads of this pass are done
    const uint32_t bin = s_sel[0];
    remaining = (int)s_sel[1];
    prefix |= bin << shift;
    prefix_mask |= (uint32_t)(nb - 1) << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;       // exact 512th-largest key; take `remaining` of the equal keys

  // ---- index-ordered compaction.  Warp w owns the contiguous chunk
  // [w*cw, (w+1)*cw) of this CTA's slice.
  const int cw = (len + kWarps - 1) / kWarps;
  const int w0 = min(len, warp * cw), w1 = min(len, w0 + cw);
  uint32_t gt = 0, eq = 0;
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    uint32_t key = 0;
    if (i < w1) key = key_at(i);
    gt += __popc(__ballot_sync(0xFFFFFFFFu, i < w1 && key > T));
    eq += __popc(__ballot_sync(0xFFFFFFFFu, i < w1 && key == T));
  }
  if (lane == 0) {
    s_warp[warp][0] = gt;
    s_warp[warp][1] = eq;
  }
  __syncthreads();
  uint32_t gt_before = 0, eq_before = 0;
  if (tid == 0) {
    uint32_t g = 0, e = 0;
    for (int w2 = 0; w2 < kWarps; ++w2) {
      g += s_warp[w2][0];
      e += s_warp[w2][1];
    }
    s_cta_counts[0] = g;
    s_cta_counts[1] = e;
  }
  cluster.sync();
  for (int q = 0; q < k; ++q) {
    gt_before += *cluster.map_shared_rank(&s_cta_counts[0], q);
    eq_before += *cluster.map_shared_rank(&s_cta_counts[1], q);
  }
  for (int w2 = 0; w2 < warp; ++w2) {
    gt_before += s_warp[w2][0];
    eq_before += s_warp[w2][1];
  }
  const uint32_t take_eq = (uint32_t)remaining;
  uint32_t sel_before = gt_before + min(eq_before, take_eq);
  uint32_t eq_rank = eq_before;
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    uint32_t key = 0;
    if (i < w1) key = key_at(i);
    const bool is_eq = i < w1 && key == T;
    const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, is_eq);
    const uint32_t my_eq_rank = eq_rank + __popc(eqm & ((1u << lane) - 1u));
    const bool sel = (i < w1 && key > T) || (is_eq && my_eq_rank < take_eq);
    const uint32_t selm = __ballot_sync(0xFFFFFFFFu, sel);
    if (sel) {
      const uint32_t pos = sel_before + __popc(selm & ((1u << lane) - 1u));
      if (pos < (uint32_t)TOPK) out[pos] = lo + i;
    }
    sel_before += __popc(selm);
    eq_rank += __popc(eqm);
  }
  cluster.sync();                  // keep shared memory alive for remote readers
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.num_rows <= 0) return cudaSuccess;
  int C = (a.max_n + kStageMax - 1) / kStageMax;
  C = C < 1 ? 1 : (C > kMaxCluster ? kMaxCluster : C);
  // smaller rows: split into up to 8 CTAs of >= 4096 keys for parallelism
  while (C < kMaxCluster && (a.max_n + C - 1) / C > 8192 && (long long)a.num_rows * C < 296) C *= 2;
  if (C > kMaxCluster) C = kMaxCluster;
  const int slice_cap = (a.max_n + C - 1) / C;
  const int staged = slice_cap <= kStageMax;
  const size_t smem = kBins * 4 + (staged ? (size_t)slice_cap * 4 : 0);
  cudaError_t e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, a.num_rows, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_topk, a, C, slice_cap, staged);
}

}  // namespace csa
