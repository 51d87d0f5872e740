// csa_topk: exact top-512 per row by (score descending, index ascending),
// output in ascending index order, padded with -1.
//
// [SGL] "DeepSeek-V4.1 Flash on SGLang: from 35 to 873 tokens/s",
//   "Architecture changes and KV cache compression": only the top 512 global
//   positions take part in attention; "DSpark adaptation and optimization":
//   invalid-position filtering is fused with the selection (rows with n <= 512
//   return every visible index, the rest of the row is -1).
//
// Two kernels, both one thread-block cluster per row:
//  k_topk_row  rows up to 256K entries (every decode shape here): C <= 8
//              CTAs per row stream slices of the
//              L2-resident row; value range and value histogram are combined
//              over distributed shared memory, the entries in or above the
//              bin of rank 512 are compacted in row order into CTA 0, which
//              finds the exact 512th key and the ties' cut on that list.
//  k_topk      longer rows: C CTAs per row with each slice staged in shared
//              memory as order-preserving uint32 keys (-0 folded onto +0); a
//              4096-bin value-space histogram summed over the cluster finds
//              the bin of rank 512, whose keys are gathered into CTA 0 for a
//              radix select of the exact key T.
// In both, a candidate list that overflows (many ties at the cut) or a
// non-finite value range falls back to a three-pass radix select over all
// keys (11/11/10 bits), and an index-ordered compaction writes every key > T
// and the lowest-index keys == T until 512 are taken.  Cluster barriers are
// hardware barriers, so there is no spin-wait here.
#include <cooperative_groups.h>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;
constexpr int kCandCap = 4096;
constexpr int kStageMax = 32768;   // keys staged per CTA (128 KB)
constexpr int kMaxCluster = 8;

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

struct alignas(16) TopkSmem {
  uint64_t stage_bar;
  uint32_t hist[kBins];
  uint32_t cand_key[kCandCap];
  uint32_t cand_cnt;
  uint32_t warp_a[kWarps], warp_b[kWarps];
  float fmin, fmax;
  uint32_t sel_bin, sel_need, sel_T, sel_take, sel_mode;
  uint32_t cta_gt, cta_eq;
};

// Block-wide: find the bin holding the `need`-th largest among `nb` bins whose
// counts come from `count(bin)`.  Writes bin and the rank left inside it.
template <typename F>
__device__ void find_bin(F count, int nb, uint32_t need, TopkSmem& sm, uint32_t* bin_out, uint32_t* need_out) {
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  const int per = nb / kThreads;                        // bins per thread (nb multiple of 512)
  uint32_t c[8];
  uint32_t mine = 0;
  for (int j = 0; j < per; ++j) {
    c[j] = count(per * tid + j);
    mine += c[j];
  }
  uint32_t incl = mine;                                  // suffix sums over higher threads
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, incl, o);
    if (lane + o < 32) incl += y;
  }
  if (lane == 0) sm.warp_a[warp] = incl;
  __syncthreads();
  uint32_t acc = incl - mine;
  for (int w2 = warp + 1; w2 < kWarps; ++w2) acc += sm.warp_a[w2];
  for (int j = per - 1; j >= 0; --j) {
    if (acc < need && acc + c[j] >= need) {
      *bin_out = (uint32_t)(per * tid + j);
      *need_out = need - acc;
    }
    acc += c[j];
  }
  __syncthreads();
}

// Radix select over `m` keys in shared memory (one CTA): the need-th largest
// key T and how many keys are strictly larger.
__device__ void radix_select_block(const uint32_t* keys, int m, uint32_t need, TopkSmem& sm, uint32_t* T_out,
                                   uint32_t* gt_out) {
  uint32_t prefix = 0, mask = 0;
  uint32_t rem = need;
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
  for (int p = 0; p < 3; ++p) {
    const int sh = shifts[p], nbv = 1 << widths[p];
    for (int i = threadIdx.x; i < kBins; i += kThreads) sm.hist[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += kThreads) {
      const uint32_t k = keys[i];
      if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> sh) & (uint32_t)(nbv - 1)], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) sm.sel_bin = 0xFFFFFFFFu;
    __syncthreads();
    find_bin([&](int b) { return b < nbv ? sm.hist[b] : 0u; }, 2048, rem, sm, &sm.sel_bin, &sm.sel_need);
    prefix |= sm.sel_bin << sh;
    mask |= (uint32_t)(nbv - 1) << sh;
    rem = sm.sel_need;
    __syncthreads();
  }
  *T_out = prefix;
  *gt_out = need - rem;
}

__global__ void __launch_bounds__(kThreads, 1) k_topk(TopkArgs a, int C, int slice_cap, int staged) {
  pdl_trigger();
  pdl_wait();                    // the scores come from the previous kernel
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) uint8_t smem[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + sizeof(TopkSmem));  // [slice_cap] when staged

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
  const int per = (((n + C - 1) / C) + 3) & ~3;        // slices start on 16-byte boundaries
  const int lo = min(n, k * per), hi = min(n, lo + per);
  const int len = hi - lo;

  // ---- stage the slice (one bulk copy of its 16-byte part, plain loads for the
  // tail), then convert to keys and take the local value range --------------------------
  float vmin = INFINITY, vmax = -INFINITY;
  if (staged) {
    const int body = len & ~3;
    if (tid == 0) {
      mbar_init(&sm.stage_bar, 1);
      fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
      mbar_expect_tx(&sm.stage_bar, (uint32_t)body * 4u);
      if (body > 0) bulk_load(keys, row + lo, (uint32_t)body * 4u, &sm.stage_bar);
    }
    if (tid < len - body) keys[body + tid] = __float_as_uint(__ldg(row + lo + body + tid));
    if (!mbar_wait(&sm.stage_bar, 0)) {
      if (tid == 0) raise_flag(a.status, CSA_FLAG_TIMEOUT);
    }
    __syncthreads();
    for (int i = tid; i < len; i += kThreads) {
      float v = __uint_as_float(keys[i]);
      if (v == 0.0f) v = 0.0f;                          // fold -0 onto +0
      vmin = fminf(vmin, v);
      vmax = fmaxf(vmax, v);
      keys[i] = score_key(v);
    }
  } else {
    for (int i0 = tid * 4; i0 < len; i0 += kThreads * 4) {
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = (i0 + j < len) ? __ldg(row + lo + i0 + j) : NAN;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (i0 + j < len) {
          vmin = fminf(vmin, v[j]);
          vmax = fmaxf(vmax, v[j]);
        }
      }
    }
  }
  auto key_at = [&](int i) -> uint32_t { return staged ? keys[i] : score_key(__ldg(row + lo + i)); };
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    vmin = fminf(vmin, __shfl_xor_sync(0xFFFFFFFFu, vmin, o));
    vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, o));
  }
  if (lane == 0) {
    sm.warp_a[warp] = __float_as_uint(vmin);
    sm.warp_b[warp] = __float_as_uint(vmax);
  }
  for (int i = tid; i < kBins; i += kThreads) sm.hist[i] = 0u;
  if (tid == 0) sm.cand_cnt = 0u;
  __syncthreads();
  if (tid == 0) {
    float a0 = INFINITY, b0 = -INFINITY;
    for (int w2 = 0; w2 < kWarps; ++w2) {
      a0 = fminf(a0, __uint_as_float(sm.warp_a[w2]));
      b0 = fmaxf(b0, __uint_as_float(sm.warp_b[w2]));
    }
    sm.fmin = a0;
    sm.fmax = b0;
  }
  cluster.sync();
  float smin = INFINITY, smax = -INFINITY;
  for (int q = 0; q < C; ++q) {
    const TopkSmem* rs = cluster.map_shared_rank(&sm, q);
    smin = fminf(smin, rs->fmin);
    smax = fmaxf(smax, rs->fmax);
  }
  const float range = smax - smin;
  const bool binning = isfinite(range) && range > 0.0f;
  const float scale = binning ? (float)kBins / range : 0.0f;
  auto bin_of = [&](uint32_t key) -> uint32_t {
    const float v = key_value(key);
    const float f = (v - smin) * scale;
    const int b = (int)f;
    return (uint32_t)(b < 0 ? 0 : (b >= kBins ? kBins - 1 : b));
  };

  uint32_t T = 0, take_eq = 0;
  int mode = 0;                    // 0: value bins, 1: all keys equal, 2: radix fallback
  if (!binning) mode = (range == 0.0f) ? 1 : 2;
  if (mode == 1) {
    T = score_key(smin);
    take_eq = TOPK;
  } else if (mode == 0) {
    // ---- 4096-bin histogram in value space ------------------------------------------
    for (int i = tid; i < len; i += kThreads) atomicAdd(&sm.hist[bin_of(key_at(i))], 1u);
    cluster.sync();
    find_bin(
        [&](int b) {
          uint32_t s = 0;
          for (int q = 0; q < C; ++q) s += *cluster.map_shared_rank(&sm.hist[b], q);
          return s;
        },
        kBins, TOPK, sm, &sm.sel_bin, &sm.sel_need);
    const uint32_t tb = sm.sel_bin, need = sm.sel_need;
    uint32_t in_bin = 0, before = 0;
    for (int q = 0; q < C; ++q) {
      const uint32_t c = *cluster.map_shared_rank(&sm.hist[tb], q);
      in_bin += c;
      if (q < k) before += c;
    }
    if (in_bin > (uint32_t)kCandCap) {
      mode = 2;
    } else {
      // ---- gather the threshold bin's keys into CTA 0, select there -------------------
      uint32_t* cand0 = cluster.map_shared_rank(sm.cand_key, 0);
      for (int i0 = 0; i0 < len; i0 += kThreads) {
        const int i = i0 + tid;
        bool hit = false;
        uint32_t key = 0;
        if (i < len) {
          key = key_at(i);
          hit = bin_of(key) == tb;
        }
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, hit);
        uint32_t base = 0;
        if (lane == 0 && bal) base = atomicAdd(&sm.cand_cnt, (uint32_t)__popc(bal));
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
        if (hit) cand0[before + base + __popc(bal & ((1u << lane) - 1u))] = key;
      }
      cluster.sync();
      if (k == 0) {
        uint32_t Tc, gt;
        radix_select_block(sm.cand_key, (int)in_bin, need, sm, &Tc, &gt);
        if (tid == 0) {
          sm.sel_T = Tc;
          sm.sel_take = need - gt;
        }
      }
      cluster.sync();
      const TopkSmem* s0 = cluster.map_shared_rank(&sm, 0);
      T = s0->sel_T;
      take_eq = s0->sel_take;
    }
  }
  if (mode == 2) {
    // ---- fallback: three radix passes over every key ----------------------------------
    uint32_t prefix = 0, mask = 0, rem = TOPK;
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int p = 0; p < 3; ++p) {
      const int sh = shifts[p], nbv = 1 << widths[p];
      cluster.sync();              // everyone is done reading the previous histograms
      for (int i = tid; i < kBins; i += kThreads) sm.hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < len; i += kThreads) {
        const uint32_t key = key_at(i);
        if ((key & mask) == prefix) atomicAdd(&sm.hist[(key >> sh) & (uint32_t)(nbv - 1)], 1u);
      }
      cluster.sync();
      find_bin(
          [&](int b) {
            uint32_t s = 0;
            if (b < nbv)
              for (int q = 0; q < C; ++q) s += *cluster.map_shared_rank(&sm.hist[b], q);
            return s;
          },
          2048, rem, sm, &sm.sel_bin, &sm.sel_need);
      prefix |= sm.sel_bin << sh;
      mask |= (uint32_t)(nbv - 1) << sh;
      rem = sm.sel_need;
    }
    T = prefix;
    take_eq = rem;
  }

  // ---- index-ordered compaction.  Warp w owns [w*cw, (w+1)*cw) of the slice.
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
    sm.warp_a[warp] = gt;
    sm.warp_b[warp] = eq;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t g = 0, e = 0;
    for (int w2 = 0; w2 < kWarps; ++w2) {
      g += sm.warp_a[w2];
      e += sm.warp_b[w2];
    }
    sm.cta_gt = g;
    sm.cta_eq = e;
  }
  cluster.sync();
  uint32_t gt_before = 0, eq_before = 0;
  for (int q = 0; q < k; ++q) {
    const TopkSmem* rs = cluster.map_shared_rank(&sm, q);
    gt_before += rs->cta_gt;
    eq_before += rs->cta_eq;
  }
  for (int w2 = 0; w2 < warp; ++w2) {
    gt_before += sm.warp_a[w2];
    eq_before += sm.warp_b[w2];
  }
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

// ---------------------------------------------------------------------------
// Rows up to kRowMax entries: a cluster of C CTAs per row (C set at launch),
// CTA k streaming the contiguous slice [k*S, min(n, (k+1)*S)) of the
// L2-resident row with 16-byte loads (S a multiple of 4), or reading it from
// shared memory where its layout stages the slice (the packed launch).  The cluster
//   1. reduces the slices' value ranges through distributed shared memory,
//   2. sums the CTAs' kRowBins-bin value histograms (read remotely); every CTA
//      derives the same bin tb holding rank 512, the count above it and the
//      count inside it,
//   3. each CTA lists its slice's entries above tb (all selected) and in tb
//      (the cut's candidates) in its own shared memory, a warp at a time with
//      one atomic per list per warp, then copies its lists into CTA 0's at
//      the offsets the CTAs' counts give; the lists are unordered,
// and CTA 0 picks the cut bin's entries by (score desc, index asc) -- by
// pairwise rank when there are few, else by radix select -- marks every
// selected index in a bitmap of the row and writes the bitmap out in index
// order.  A cut bin with more entries than the layout's tie capacity (many
// ties) or a non-finite range falls back to a whole-row radix select in CTA 0.  A CTA leaves only
// after a cluster barrier that follows every remote access to its shared memory.
constexpr int kRowMax = 262144;
constexpr int kRowBins = 2048;
constexpr int kTieCap = 4096;
constexpr int kPairwiseMax = 256;   // cut bins up to this size are ranked pairwise
constexpr int kRowCluster = 8;

// Shared memory of a row's CTA for rows of up to kMaxN entries, a cut bin of
// up to kTies entries, and (kCache > 0) this CTA's slice of the row staged
// once by a bulk copy and read from there by all three passes.
template <int kMaxN, int kTies, int kCache>
struct alignas(16) RowSmemT {
  static constexpr int kTieCapacity = kTies;
  static constexpr int kCacheFloats = kCache;
  uint32_t hist[kRowBins];         // value histogram; the radix passes reuse it
  uint32_t bitmap[kMaxN / 32];     // CTA 0: selected indices of the row
  uint32_t tie_key[kTies];         // CTA 0: the cut bin's entries (unordered)
  int32_t tie_idx[kTies];
  int32_t gt_idx[TOPK];            // the entries above the cut bin (unordered)
  uint32_t warp_a[kWarps], warp_b[kWarps];
  uint32_t gt_cnt, tie_cnt;        // this CTA's list lengths
  uint32_t sel_bin, sel_need, sel_tie;
  float fmin, fmax;
  uint64_t cache_bar;              // the slice's bulk copy
  alignas(16) float cache[kCache > 0 ? kCache : 4];
};
using RowSmem = RowSmemT<kRowMax, kTieCap, 0>;

template <typename SM>
__device__ __forceinline__ void block_minmax(float& vmin, float& vmax, SM& sm) {
  const int lane = lane_id(), warp = warp_id();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    vmin = fminf(vmin, __shfl_xor_sync(0xFFFFFFFFu, vmin, o));
    vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, o));
  }
  if (lane == 0) {
    sm.warp_a[warp] = __float_as_uint(vmin);
    sm.warp_b[warp] = __float_as_uint(vmax);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a0 = INFINITY, b0 = -INFINITY;
    for (int w2 = 0; w2 < kWarps; ++w2) {
      a0 = fminf(a0, __uint_as_float(sm.warp_a[w2]));
      b0 = fmaxf(b0, __uint_as_float(sm.warp_b[w2]));
    }
    sm.fmin = a0;
    sm.fmax = b0;
  }
  __syncthreads();
}

// Block-wide exclusive scan of one count per thread; returns the thread's
// offset and the block total (uses warp_a).
template <typename SM>
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* total, SM& sm) {
  const int lane = lane_id(), warp = warp_id();
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm.warp_a[warp] = x;
  __syncthreads();
  uint32_t off = 0, tot = 0;
  for (int w2 = 0; w2 < kWarps; ++w2) {
    const uint32_t c = sm.warp_a[w2];
    if (w2 < warp) off += c;
    tot += c;
  }
  __syncthreads();
  *total = tot;
  return off + x - v;
}

// Block-wide radix select (11/11/10 bits) of the need-th largest key among the
// m keys key_at(i) with valid(i): the key T and how many of the keys equal to T
// are taken (need minus the keys above T).  Uses hist, warp_a, sel_bin, sel_need.
template <typename K, typename V, typename SM>
__device__ void row_radix(K key_at, V valid, int m, uint32_t need, SM& sm, uint32_t* T_out, uint32_t* take_out) {
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  uint32_t prefix = 0, mask = 0, rem = need;
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
  for (int p = 0; p < 3; ++p) {
    const int sh = shifts[p], nbv = 1 << widths[p];
    for (int i = tid; i < 2048; i += kThreads) sm.hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < m; i += kThreads) {
      if (!valid(i)) continue;
      const uint32_t kk = key_at(i);
      if ((kk & mask) == prefix) atomicAdd(&sm.hist[(kk >> sh) & (uint32_t)(nbv - 1)], 1u);
    }
    __syncthreads();
    constexpr int per = 2048 / kThreads;
    uint32_t c[per], mine = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      const int b = per * tid + j;
      c[j] = b < nbv ? sm.hist[b] : 0u;
      mine += c[j];
    }
    uint32_t incl = mine;                         // suffix sums over higher lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, incl, o);
      if (lane + o < 32) incl += y;
    }
    if (lane == 0) sm.warp_a[warp] = incl;
    __syncthreads();
    uint32_t acc = incl - mine;
    for (int w2 = warp + 1; w2 < kWarps; ++w2) acc += sm.warp_a[w2];
#pragma unroll
    for (int j = per - 1; j >= 0; --j) {
      if (acc < rem && acc + c[j] >= rem) {
        sm.sel_bin = (uint32_t)(per * tid + j);
        sm.sel_need = rem - acc;
      }
      acc += c[j];
    }
    __syncthreads();
    prefix |= sm.sel_bin << sh;
    mask |= (uint32_t)(nbv - 1) << sh;
    rem = sm.sel_need;
    __syncthreads();
  }
  *T_out = prefix;
  *take_out = rem;
}

template <typename SM>
__device__ __forceinline__ void mark(SM& sm, int idx) {
  atomicOr(&sm.bitmap[idx >> 5], 1u << (idx & 31));
}

// The CTAs that share a row: a thread-block cluster of C (C > 1), or this CTA
// alone (C == 1), whose barrier is then the CTA's own and whose "remote" shared
// memory is its own.
template <int N>
struct IntConst {
  static constexpr int value = N;
};

template <int C>
struct RowGroup {
  __device__ __forceinline__ void sync() const {
    if constexpr (C == 1) __syncthreads();
    else cg::this_cluster().sync();
  }
  template <typename T>
  __device__ __forceinline__ T* at(T* p, int q) const {
    if constexpr (C == 1) return p;
    else return cg::this_cluster().map_shared_rank(p, q);
  }
};

// The entries row r sees, as given (n_valid) or from its position: a call
// input, read before the wait for the scores.
__device__ __forceinline__ int row_n(const TopkArgs& a, int r) {
  return a.n_valid ? __ldg(a.n_valid + r) : (__ldg(a.row_pos + r) + 1) / a.P;
}

// Row r's top-512 by its C CTAs; this is CTA kq of them; n_row = row_n(a, r).
template <int C, typename SM>  // CTAs per row: 1, 2, 4 or 8; the shared memory's layout
__device__ __forceinline__ void topk_row(const TopkArgs& a, SM& sm, int r, int kq, int n_row) {
  const RowGroup<C> grp;
  const int tid = threadIdx.x, lane = lane_id();
  const float* row = a.scores + (size_t)r * a.ld;
  int32_t* out = a.out + (size_t)r * TOPK;

  int n = n_row;
  if (n < 0 || n > a.max_n) {
    if (tid == 0 && kq == 0) raise_flag(a.status, CSA_FLAG_ROW_INVALID);
    n = n < 0 ? 0 : a.max_n;
  }
  if (n <= TOPK) {                 // the same branch in every CTA of the cluster
    if (kq == 0)
      for (int i = tid; i < TOPK; i += kThreads) out[i] = i < n ? i : -1;
    return;
  }
  const int S = (((n + C - 1) / C) + 3) & ~3;
  const int lo = min(n, kq * S), len = min(n, lo + S) - lo;
  const float* sl = row + lo;
  const float4* sl4 = reinterpret_cast<const float4*>(sl);   // lo is a multiple of 4
  const int n4 = len >> 2;
  auto fold = [](float v) { return v == 0.0f ? 0.0f : v; };   // -0 onto +0
  // the slice's values: from the staged copy in shared memory, or from global
  // memory (L2)
  constexpr bool kCached = SM::kCacheFloats > 0;
  auto ld4 = [&](int i) -> float4 {
    if constexpr (kCached) return reinterpret_cast<const float4*>(sm.cache)[i];
    else return __ldg(sl4 + i);
  };
  auto ld1 = [&](int i) -> float {
    if constexpr (kCached) return sm.cache[i];
    else return __ldg(sl + i);
  };
  if constexpr (kCached) {
    // one bulk copy of the slice rounded up to 16 bytes (the row's stride is a
    // multiple of 4 entries, so the copy stays inside the row)
    const int len4 = (len + 3) & ~3;
    const uint32_t bytes = len4 <= SM::kCacheFloats ? (uint32_t)len4 * 4u : 0u;
    if (len4 > SM::kCacheFloats && tid == 0) raise_flag(a.status, CSA_FLAG_ROW_INVALID);
    if (tid == 0) {
      mbar_init(&sm.cache_bar, 1);
      fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0 && bytes > 0u) {
      mbar_expect_tx(&sm.cache_bar, bytes);
      bulk_load(sm.cache, sl, bytes, &sm.cache_bar);
    }
    if (bytes > 0u && !mbar_wait(&sm.cache_bar, 0)) {
      raise_flag(a.status, CSA_FLAG_TIMEOUT);
      (void)mbar_wait(&sm.cache_bar, 0);       // the copy is not left in flight
    }
  }

  // ---- pass 1: value range of the slice, then of the row ----------------------------
  float vmin = INFINITY, vmax = -INFINITY;
  for (int b0 = tid; b0 < n4; b0 += 4 * kThreads) {
    float4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = b0 + j * kThreads;
      v[j] = i < n4 ? ld4(i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (b0 + j * kThreads < n4) {
        vmin = fminf(vmin, fminf(fminf(v[j].x, v[j].y), fminf(v[j].z, v[j].w)));
        vmax = fmaxf(vmax, fmaxf(fmaxf(v[j].x, v[j].y), fmaxf(v[j].z, v[j].w)));
      }
    }
  }
  for (int i = 4 * n4 + tid; i < len; i += kThreads) {
    const float v = ld1(i);
    vmin = fminf(vmin, v);
    vmax = fmaxf(vmax, v);
  }
  for (int i = tid; i < kRowBins; i += kThreads) sm.hist[i] = 0u;
  if (kq == 0)                     // CTA 0's bitmap starts empty
    for (int i = tid; i < (n + 31) >> 5; i += kThreads) sm.bitmap[i] = 0u;
  if (tid == 0) sm.gt_cnt = sm.tie_cnt = 0u;
  block_minmax(vmin, vmax, sm);
  grp.sync();                                  // every slice's range is published
  vmin = INFINITY;
  vmax = -INFINITY;
  for (int q = 0; q < C; ++q) {
    const SM* rs = grp.at(&sm, q);
    vmin = fminf(vmin, rs->fmin);
    vmax = fmaxf(vmax, rs->fmax);
  }
  vmin = fold(vmin);
  vmax = fold(vmax);
  const float range = vmax - vmin;
  const bool binning = range != 0.0f && isfinite(range) && isfinite((float)kRowBins / range);
  const float scale = binning ? (float)kRowBins / range : 0.0f;
  auto bin_of = [&](float v) -> int {
    const int b = (int)((fold(v) - vmin) * scale);
    return b < 0 ? 0 : (b >= kRowBins ? kRowBins - 1 : b);
  };

  bool done = false;
  if (binning) {
    // ---- pass 2: histogram of the slice ---------------------------------------------
    for (int b0 = tid; b0 < n4; b0 += 4 * kThreads) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = b0 + j * kThreads;
        v[j] = i < n4 ? ld4(i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (b0 + j * kThreads < n4) {
          atomicAdd(&sm.hist[bin_of(v[j].x)], 1u);
          atomicAdd(&sm.hist[bin_of(v[j].y)], 1u);
          atomicAdd(&sm.hist[bin_of(v[j].z)], 1u);
          atomicAdd(&sm.hist[bin_of(v[j].w)], 1u);
        }
      }
    }
    for (int i = 4 * n4 + tid; i < len; i += kThreads) atomicAdd(&sm.hist[bin_of(ld1(i))], 1u);
  }
  grp.sync();                                  // histograms complete; range reads done
  if (!binning) {
    if (kq != 0) return;           // CTA 0 alone: all equal, or the whole-row radix below
    if (range == 0.0f) {           // all equal: the lowest 512 indices
      for (int i = tid; i < TOPK; i += kThreads) out[i] = i;
      return;
    }
  } else {
    // ---- the bin of rank 512 in the summed histogram, the count above it and
    // the count inside it (the same in every CTA) ---------------------------------------
    const int warp = warp_id();
    constexpr int per = kRowBins / kThreads;
    uint32_t c[per], mine = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) c[j] = 0u;
#pragma unroll
    for (int q = 0; q < C; ++q) {
      const uint4 h = *reinterpret_cast<const uint4*>(grp.at(sm.hist, q) + per * tid);
      c[0] += h.x; c[1] += h.y; c[2] += h.z; c[3] += h.w;
    }
#pragma unroll
    for (int j = 0; j < per; ++j) mine += c[j];
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, incl, o);
      if (lane + o < 32) incl += y;
    }
    if (lane == 0) sm.warp_a[warp] = incl;
    __syncthreads();
    uint32_t acc = incl - mine;
    for (int w2 = warp + 1; w2 < kWarps; ++w2) acc += sm.warp_a[w2];
#pragma unroll
    for (int j = per - 1; j >= 0; --j) {
      if (acc < (uint32_t)TOPK && acc + c[j] >= (uint32_t)TOPK) {
        sm.sel_bin = (uint32_t)(per * tid + j);
        sm.sel_need = acc;                          // entries above the bin
        sm.sel_tie = c[j];                          // entries in the bin
      }
      acc += c[j];
    }
    __syncthreads();
    const int tb = (int)sm.sel_bin;
    const uint32_t n_gt = sm.sel_need, n_tie = sm.sel_tie;
    if (n_tie > (uint32_t)SM::kTieCapacity) {
      grp.sync();                              // every remote histogram read is done
      if (kq != 0) return;         // CTA 0 alone: the whole-row radix below
    } else {
      // ---- pass 3: list the slice's entries in or above tb --------------------------
      const float tbf = (float)tb;
      // a thread's up-to-16 values: count its entries above tb and in tb, one
      // warp scan each, one atomic per list per warp, then the writes
      // a value's class by the same arithmetic as bin_of: its bin above tb
      // (floor(x) >= tb + 1, and tb not the last bin), or equal to tb; a NaN
      // value's bin is 0
      const float tbf1 = (float)(tb + 1);
      const bool gt_possible = tb < kRowBins - 1;
      // (-0 and +0 class alike here: x differs at most in the sign of a zero)
      auto classify = [&](float v, bool valid, uint32_t bit, uint32_t& gtm, uint32_t& tiem) {
        const float x = (v - vmin) * scale;
        if (!valid) return;
        if (gt_possible && x >= tbf1) gtm |= bit;
        else if (tb == 0 || x >= tbf) tiem |= bit;
      };
      // a thread's candidates (bit j: its value j, entry ibase + (j / 4) * 4 *
      // kThreads + j % 4): one warp scan per list, one atomic per list per warp,
      // then the writes -- the indices above the cut bin by their set bits, the
      // cut bin's keys and indices (few) only in warps that hold some
      auto collect = [&](auto cnt_c, uint32_t gtm, uint32_t tiem, const float* v, int ibase) {
        [[maybe_unused]] constexpr int kCnt = decltype(cnt_c)::value;
        const uint32_t ng = (uint32_t)__popc(gtm), nt = (uint32_t)__popc(tiem);
        uint32_t ig = ng, it = nt;                  // inclusive warp scans
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t yg = __shfl_up_sync(0xFFFFFFFFu, ig, o), yt = __shfl_up_sync(0xFFFFFFFFu, it, o);
          if (lane >= o) { ig += yg; it += yt; }
        }
        uint32_t bg = 0, bt = 0;
        if (lane == 31) {
          if (ig) bg = atomicAdd(&sm.gt_cnt, ig);
          if (it) bt = atomicAdd(&sm.tie_cnt, it);
        }
        bg = __shfl_sync(0xFFFFFFFFu, bg, 31) + ig - ng;
        bt = __shfl_sync(0xFFFFFFFFu, bt, 31) + it - nt;
        for (uint32_t m = gtm; m != 0u; m &= m - 1u) {
          const int j = __ffs(m) - 1;
          sm.gt_idx[bg++] = lo + ibase + (j >> 2) * (4 * kThreads) + (j & 3);
        }
        if constexpr (kCached) {
          // the staged slice gives a value by its index: one pass over the set bits
          for (uint32_t m = tiem; m != 0u; m &= m - 1u) {
            const int j = __ffs(m) - 1;
            const int e = ibase + (j >> 2) * (4 * kThreads) + (j & 3);
            sm.tie_key[bt] = score_key(fold(sm.cache[e]));
            sm.tie_idx[bt] = lo + e;
            ++bt;
          }
        } else if (__any_sync(0xFFFFFFFFu, tiem != 0u)) {
#pragma unroll
          for (int j = 0; j < kCnt; ++j)
            if (tiem & (1u << j)) {
              sm.tie_key[bt] = score_key(fold(v[j]));
              sm.tie_idx[bt] = lo + ibase + (j >> 2) * (4 * kThreads) + (j & 3);
              ++bt;
            }
        }
      };
      const int n4r = (n4 + 4 * kThreads - 1) / (4 * kThreads) * (4 * kThreads);   // warp-uniform trip count
      for (int base4 = 0; base4 < n4r; base4 += 4 * kThreads) {
        float v[16];
        uint32_t gtm = 0u, tiem = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = base4 + tid + j * kThreads;
          const bool valid = i < n4;
          const float4 x = valid ? ld4(i) : make_float4(vmin, vmin, vmin, vmin);
          v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
#pragma unroll
          for (int c = 0; c < 4; ++c) classify(v[4 * j + c], valid, 1u << (4 * j + c), gtm, tiem);
        }
        if (!__any_sync(0xFFFFFFFFu, (gtm | tiem) != 0u)) continue;
        collect(IntConst<16>(), gtm, tiem, v, 4 * (base4 + tid));
      }
      if (tid < 32) {                              // the slice's last (len mod 4) entries
        const int i = 4 * n4 + lane;
        const bool valid = i < len;
        float v1[1] = {valid ? ld1(i) : vmin};
        uint32_t gtm = 0u, tiem = 0u;
        classify(v1[0], valid, 1u, gtm, tiem);
        collect(IntConst<1>(), gtm, tiem, v1, i);
      }
      grp.sync();                              // every CTA's counts are final
      // ---- CTA q's lists go to CTA 0's at the offsets of CTAs 0..q-1 ---------------
      if (kq != 0) {
        uint32_t og = 0, ot = 0;
        for (int q = 0; q < kq; ++q) {
          const SM* rs = grp.at(&sm, q);
          og += rs->gt_cnt;
          ot += rs->tie_cnt;
        }
        int32_t* r_gt_idx = grp.at(sm.gt_idx, 0);
        uint32_t* r_tie_key = grp.at(sm.tie_key, 0);
        int32_t* r_tie_idx = grp.at(sm.tie_idx, 0);
        for (uint32_t t = tid; t < sm.gt_cnt; t += kThreads) r_gt_idx[og + t] = sm.gt_idx[t];
        for (uint32_t t = tid; t < sm.tie_cnt; t += kThreads) {
          r_tie_key[ot + t] = sm.tie_key[t];
          r_tie_idx[ot + t] = sm.tie_idx[t];
        }
      }
      grp.sync();                              // the lists are complete in CTA 0
      if (kq != 0) return;
      // ---- CTA 0: the cut bin's entries by (score desc, index asc) ----------------
      const uint32_t need = (uint32_t)TOPK - n_gt;  // 1 <= need <= n_tie
      for (int t = tid; t < (int)n_gt; t += kThreads) mark(sm, sm.gt_idx[t]);
      if (n_tie <= (uint32_t)kPairwiseMax) {
        if (tid < (int)n_tie) {
          const uint32_t k0 = sm.tie_key[tid];
          const int i0 = sm.tie_idx[tid];
          uint32_t rank = 0;
          for (int j = 0; j < (int)n_tie; ++j) {
            const uint32_t kj = sm.tie_key[j];
            rank += (kj > k0 || (kj == k0 && sm.tie_idx[j] < i0)) ? 1u : 0u;
          }
          if (rank < need) mark(sm, i0);
        }
      } else {
        uint32_t T, take;
        row_radix([&](int i) { return sm.tie_key[i]; }, [](int) { return true; }, (int)n_tie, need, sm, &T, &take);
        // the keys above T, and the `take` lowest indices among the keys equal to
        // T: the take-th largest of (kRowMax - index) over those
        uint32_t U = 0, take_u = 0;
        row_radix([&](int i) { return (uint32_t)(kRowMax - sm.tie_idx[i]); },
                  [&](int i) { return sm.tie_key[i] == T; }, (int)n_tie, take, sm, &U, &take_u);
        for (int t = tid; t < (int)n_tie; t += kThreads) {
          const uint32_t kk = sm.tie_key[t];
          if (kk > T || (kk == T && (uint32_t)(kRowMax - sm.tie_idx[t]) >= U)) mark(sm, sm.tie_idx[t]);
        }
      }
      __syncthreads();
      // ---- output: the bitmap in index order ---------------------------------------
      const int nw = (n + 31) >> 5;
      const int wper = (nw + kThreads - 1) / kThreads;
      const int w0 = min(nw, tid * wper), w1 = min(nw, w0 + wper);
      uint32_t cnt = 0;
      for (int w = w0; w < w1; ++w) cnt += (uint32_t)__popc(sm.bitmap[w]);
      uint32_t tot;
      uint32_t pos = block_scan(cnt, &tot, sm);
      for (int w = w0; w < w1; ++w) {
        uint32_t bits = sm.bitmap[w];
        while (bits) {
          const int b = __ffs(bits) - 1;
          bits &= bits - 1u;
          if (pos < (uint32_t)TOPK) out[pos] = 32 * w + b;
          ++pos;
        }
      }
      done = true;
    }
  }
  if (!done) {
    // ---- fallback: radix select over the whole row, then an ordered pass ----------
    uint32_t prefix = 0, mask = 0, rem = TOPK;
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int p = 0; p < 3; ++p) {
      const int sh = shifts[p], nbv = 1 << widths[p];
      for (int i = tid; i < 2048; i += kThreads) sm.hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < n; i += kThreads) {
        const uint32_t kk = score_key(__ldg(row + i));
        if ((kk & mask) == prefix) atomicAdd(&sm.hist[(kk >> sh) & (uint32_t)(nbv - 1)], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t acc = 0;
        for (int b = nbv - 1; b >= 0; --b) {
          const uint32_t c = sm.hist[b];
          if (acc < rem && acc + c >= rem) {
            sm.sel_bin = (uint32_t)b;
            sm.sel_need = rem - acc;
            break;
          }
          acc += c;
        }
      }
      __syncthreads();
      prefix |= sm.sel_bin << sh;
      mask |= (uint32_t)(nbv - 1) << sh;
      rem = sm.sel_need;
      __syncthreads();
    }
    const uint32_t T = prefix, take = rem;
    uint32_t eq_base = 0, sel_base = 0;
    for (int c0 = 0; c0 < n; c0 += kThreads) {
      const int i = c0 + tid;
      const uint32_t kk = i < n ? score_key(__ldg(row + i)) : 0u;
      const uint32_t is_eq = (i < n && kk == T) ? 1u : 0u;
      uint32_t tot_eq;
      const uint32_t eq_rank = eq_base + block_scan(is_eq, &tot_eq, sm);
      const uint32_t sel = (i < n && (kk > T || (is_eq && eq_rank < take))) ? 1u : 0u;
      uint32_t tot_sel;
      const uint32_t pos = sel_base + block_scan(sel, &tot_sel, sm);
      if (sel && pos < (uint32_t)TOPK) out[pos] = i;
      eq_base += tot_eq;
      sel_base += tot_sel;
    }
  }
}

template <int C>                   // CTAs per row: 1, 2, 4 or 8
__global__ void __launch_bounds__(kThreads) k_topk_row(TopkArgs a) {
  pdl_trigger();
  const int r = (int)blockIdx.x / C;
  const int n_row = row_n(a, r);
  pdl_wait();                    // the scores come from the previous kernel
  extern __shared__ __align__(16) uint8_t smem[];
  RowSmem& sm = *reinterpret_cast<RowSmem*>(smem);
  const int kq = C == 1 ? 0 : (int)cg::this_cluster().block_rank();
  topk_row<C>(a, sm, r, kq, n_row);
}

// Rows of very different lengths (up to kPackC * kPackLong entries): clusters
// of kPackC CTAs, the rows longer than kPackLong one to a cluster, then the
// others one to a CTA, four to a cluster, each in row order; so no CTA streams
// more than kPackLong entries and short rows do not tie up a whole cluster.
// Every CTA derives the same assignment from the rows' lengths; clusters past
// the work return at once.
constexpr int kPackC = 4;
constexpr int kPackLong = 16384;
// Rows of up to kPackC * kPackLong entries, slices of up to kPackLong staged in
// shared memory; 3072 cut-bin entries keep two CTAs per SM (106 KB each).
using PackSmem = RowSmemT<kPackC * kPackLong, 3072, kPackLong>;
static_assert(2 * (sizeof(PackSmem) + 1024) <= 228 * 1024, "two packed CTAs per SM");

__global__ void __launch_bounds__(kThreads) k_topk_packed(TopkArgs a) {
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  PackSmem& sm = *reinterpret_cast<PackSmem*>(smem);
  const int tid = threadIdx.x;
  const int c = (int)blockIdx.x / kPackC, kq = (int)cg::this_cluster().block_rank();
  auto row_len = [&](int r) {
    const int n = row_n(a, r);
    return n < 0 ? 0 : (n > a.max_n ? a.max_n : n);
  };
  // the long rows come first: how many there are
  int n_long = 0;
  for (int base = 0; base < a.num_rows; base += kThreads) {
    const int r = base + tid;
    n_long += __syncthreads_count(r < a.num_rows && row_len(r) > kPackLong);
  }
  // this cluster's long row, or this CTA's short row: the target-th of its kind
  const bool want_long = c < n_long;
  const uint32_t target = want_long ? (uint32_t)c : (uint32_t)(c - n_long) * kPackC + (uint32_t)kq;
  if (tid == 0) sm.sel_bin = 0xFFFFFFFFu;
  uint32_t seen = 0;
  for (int base = 0; base < a.num_rows; base += kThreads) {
    const int r = base + tid;
    const uint32_t kind = (r < a.num_rows && (row_len(r) > kPackLong) == want_long) ? 1u : 0u;
    uint32_t tot;
    const uint32_t pre = seen + block_scan(kind, &tot, sm);
    if (kind && pre == target) sm.sel_bin = (uint32_t)r;
    seen += tot;
    if (seen > target) break;    // the same for every thread
  }
  __syncthreads();
  const uint32_t row = sm.sel_bin;
  __syncthreads();               // every thread has the row before sm is reused
  const int n_row = row != 0xFFFFFFFFu ? row_n(a, (int)row) : 0;
  // the assignment reads only the call's inputs (row lengths); the scores come
  // from the previous kernel
  pdl_wait();
  if (want_long) topk_row<kPackC>(a, sm, (int)row, kq, n_row);      // the whole cluster: c < n_long
  else if (row != 0xFFFFFFFFu) topk_row<1>(a, sm, (int)row, 0, n_row);
}

// ---------------------------------------------------------------------------
// Two-level candidate filter (CSA2 reading): blocks of 64 entries scored by
// their largest score, the first `blocks` of them by (block score desc, block
// index asc) kept, then the exact top-512 among the kept blocks' entries.  One
// CTA per row: block maxima from the L2-resident scores, an exact radix select
// of the B-th block key (ties to the lower block), the kept blocks' entries
// compacted in ascending order (only the row's last block can be ragged, so
// the candidate list is contiguous), an exact radix select of the 512th
// candidate, output in ascending order.
constexpr int kTwoMaxBlocks = 4096;        // rows up to 262144 entries
constexpr int kTwoMaxKept = 128;           // blocks kept: at most 8192 candidates
constexpr int kTwoCand = kTwoMaxKept * 64;

struct alignas(16) TwoSmem {
  uint32_t bkey[kTwoMaxBlocks];            // block maxima as order-preserving keys
  uint32_t cand_key[kTwoCand];
  int32_t kept[kTwoMaxKept];               // kept blocks, ascending
  uint32_t hist[2048];
  uint32_t warp_a[kWarps];
  uint32_t sel_bin, sel_need;
};

// Radix select of the need-th largest of `m` keys given by key_at (a block-wide
// three-pass 11/11/10-bit select): the key T and how many of those equal to T
// are taken (need - keys strictly above T).
template <typename F>
__device__ void two_radix(F key_at, int m, uint32_t need, TwoSmem& sm, uint32_t* T_out, uint32_t* take_out) {
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  uint32_t prefix = 0, mask = 0, rem = need;
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
  for (int p = 0; p < 3; ++p) {
    const int sh = shifts[p], nbv = 1 << widths[p];
    for (int i = tid; i < 2048; i += kThreads) sm.hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < m; i += kThreads) {
      const uint32_t k = key_at(i);
      if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> sh) & (uint32_t)(nbv - 1)], 1u);
    }
    __syncthreads();
    constexpr int per = 2048 / kThreads;
    uint32_t c[per], mine = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      const int b = per * tid + j;
      c[j] = b < nbv ? sm.hist[b] : 0u;
      mine += c[j];
    }
    uint32_t incl = mine;                       // suffix sums over higher threads
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, incl, o);
      if (lane + o < 32) incl += y;
    }
    if (lane == 0) sm.warp_a[warp] = incl;
    __syncthreads();
    uint32_t acc = incl - mine;
    for (int w2 = warp + 1; w2 < kWarps; ++w2) acc += sm.warp_a[w2];
#pragma unroll
    for (int j = per - 1; j >= 0; --j) {
      if (acc < rem && acc + c[j] >= rem) {
        sm.sel_bin = (uint32_t)(per * tid + j);
        sm.sel_need = rem - acc;
      }
      acc += c[j];
    }
    __syncthreads();
    prefix |= sm.sel_bin << sh;
    mask |= (uint32_t)(nbv - 1) << sh;
    rem = sm.sel_need;
    __syncthreads();
  }
  *T_out = prefix;
  *take_out = rem;
}

// Block-wide exclusive scan of one count per thread (512 threads).
__device__ __forceinline__ uint32_t two_scan(uint32_t v, uint32_t* total, TwoSmem& sm) {
  const int lane = lane_id(), warp = warp_id();
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm.warp_a[warp] = x;
  __syncthreads();
  uint32_t off = 0, tot = 0;
  for (int w2 = 0; w2 < kWarps; ++w2) {
    const uint32_t c = sm.warp_a[w2];
    if (w2 < warp) off += c;
    tot += c;
  }
  __syncthreads();
  *total = tot;
  return off + x - v;
}

__global__ void __launch_bounds__(kThreads) k_topk_two_level(TopkArgs a, int32_t blocks) {
  pdl_trigger();
  pdl_wait();                    // the scores come from the previous kernel
  extern __shared__ __align__(16) uint8_t smem[];
  TwoSmem& sm = *reinterpret_cast<TwoSmem*>(smem);
  const int r = blockIdx.x, tid = threadIdx.x;
  const float* row = a.scores + (size_t)r * a.ld;
  int32_t* out = a.out + (size_t)r * TOPK;
  int n = a.n_valid ? __ldg(a.n_valid + r) : (__ldg(a.row_pos + r) + 1) / a.P;
  if (n < 0 || n > a.max_n) {
    if (tid == 0) raise_flag(a.status, CSA_FLAG_ROW_INVALID);
    n = n < 0 ? 0 : a.max_n;
  }
  const int nb = (n + 63) / 64;
  // ---- block maxima (16-byte loads: a block is 64 consecutive scores) --------------
  for (int bl = tid; bl < nb; bl += kThreads) {
    const float4* p4 = reinterpret_cast<const float4*>(row + (size_t)bl * 64);
    const int cnt = min(64, n - bl * 64);
    float m = -INFINITY;
    if (cnt == 64) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 v = __ldg(p4 + j);
        m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
      }
    } else {
      for (int j = 0; j < cnt; ++j) m = fmaxf(m, __ldg(row + (size_t)bl * 64 + j));
    }
    sm.bkey[bl] = score_key(m == 0.0f ? 0.0f : m);
  }
  __syncthreads();
  // ---- the kept blocks: keys above the B-th, then equal keys by lower index --------
  const int kb = min(blocks, nb);
  uint32_t Tb = 0, take_b = (uint32_t)kb;
  if (kb < nb) two_radix([&](int i) { return sm.bkey[i]; }, nb, (uint32_t)kb, sm, &Tb, &take_b);
  {
    uint32_t eq_base = 0, kept_base = 0;
    for (int c0 = 0; c0 < nb; c0 += kThreads) {
      const int bl = c0 + tid;
      const uint32_t k = bl < nb ? sm.bkey[bl] : 0u;
      const uint32_t is_eq = (bl < nb && kb < nb && k == Tb) ? 1u : 0u;
      uint32_t tot_eq;
      const uint32_t eq_rank = eq_base + two_scan(is_eq, &tot_eq, sm);
      const uint32_t keep = (bl < nb && (kb >= nb || k > Tb || (is_eq && eq_rank < take_b))) ? 1u : 0u;
      uint32_t tot_keep;
      const uint32_t pos = kept_base + two_scan(keep, &tot_keep, sm);
      if (keep && pos < (uint32_t)kTwoMaxKept) sm.kept[pos] = bl;
      eq_base += tot_eq;
      kept_base += tot_keep;
    }
  }
  __syncthreads();
  // ---- candidates: the kept blocks' entries in ascending order ----------------------
  const int last_cnt = n - 64 * (nb - 1);                  // entries of the row's last block
  const int m = kb == 0 ? 0 : (sm.kept[kb - 1] == nb - 1 ? 64 * (kb - 1) + last_cnt : 64 * kb);
  for (int c = tid; c < m; c += kThreads) {
    const float v = __ldg(row + (size_t)sm.kept[c >> 6] * 64 + (c & 63));
    sm.cand_key[c] = score_key(v == 0.0f ? 0.0f : v);
  }
  __syncthreads();
  auto entry = [&](int c) { return sm.kept[c >> 6] * 64 + (c & 63); };
  if (m <= TOPK) {
    for (int i = tid; i < TOPK; i += kThreads) out[i] = i < m ? entry(i) : -1;
    return;
  }
  uint32_t T, take;
  two_radix([&](int i) { return sm.cand_key[i]; }, m, (uint32_t)TOPK, sm, &T, &take);
  uint32_t eq_base = 0, sel_base = 0;
  for (int c0 = 0; c0 < m; c0 += kThreads) {
    const int c = c0 + tid;
    const uint32_t k = c < m ? sm.cand_key[c] : 0u;
    const uint32_t is_eq = (c < m && k == T) ? 1u : 0u;
    uint32_t tot_eq;
    const uint32_t eq_rank = eq_base + two_scan(is_eq, &tot_eq, sm);
    const uint32_t sel = (c < m && (k > T || (is_eq && eq_rank < take))) ? 1u : 0u;
    uint32_t tot_sel;
    const uint32_t pos = sel_base + two_scan(sel, &tot_sel, sm);
    if (sel && pos < (uint32_t)TOPK) out[pos] = entry(c);
    eq_base += tot_eq;
    sel_base += tot_sel;
  }
}

}  // namespace

cudaError_t launch_topk_two_level(const TopkArgs& a, int32_t blocks, Order order, cudaStream_t stream) {
  if (a.num_rows <= 0) return cudaSuccess;
  const size_t smem = sizeof(TwoSmem);
  cudaError_t e = cudaFuncSetAttribute(k_topk_two_level, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(order, k_topk_two_level, dim3(a.num_rows), dim3(kThreads), smem, stream, a, blocks);
}

cudaError_t launch_topk(const TopkArgs& a, Order order, cudaStream_t stream) {
  if (a.num_rows <= 0) return cudaSuccess;
  const bool row_ok = (a.ld % 4) == 0 && ((uintptr_t)a.scores & 15u) == 0;
  if (row_ok && a.max_n > kPackLong && a.max_n <= kPackC * kPackLong) {
    // rows of up to 64K entries: long rows a cluster each, short ones a CTA each
    const size_t smem = sizeof(PackSmem);
    cudaError_t e = cudaFuncSetAttribute(k_topk_packed, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_rows * kPackC, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPackC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1 + order_attr(order, attr + 1);
    return cudaLaunchKernelEx(&cfg, k_topk_packed, a);
  }
  if (a.max_n <= kRowMax && row_ok) {
    // CTAs per row: about one per 8K entries, up to 8, at most two CTAs per
    // SM over the grid, rounded down to a power of two (measured on the
    // serving batch, 128 rows of up to 60K entries: 1 per row 34 us, 2 per
    // row 26 us, 4 per row 37 us, 8 per row 83 us)
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int C = (a.max_n + 8191) / 8192;
    C = C < 1 ? 1 : (C > kRowCluster ? kRowCluster : C);
    while (C > 1 && (long long)a.num_rows * C > 2LL * sms) --C;
    C = C >= 8 ? 8 : (C >= 4 ? 4 : (C >= 2 ? 2 : 1));             // a power of two
    void (*kern)(TopkArgs) = C == 8 ? k_topk_row<8> : (C == 4 ? k_topk_row<4> : (C == 2 ? k_topk_row<2> : k_topk_row<1>));
    const size_t smem = sizeof(RowSmem);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_rows * C, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1 + order_attr(order, attr + 1);
    return cudaLaunchKernelEx(&cfg, kern, a);
  }
  int C = (a.max_n + kStageMax - 1) / kStageMax;
  C = C < 1 ? 1 : (C > kMaxCluster ? kMaxCluster : C);
  // few rows: spread each row over more CTAs
  while (2 * C <= kMaxCluster && (a.max_n + 2 * C - 1) / (2 * C) >= 4096 && (long long)a.num_rows * C * 2 <= 300)
    C *= 2;
  const int slice_cap = (((a.max_n + C - 1) / C) + 3) & ~3;   // matches the kernel's 16-byte slices
  const int staged = slice_cap <= kStageMax;
  const size_t smem = sizeof(TopkSmem) + (staged ? (size_t)slice_cap * 4 : 0);
  cudaError_t e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, a.num_rows, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1 + order_attr(order, attr + 1);
  return cudaLaunchKernelEx(&cfg, k_topk, a, C, slice_cap, staged);
}

}  // namespace csa
