// csa_index_score: score[r, i] = sum_h w[r,h] * relu(qhat[r,h] . khat[i])
// over the paged MXFP4 indexer cache, as a block-scaled FP4 tcgen05 MMA.
//
// [SGL] "DeepSeek-V4.1 Flash on SGLang: from 35 to 873 tokens/s",
//   "Architecture changes and KV cache compression": the indexer K entries are
//   FP4 (68 B) and the indexer picks the top 512 global positions;
//   "DSpark adaptation and optimization": the valid-length check is fused with
//   candidate handling (rows only score their visible entries).
//
// Two kernels:
//  k_score_prep  block 0 builds the segment table (a segment = up to
//                `group_rows` consecutive rows of one request that see at
//                least one entry, scored by one MMA N dimension) and each
//                score CTA's first segment; blocks 1..R quantise each row's
//                q_idx to MXFP4 straight into the shared-memory image the MMA
//                reads.
//  k_index_score persistent, one CTA per SM.  A work table of (segment, tile,
//                pages) items is built in shared memory first, so no role
//                touches global metadata per tile.  Roles:
//                4 producer warps  one bulk copy per indexer page (4352 B: the
//                        page layout is already the MMA operand layout), two
//                        pages = one 128-entry tile per stage, 20 stages; several
//                        warps feed the copy engine because one warp's copy
//                        issue rate caps its bandwidth.
//                3 MMA warps, one per reduction group, each walking its
//                        group's tiles in order: gathers a tile's
//                        E8M0 bytes into the tcgen05 scale-factor atom, and one
//                        lane issues tcgen05.cp of the scales and two kind::mxf4
//                        MMAs (K = 64 each): A = 128 entries x 128 dims, B =
//                        rows*heads x 128 dims, D = fp32 [entry lane,
//                        row*head column] in an accumulator of the tile's group.
//                3 reduction warpgroups  tile t goes to group t mod 3, which
//                        owns two TMEM accumulators: the MMA of its next tile
//                        runs while its four warps (one per TMEM lane quarter)
//                        reduce the current one, per entry lane
//                        sum_h w*relu(D) with packed fp32x2 fused multiply-adds
//                        in four independent chains, then coalesced fp32 score
//                        stores.  Each warp waits for the accumulator and frees
//                        it on its own: no barrier couples the warps of a group
//                        or the groups to their MMA warp beyond the accumulator
//                        hand-off itself.  (One issuing warp alone could not keep
//                        up: the per-tile issue path, from the page's arrival to
//                        the MMAs, takes several hundred cycles.)
//
// Every wait is bounded by the call's wait budget (SM clocks).  A wait that
// runs out raises CSA_FLAG_TIMEOUT and stops the CTA's pipeline; before the
// CTA exits it waits (with the default budget) for every bulk copy and tcgen05
// operation it issued, then frees its TMEM.
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

struct Seg {
  int32_t b, r0, nrows, n;
};

constexpr int kStages = 20;
constexpr int kGroups = 3;                         // reduction warpgroups, one MMA warp each
constexpr int kMma0 = 0;                           // MMA warps 0..2 (warp g serves group g)
constexpr int kCons0 = 4;                          // reduction warps 4..15
constexpr int kProducers = 4;                      // producer warps 3, 16, 17, 18
constexpr int kWarps = kCons0 + 4 * kGroups + kProducers - 1;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxAcc = 2 * kGroups;               // TMEM accumulators in flight
__host__ __device__ constexpr int producer_of_warp(int w) {
  return w == 3 ? 0 : (w >= kCons0 + 4 * kGroups ? 1 + w - (kCons0 + 4 * kGroups) : -1);
}
constexpr int kTileEntries = 128;
constexpr int kStageA = 2 * IDX_PAGE;              // two whole pages = 16 groups of 544 B
constexpr int kMaxN = CSA_MAX_ROW_GROUP_COLS;      // rows x padded heads per MMA (128)
constexpr int kQData = kMaxN * 64;                 // 8192
constexpr int kQSF = kMaxN * 4;                    // 512
constexpr int kItemCap = 256;                      // work items per table chunk
constexpr int kMaxGroupRows = kMaxN / 8;           // rows per segment (8 heads at least)
static_assert(kStages % kProducers == 0, "a stage belongs to one producer warp");
static_assert(kGroups < kStages, "an MMA warp's stage index wraps at most once per step");
static_assert(kMaxN == 128, "one scale-factor atom and one MMA N chunk per segment");
// TMEM columns: q scale factors (2 parities x 4), then 4 per accumulator for the
// tile's scale factors, then the accumulators.
constexpr int kTmemSFB = 0, kTmemSFA = 8, kTmemD = kTmemSFA + 4 * kMaxAcc;

struct Item {
  int32_t seg, tile, pg0, pg1;       // local segment index, tile in segment, pages (-1: none)
};

struct ScoreSmem {
  uint8_t qdata[2][kQData];                    // 1024-aligned (64-byte swizzle)
  uint8_t a[kStages][kStageA];                 // 16-aligned (8704 = 544 * 16)
  uint8_t sfb_raw[2][kQSF];
  uint8_t sfb_atom[2][kQSF];
  uint8_t sfa_atom[kStages][512];              // a stage's scale atom, rewritten after the stage is refilled
  Item items[kItemCap];
  Seg segs[kItemCap];
  int32_t pref[kItemCap + 1];
  alignas(16) float wseg[4 * kGroups][kMaxN];  // per consumer warp: row kr's w at kr * Hp
  int32_t rown[4 * kGroups][kMaxGroupRows];
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[kMaxAcc], acc_empty[kMaxAcc];
  uint64_t qfull[2], qempty[2], qready[2];
  uint64_t drain[kGroups];
  int32_t q_last[2];                           // latest segment whose q was loaded into each buffer
  int32_t q_next;                              // the segment whose q load goes out next
  uint32_t tmem_base;
  int32_t abort_flag;
};

static_assert(sizeof(ScoreSmem) + 1024 <= 227 * 1024, "one CTA per SM, within the opt-in shared memory");

__host__ __device__ inline int hi_pad(int Hi) { return (Hi + 7) & ~7; }
// MMA N for a group of N score columns: a multiple of 16, at least 64
// (columns past N multiply stale rows of the B buffer and are never read).
__host__ __device__ inline int mma_n(int N) { return N < 64 ? 64 : (N + 15) & ~15; }

// Reduction groups and accumulators per group for accumulators of `cols`
// TMEM columns: two per group (the next tile's MMA overlaps the current
// reduction) when six fit, else as many groups as accumulators fit.
__host__ __device__ inline void score_groups(int cols, int* G, int* NB) {
  int A = (512 - kTmemD) / cols;
  A = A < kMaxAcc ? A : kMaxAcc;
  if (A >= 2 * kGroups) { *G = kGroups; *NB = 2; }
  else if (A >= 4) { *G = 2; *NB = 2; }
  else { *G = A < 1 ? 1 : (A > kGroups ? kGroups : A); *NB = 1; }
}

// Workspace carve-out of the score step (after the status word).
constexpr int kMaxGrid = 1024;

struct ScoreWs {
  int32_t* nseg;       // [0] segments, [1] total work items (128-entry tiles)
  int32_t* cta_seg;    // [kMaxGrid] segment holding each score CTA's first item
  Seg* seg;            // [R]
  int32_t* tile_pref;  // [R + 1]
  uint8_t* qimg;       // [R * Hi_pad * 64]
  uint8_t* qsf;        // [R * Hi_pad * 4]
};

__device__ __host__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline ScoreWs carve_score_ws(uint8_t* base, int R, int Hi) {
  ScoreWs w;
  size_t o = kStatusBytes;
  w.nseg = reinterpret_cast<int32_t*>(base + o);
  o = align256(o + 16);
  w.cta_seg = reinterpret_cast<int32_t*>(base + o);
  o = align256(o + sizeof(int32_t) * kMaxGrid);
  w.seg = reinterpret_cast<Seg*>(base + o);
  o = align256(o + sizeof(Seg) * (size_t)(R > 0 ? R : 1));
  w.tile_pref = reinterpret_cast<int32_t*>(base + o);
  o = align256(o + sizeof(int32_t) * (size_t)(R + 1));
  w.qimg = base + o;
  o = align256(o + (size_t)R * hi_pad(Hi) * 64);
  w.qsf = base + o;
  return w;
}

__device__ __forceinline__ int lower_bound_req(const int32_t* row_req, int R, int v) {
  int lo = 0, hi = R;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(row_req + mid) < v) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Block-wide exclusive scan of one int per thread (blockDim = 128).
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* sm_warp) {
  const int lane = lane_id(), w = warp_id();
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm_warp[w] = x;
  __syncthreads();
  int off = 0, tot = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
    if (i < w) off += sm_warp[i];
    tot += sm_warp[i];
  }
  __syncthreads();
  *total = tot;
  return off + x - v;
}

// Launched in plain stream order as its call's first kernel, or chained after
// the step's cache append (csa_step), beside which it runs: it reads only the
// call's inputs and writes only the score workspace.  It waits for the
// previous kernel before it exits, so that everything after it also sees
// that kernel's writes.
__global__ void __launch_bounds__(128) k_score_prep(ScoreArgs a, uint8_t* ws) {
  pdl_trigger();
  const int R = a.num_rows, Hi = a.Hi, Hp = hi_pad(Hi);
  ScoreWs W = carve_score_ws(ws, R, Hi);
  if (blockIdx.x == 0) {
    // ---- segment table: rows grouped by request, at most group_rows per
    // segment; segments whose rows see no entry are left out, so every segment
    // has at least one tile
    __shared__ int sm_warp[4];
    __shared__ int carry_seg;
    if (threadIdx.x == 0) carry_seg = 0;
    __syncthreads();
    for (int base = 0; base < R; base += 128) {
      const int r = base + threadIdx.x;
      int keep = 0;
      Seg s;
      if (r < R) {
        const int b = __ldg(a.row_req + r);
        if (b < 0 || b >= a.num_requests || (r > 0 && __ldg(a.row_req + r - 1) > b))
          raise_flag(a.status, CSA_FLAG_ROW_INVALID);
        const int k_in_req = r - lower_bound_req(a.row_req, R, b);
        if (k_in_req >= 0 && (k_in_req % a.group_rows) == 0) {
          const int rend = lower_bound_req(a.row_req, R, b + 1);
          const int nrows = max(0, min(a.group_rows, rend - r));
          int n = 0;
          for (int k = 0; k < nrows; ++k) n = max(n, (__ldg(a.row_pos + r + k) + 1) / a.P);
          const int cap = min(a.max_entries, a.max_pages * PAGE);
          if (n > cap) {
            raise_flag(a.status, CSA_FLAG_ROW_INVALID);
            n = cap;
          }
          if (b < 0 || b >= a.num_requests) n = 0;
          s.b = b; s.r0 = r; s.nrows = nrows; s.n = n;
          keep = n > 0 ? 1 : 0;
        }
      }
      int tot;
      const int sid = block_exclusive_scan(keep, &tot, sm_warp) + carry_seg;
      if (keep) W.seg[sid] = s;
      __syncthreads();
      if (threadIdx.x == 0) carry_seg += tot;
      __syncthreads();
    }
    const int S = carry_seg;
    // ---- tile prefix over segments
    __shared__ int carry_t;
    if (threadIdx.x == 0) carry_t = 0;
    __syncthreads();
    for (int base = 0; base < S; base += 128) {
      const int s = base + threadIdx.x;
      const int t = (s < S) ? (W.seg[s].n + kTileEntries - 1) / kTileEntries : 0;
      int tot;
      const int ex = block_exclusive_scan(t, &tot, sm_warp) + carry_t;
      if (s < S) W.tile_pref[s] = ex;
      __syncthreads();
      if (threadIdx.x == 0) carry_t += tot;
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      W.tile_pref[S] = carry_t;
      W.nseg[0] = S;
      W.nseg[1] = carry_t;
    }
    __syncthreads();
    // first segment of every score CTA's contiguous item range
    const int total = carry_t;
    const int per = (total + a.grid - 1) / a.grid;
    for (int g = threadIdx.x; g < a.grid; g += blockDim.x) {
      const int item = g * per;
      int seg = S;
      if (item < total) {
        int lo = 0, hi = S - 1;              // largest s with tile_pref[s] <= item
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (W.tile_pref[mid] <= item) lo = mid; else hi = mid - 1;
        }
        seg = lo;
      }
      W.cta_seg[g] = seg;
    }
    pdl_wait();
    return;
  }
  // ---- MXFP4 quantisation of row r's indexer queries into the MMA B image.
  // Head h of row r is image row n = r*Hp + h; its 4 blocks of 32 values are
  // the 4 16-byte chunks of a 64-byte row, stored with the 64-byte swizzle
  // (chunk c at c ^ ((n >> 1) & 3)) that the MMA descriptor expects.
  const int r = blockIdx.x - 1;
  for (int job = threadIdx.x; job < Hp * 4; job += blockDim.x) {
    const int h = job >> 2, kb = job & 3;
    const size_t n = (size_t)r * Hp + h;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    uint32_t E8 = 0u;
    if (h < Hi) {
      const uint4* src = reinterpret_cast<const uint4*>(a.q_idx + ((size_t)r * Hi + h) * DI + kb * 32);
      float v[32];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = __ldg(src + i);
        const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[8 * i + 2 * k] = __uint_as_float(ww[k] << 16);
          v[8 * i + 2 * k + 1] = __uint_as_float(ww[k] & 0xFFFF0000u);
        }
      }
      float am = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(v[i]));
      E8 = e8m0_block_code(am);
      if (am != 0.0f) {
        const float inv = e8m0_inv_scale(E8);
        uint32_t wv[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 32; ++i) wv[i >> 3] |= e2m1_rne(v[i] * inv) << (4 * (i & 7));
        out = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
    }
    const int sw = kb ^ (int)((n >> 1) & 3);
    *reinterpret_cast<uint4*>(W.qimg + n * 64 + sw * 16) = out;
    W.qsf[n * 4 + kb] = (uint8_t)E8;
  }
  pdl_wait();
}

// Rearrange 4-byte scale words of up to 128 rows into the tcgen05 scale-factor
// atom: the word of row m goes to word 4*(m % 32) + m / 32 (32 rows x 16 B,
// row m%32 holding the words of rows m%32, +32, +64, +96).
__device__ __forceinline__ void sf_to_atom(const uint8_t* raw, uint8_t* atom, int lane) {
  const uint32_t* src = reinterpret_cast<const uint32_t*>(raw);
  uint4 v;
  v.x = src[lane];
  v.y = src[lane + 32];
  v.z = src[lane + 64];
  v.w = src[lane + 96];
  reinterpret_cast<uint4*>(atom)[lane] = v;
}

__device__ __forceinline__ float relu(uint32_t bits) { return fmaxf(__uint_as_float(bits), 0.0f); }
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo_f32(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f32(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
// d = a * b + c on both fp32 halves, each rounded once
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// One thread's bounded wait; on time-out the CTA's pipeline is stopped.
template <bool kPoll>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, ScoreSmem& sm, const ScoreArgs& a) {
  if (mbar_wait_for<kPoll>(bar, parity, a.wait_budget)) return true;
  raise_flag(a.status, CSA_FLAG_TIMEOUT);
  atomicExch(&sm.abort_flag, 1);
  return false;
}

// Whole-warp wait: every lane probes the barrier and the warp leaves at once
// when all see the phase complete (the usual case on the per-tile path: one
// probe and one vote, no hand-off from a polling lane); otherwise every lane
// waits and the warp agrees on the outcome, so a time-out never leaves some
// lanes of a warp inside the loop and others out.
template <bool kPoll>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, ScoreSmem& sm, const ScoreArgs& a) {
  if (__all_sync(0xFFFFFFFFu, mbar_try_wait_poll(bar, parity))) return true;
  const int ok = wait_or_abort<kPoll>(bar, parity, sm, a) ? 1 : 0;
  return __all_sync(0xFFFFFFFFu, ok) != 0;
}

// A producer's wait for a free stage: the pipeline is usually full, so it
// backs off between probes instead of taking issue slots from the consumers.
__device__ __forceinline__ bool producer_wait(uint64_t* bar, uint32_t parity, ScoreSmem& sm, const ScoreArgs& a) {
  if (mbar_try_wait_poll(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_poll(bar, parity)) {
    __nanosleep(64);
    if (clock64() - t0 > a.wait_budget) {
      raise_flag(a.status, CSA_FLAG_TIMEOUT);
      atomicExch(&sm.abort_flag, 1);
      return false;
    }
  }
  return true;
}

// A producer's bounded wait for its turn to load segment ord's q image.
__device__ __forceinline__ bool producer_wait_turn(const int32_t* next, int ord, ScoreSmem& sm, const ScoreArgs& a) {
  const volatile int32_t* v = next;
  if (*v == ord) return true;
  const long long t0 = clock64();
  while (*v != ord) {
    __nanosleep(64);
    if (clock64() - t0 > a.wait_budget || *reinterpret_cast<volatile int32_t*>(&sm.abort_flag)) {
      raise_flag(a.status, CSA_FLAG_TIMEOUT);
      atomicExch(&sm.abort_flag, 1);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool aborted(const ScoreSmem& sm) {
  return *reinterpret_cast<const volatile int32_t*>(&sm.abort_flag) != 0;
}

__global__ void __launch_bounds__(kThreads, 1) k_index_score(ScoreArgs a, uint8_t* ws) {
  extern __shared__ uint8_t smem_raw[];
  ScoreSmem& sm = *reinterpret_cast<ScoreSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int Hi = a.Hi, Hp = hi_pad(Hi);
  ScoreWs W = carve_score_ws(ws, a.num_rows, Hi);
  const int warp = warp_id(), lane = lane_id(), tid = threadIdx.x;
  const uint8_t* ipool = static_cast<const uint8_t*>(a.idx_pool);

  const int cols = mma_n(a.group_rows * Hp);           // TMEM columns of one accumulator
  int G, NB;
  score_groups(cols, &G, &NB);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int d = 0; d < kMaxAcc; ++d) {
      mbar_init(&sm.acc_full[d], 1);
      mbar_init(&sm.acc_empty[d], 4);           // the four warps of the owning group
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&sm.qfull[d], 1);
      mbar_init(&sm.qempty[d], G);             // every MMA warp leaves each segment once
      mbar_init(&sm.qready[d], 1);
    }
    for (int g = 0; g < kGroups; ++g) mbar_init(&sm.drain[g], 1);
    sm.q_last[0] = sm.q_last[1] = -1;
    sm.q_next = 0;
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  pdl_wait();                    // the segment table, q image and pages are ready from here on
  // Dependents start only once every score CTA is past its wait, i.e. after
  // the score prep and whatever it waited for (a step's cache append): the
  // attention step reads the appended window and pages before its own wait.
  pdl_trigger();

  const int S = W.nseg[0], total = W.nseg[1];
  const int per = (total + gridDim.x - 1) / gridDim.x;
  const int beg = min(total, (int)blockIdx.x * per), end = min(total, beg + per);

  // Role state kept across work chunks.  Segments are numbered in this CTA's
  // item order (ord = 0, 1, ...; every segment has a tile); ord picks the q
  // buffer (ord & 1) and the phases of the q barriers.
  const int prod = producer_of_warp(warp);
  const int grp = (warp >= kCons0 && warp < kCons0 + 4 * kGroups) ? (warp - kCons0) >> 2 : -1;
  const bool cons = grp >= 0 && grp < G;
  const int mg = warp - kMma0;                             // MMA warp of group mg
  const bool mma_warp = mg >= 0 && mg < G && warp < kMma0 + kGroups;
  int p_last_it = -1;                                      // producer: last item copied
  int l_ord = -1, l_par = 0, l_desc_ord = -1;             // MMA warp: segment entered, descriptors
  uint64_t l_bdesc = 0;
  uint32_t l_id0 = 0, l_id1 = 0;
  bool l_issued = false;
  int e_gseg = -1;                                         // consumer warp: segment staged
  int ord_base = 0;                                        // ordinal of the window's first segment

  int seg0 = (beg < end) ? W.cta_seg[blockIdx.x] : S;
  int it_base = 0;
  for (int c0 = beg; c0 < end;) {
    // ---- work table for items [c0, c1): local segment window, pages -----------
    const int nsw = min(S - seg0, kItemCap);
    for (int j = tid; j <= nsw; j += kThreads) sm.pref[j] = W.tile_pref[seg0 + j];
    for (int j = tid; j < nsw; j += kThreads) sm.segs[j] = W.seg[seg0 + j];
    __syncthreads();
    const int c1 = min(min(end, c0 + kItemCap), sm.pref[nsw]);
    const int m = c1 - c0;
    for (int i = tid; i < m; i += kThreads) {
      const int item = c0 + i;
      int lo = 0, hi = nsw - 1;              // largest j with pref[j] <= item
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm.pref[mid] <= item) lo = mid; else hi = mid - 1;
      }
      const Seg sg = sm.segs[lo];
      const int tile = item - sm.pref[lo];
      const int npages = (sg.n + PAGE - 1) / PAGE;
      int pg[2] = {-1, -1};
      for (int h = 0; h < 2; ++h) {
        const int lp = 2 * tile + h;
        if (lp < npages) {
          const int p = __ldg(a.page_table + (size_t)sg.b * a.max_pages + lp);
          if (p >= 0 && p < a.num_pages) pg[h] = p;
          else raise_flag(a.status, CSA_FLAG_PAGE_OOB);
        }
      }
      Item e;
      e.seg = lo;
      e.tile = tile;
      e.pg0 = pg[0];
      e.pg1 = pg[1];
      sm.items[i] = e;
    }
    __syncthreads();

    if (prod >= 0) {
      if (lane == 0) {
        // ================= producers: items it with it % kProducers == prod =================
        int i = prod - (it_base % kProducers);
        if (i < 0) i += kProducers;
        for (; i < m; i += kProducers) {
          if (aborted(sm)) break;
          const int it = it_base + i;
          const Item e = sm.items[i];
          const int ord = ord_base + e.seg;
          // the first item of a segment in this CTA loads its q image (a chunk's
          // first item continues the previous chunk's last segment when e.seg == 0)
          const bool first = (i > 0) ? (sm.items[i - 1].seg != e.seg) : (it_base == 0 || e.seg != 0);
          if (first) {
            const Seg sg = sm.segs[e.seg];
            const int par = ord & 1;
            // The q loads go out in segment order (segment ord - 1's first,
            // whichever producer has it), so the release of buffer par that this
            // load waits for is at most one phase ahead of the barrier: a parity
            // wait cannot tell phase k from phase k - 2.  The producer of ord - 1
            // never waits on this one: every item before this one is issued.
            if (!producer_wait_turn(&sm.q_next, ord, sm, a)) break;
            if (ord >= 2 && !producer_wait(&sm.qempty[par], ((ord >> 1) - 1) & 1, sm, a)) break;
            const uint32_t bytes_d = (uint32_t)(sg.nrows * Hp * 64), bytes_s = (uint32_t)(sg.nrows * Hp * 4);
            mbar_expect_tx(&sm.qfull[par], bytes_d + bytes_s);
            bulk_load(sm.qdata[par], W.qimg + (size_t)sg.r0 * Hp * 64, bytes_d, &sm.qfull[par]);
            bulk_load(sm.sfb_raw[par], W.qsf + (size_t)sg.r0 * Hp * 4, bytes_s, &sm.qfull[par]);
            sm.q_last[par] = ord;                    // loads into one buffer are ordered by qempty
            *reinterpret_cast<volatile int32_t*>(&sm.q_next) = ord + 1;
          }
          const int s = it % kStages, use = it / kStages;
          if (use > 0 && !producer_wait(&sm.empty[s], (use - 1) & 1, sm, a)) break;
          const uint32_t bytes = (e.pg0 >= 0 ? (uint32_t)IDX_PAGE : 0u) + (e.pg1 >= 0 ? (uint32_t)IDX_PAGE : 0u);
          mbar_expect_tx(&sm.full[s], bytes);
          if (e.pg0 >= 0) bulk_load(sm.a[s], ipool + (size_t)e.pg0 * IDX_PAGE, IDX_PAGE, &sm.full[s]);
          if (e.pg1 >= 0) bulk_load(sm.a[s] + IDX_PAGE, ipool + (size_t)e.pg1 * IDX_PAGE, IDX_PAGE, &sm.full[s]);
          p_last_it = it;
        }
      }
      __syncwarp();
    } else if (mma_warp) {
      // ================= MMA warp mg: the items of group mg =================
      const uint32_t sfb_t = tmem + kTmemSFB;
      const uint64_t adesc0 = smem_desc(smem_u32(sm.a[0]), 128, IDX_GROUP, kSwizzleNone);
      bool ok = true;
      // Enter every segment up to ordinal `ord` in order.  Every MMA warp
      // enters every segment of the CTA's range (so each q buffer is released
      // by all of them, and the warp that copies a segment's q scales to TMEM
      // always reaches it), whether or not its group has a tile there.
      auto enter_upto = [&](int ord) -> bool {
        while (l_ord < ord) {
          const int o = l_ord + 1;
          // leaving l_ord: its q buffer is free once this warp's MMAs complete
          if (l_ord >= 0 && lane == 0) tc_commit(&sm.qempty[l_ord & 1]);
          const int par = o & 1;
          if (!warp_wait<true>(&sm.qfull[par], (o >> 1) & 1, sm, a)) return false;
          if (o % G == mg) {
            // one warp per segment lays the q scales out as an atom and copies it
            // to TMEM; the commit tells the others the copy has landed.  Rows
            // past N inside the atom hold stale bytes; their D columns are never read.
            sf_to_atom(sm.sfb_raw[par], sm.sfb_atom[par], lane);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tc_fence_after();
              tmem_cp_32x128b_x4(sfb_t + 4 * par, smem_desc(smem_u32(sm.sfb_atom[par]), 16, 128, kSwizzleNone));
              tc_commit(&sm.qready[par]);
            }
            __syncwarp();
          }
          if (!warp_wait<true>(&sm.qready[par], (o >> 1) & 1, sm, a)) return false;
          l_ord = o;
          l_issued = true;
        }
        return true;
      };
      int i = mg - (it_base % G);
      if (i < 0) i += G;
      // carried per-tile state (i steps by G): the group's tile u = it / G,
      // its slot u % NB and phase (u / NB) & 1, the stage it % kStages and
      // that stage's use it / kStages
      int m_u, m_ub, m_ph, m_s, m_use;
      {
        const int it = it_base + i;
        m_u = it / G;
        m_ub = m_u % NB;
        m_ph = (m_u / NB) & 1;
        m_s = it % kStages;
        m_use = it / kStages;
      }
      for (; i < m; i += G) {
        if (aborted(sm)) { ok = false; break; }
        const Item e = sm.items[i];
        const int ord = ord_base + e.seg;
        if (l_desc_ord != ord) {                    // B operand and N of this segment
          if (!enter_upto(ord)) { ok = false; break; }
          const int N = sm.segs[e.seg].nrows * Hp;
          l_par = ord & 1;
          l_bdesc = smem_desc(smem_u32(sm.qdata[l_par]), 16, 512, kSwizzle64B);
          l_id0 = idesc_mxf4(128, (uint32_t)mma_n(N), 0, 0);
          l_id1 = idesc_mxf4(128, (uint32_t)mma_n(N), 2, 2);
          l_desc_ord = ord;
        }
        const int u = m_u;                           // the tile's index within its group
        const int slot = mg * NB + m_ub;
        const uint32_t empty_par = (uint32_t)(m_ph ^ 1);   // the slot's previous use, u - NB
        const int s = m_s, use = m_use;
        ++m_u;
        if (++m_ub == NB) { m_ub = 0; m_ph ^= 1; }
        m_s += G;                                    // G < kStages: wraps at most once
        if (m_s >= kStages) { m_s -= kStages; ++m_use; }
        if (!warp_wait<true>(&sm.full[s], use & 1, sm, a)) { ok = false; break; }
        // the tile's scale words: entry row r is page r / 64, group (r % 64) / 8, word r % 8
        {
          const uint8_t* st = sm.a[s];
          uint32_t wv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = lane + 32 * j;
            wv[j] = *reinterpret_cast<const uint32_t*>(st + (r >> 6) * IDX_PAGE + idx_scale_off(r & 63, 0));
          }
          reinterpret_cast<uint4*>(sm.sfa_atom[s])[lane] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        // the accumulator's previous tile has been reduced by its four warps
        if (u >= NB && !warp_wait<true>(&sm.acc_empty[slot], empty_par, sm, a)) { ok = false; break; }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sfa = tmem + kTmemSFA + 4 * slot;
          tmem_cp_32x128b_x4(sfa, smem_desc(smem_u32(sm.sfa_atom[s]), 16, 128, kSwizzleNone));
          // A: the two pages as they landed: 8-entry groups IDX_GROUP apart, 16-byte
          // core matrices 128 B apart along K (no swizzle); second K half at +256 B
          const uint64_t ad = adesc0 + (uint64_t)(s * (kStageA >> 4));
          const uint32_t dcol = tmem + kTmemD + slot * cols;
          const uint32_t sfb = sfb_t + 4 * l_par;
          mma_mxf4(dcol, ad, l_bdesc, l_id0, sfa, sfb, 0u);
          mma_mxf4(dcol, ad + 16, l_bdesc + 2, l_id1, sfa, sfb, 1u);
          tc_commit(&sm.empty[s]);
          tc_commit(&sm.acc_full[slot]);
        }
        __syncwarp();
        l_issued = true;
      }
      // the chunk's segments past the group's last tile
      if (ok && !aborted(sm)) enter_upto(ord_base + sm.items[m - 1].seg);
    } else if (cons) {
      // ================= reduction group grp: items it with it % G == grp =================
      const int q = warp & 3;                       // TMEM lane quarter of this warp
      const int mrow = 32 * q + lane;               // entry within the tile
      const int cw = warp - kCons0;
      float* ew = sm.wseg[cw];                      // this warp's copy of the segment's w
      int32_t* en = sm.rown[cw];                    // and of its rows' visible lengths
      int i = grp - (it_base % G);
      if (i < 0) i += G;
      // item it = it_base + i is the group's tile u = it / G, in accumulator
      // slot u % NB with phase (u / NB) & 1; i steps by G, so u steps by one
      // and both are carried instead of divided out per tile
      int c_ub, c_ph;
      {
        const int u = (it_base + i) / G;
        c_ub = u % NB;
        c_ph = (u / NB) & 1;
      }
      for (; i < m; i += G) {
        if (aborted(sm)) break;
        const Item e = sm.items[i];
        const Seg sg = sm.segs[e.seg];
        const int gseg = seg0 + e.seg;
        if (gseg != e_gseg) {                       // stage this segment's weights and row lengths
          __syncwarp();
          for (int x = lane; x < sg.nrows * Hi; x += 32) ew[(x / Hi) * Hp + x % Hi] = __ldg(a.w + (size_t)sg.r0 * Hi + x);
          for (int x = lane; x < sg.nrows; x += 32) en[x] = (__ldg(a.row_pos + sg.r0 + x) + 1) / a.P;
          __syncwarp();
          e_gseg = gseg;
        }
        const int slot = grp * NB + c_ub;
        const uint32_t full_par = (uint32_t)c_ph;
        if (++c_ub == NB) { c_ub = 0; c_ph ^= 1; }
        if (!warp_wait<true>(&sm.acc_full[slot], full_par, sm, a)) break;
        tc_fence_after();
        const int ient = e.tile * kTileEntries + mrow;
        const bool page_ok = (mrow < 64) ? (e.pg0 >= 0) : (e.pg1 >= 0);
        const uint32_t dbase = tmem + ((uint32_t)(32 * q) << 16) + kTmemD + slot * cols;
        for (int kr = 0; kr < sg.nrows; ++kr) {
          const float* wr = ew + kr * Hp;
          // four independent (even head, odd head) fp32x2 chains, +0.0f each
          uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
          float acc1 = 0.0f;                        // heads past the last full group of 32
          int h0 = 0;
          for (; h0 + 32 <= Hi; h0 += 32) {
            uint32_t v[32];
            tmem_ld32(dbase + kr * Hp + h0, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 w4 = *reinterpret_cast<const float4*>(wr + h0 + j);
              uint64_t& c = acc2[(j >> 2) & 3];
              c = ffma2(pack2(w4.x, w4.y), pack2(relu(v[j]), relu(v[j + 1])), c);
              c = ffma2(pack2(w4.z, w4.w), pack2(relu(v[j + 2]), relu(v[j + 3])), c);
            }
          }
          for (; h0 < Hi; h0 += 16) {
            uint32_t v[16];
            tmem_ld16(dbase + kr * Hp + h0, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (h0 + j < Hi) acc1 = fmaf(wr[h0 + j], relu(v[j]), acc1);
          }
          const float s0 = lo_f32(acc2[0]) + hi_f32(acc2[0]), s1 = lo_f32(acc2[1]) + hi_f32(acc2[1]);
          const float s2 = lo_f32(acc2[2]) + hi_f32(acc2[2]), s3 = lo_f32(acc2[3]) + hi_f32(acc2[3]);
          const float acc = ((s0 + s1) + (s2 + s3)) + acc1;
          if (ient < en[kr] && ient < sg.n)
            a.scores[(size_t)(sg.r0 + kr) * a.ld + ient] = page_ok ? acc : -INFINITY;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[slot]);
      }
    }
    // ---- chunk done: every role has finished with this work table ----------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int last_seg = sm.items[m - 1].seg;
    ord_base += last_seg;
    seg0 += last_seg;
    it_base += m;
    c0 = c1;
    __syncthreads();
    if (aborted(sm)) break;                         // read after a barrier: uniform
  }

  // ---- drain: every bulk copy this CTA issued has landed and every tcgen05
  // operation has completed before shared memory and TMEM are released.  A
  // stage belongs to one producer warp, so its latest use is that warp's; a q
  // buffer is reloaded only after every group waited for its previous load,
  // so only the latest load into each buffer can still be in flight.
  __syncthreads();
  if (prod >= 0 && lane == 0) {
    for (int k = 0; k < kStages / kProducers; ++k) {
      const int it = p_last_it - kProducers * k;   // this producer's most recent use of each of its stages
      if (it < 0) break;
      if (!mbar_wait(&sm.full[it % kStages], (it / kStages) & 1)) raise_flag(a.status, CSA_FLAG_TIMEOUT);
    }
    if (prod < 2) {                                 // producers 0 and 1 drain q buffers 0 and 1
      const int ql = sm.q_last[prod];
      if (ql >= 0 && !mbar_wait(&sm.qfull[ql & 1], (ql >> 1) & 1)) raise_flag(a.status, CSA_FLAG_TIMEOUT);
    }
  }
  if (mma_warp && lane == 0 && l_issued) {
    tc_commit(&sm.drain[mg]);
    if (!mbar_wait(&sm.drain[mg], 0)) raise_flag(a.status, CSA_FLAG_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t score_ws_bytes(int32_t R, int32_t Hi) {
  ScoreWs w = carve_score_ws(nullptr, R, Hi);
  return reinterpret_cast<size_t>(w.qsf) + align256((size_t)R * hi_pad(Hi) * 4);
}

// Rows of one request scored by one MMA: as many as keep the MMA's N (rows x
// padded heads) within kMaxN; the score kernel then keeps at least three
// accumulators in flight (six, two per consumer group, when N <= 80).
int score_group_rows(int32_t Hi, int32_t max_rows_per_req) {
  int g = kMaxN / hi_pad(Hi);
  if (g > kMaxGroupRows) g = kMaxGroupRows;
  if (max_rows_per_req >= 1 && g > max_rows_per_req) g = max_rows_per_req;
  return g < 1 ? 1 : g;
}

cudaError_t launch_index_score(const ScoreArgs& a, int num_sms, Order prep_order, cudaStream_t stream) {
  if (a.num_rows <= 0) return cudaSuccess;
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.status);
  ScoreArgs ap = a;
  ap.grid = num_sms < kMaxGrid ? num_sms : kMaxGrid;
  // the prep reads the call's inputs and overwrites the workspace at once:
  // plain stream order when it is the call's first kernel, chained only after
  // a kernel of the same call that touches neither (the step's append)
  cudaError_t e = launch_kernel(prep_order, k_score_prep, dim3(1 + a.num_rows), dim3(128), 0, stream, ap, ws);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(ScoreSmem) + 1024;
  e = cudaFuncSetAttribute(k_index_score, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(Order::kChained, k_index_score, dim3(ap.grid), dim3(kThreads), smem, stream, ap, ws);
}

}  // namespace csa
