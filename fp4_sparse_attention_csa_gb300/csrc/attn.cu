// csa_sparse_attn: MQA softmax attention of each row's heads over the
// selected FP4 main-KV entries plus the FP8 local window.
//
// [SGL] "DeepSeek-V4.1 Flash on SGLang: from 35 to 873 tokens/s",
//   "Architecture changes and KV cache compression": only the top 512 global
//   positions take part in attention; main-KV entries are FP4 (288 B);
//   "DSpark adaptation and optimization": KV page address translation is done
//   in the same step as the post-top-k validity filter.
// [VLLM] "DeepSeek-V4.1-Flash runs 5.3x faster on vLLM...", "SWA bounded
//   replay": the window is uncompressed FP8 over the most recent 128 positions.
// [KT] "Support for Deepseek V4.1 Flash": SM120 sparse MLA keeps a full-BF16
//   route besides one that rounds Q and P to MXFP8; here every MMA operand is
//   fp16 and exact except P (rounded once to fp16).
//
// Per CTA: one row and a contiguous run of its 128-key tiles (the window
// first, then the selected entries' tiles in ascending order).  Each
// tile is gathered and dequantised to fp16 into one shared-memory buffer
// [128 keys x 512 dims] (128-byte swizzle), which serves as
//   the K-major A operand of  S^T = K Q^T        (M = 128 keys, N = H heads)
//   and the MN-major A operand of O^T += V^T P^T (M = 128 dims x 4, N = H).
// Keys = values = the latent (MQA).  Window keys are stored as e4m3 * 2^e
// (exact in fp16) with the rest of their fp32 scale, mu in [1, 2), applied to
// the logit and to p.  Online softmax across tiles in the log2 domain; the
// O^T accumulators live in TMEM and are rescaled when a head's max grows.
// With several CTAs per row (few rows), the row's CTAs form a thread-block
// cluster: each stages its unnormalised O and (m, l) in shared memory and the
// CTAs merge them by log-sum-exp over distributed shared memory, each taking
// every splits-th head.
//
// Latency: every selected entry's page is resolved once, up front, by all
// threads together; the raw FP4/FP8 bytes of tile t+1 are loaded into
// registers while tile t is dequantised and multiplied, so the HBM gather of
// one tile overlaps the tensor-core and softmax work of the previous one.
// Dequantisation uses the packed e2m1x2 / e4m3x2 -> f16x2 conversions.  MMA
// descriptors are formed once and advanced by constant offsets, so the
// issuing thread keeps the tensor pipe busy.  The output is normalised by a
// per-head reciprocal and leaves through shared memory in 16-byte stores.
#include <cooperative_groups.h>

#include <atomic>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

constexpr int kThreads = 512;
constexpr int kTileKeys = 128;
constexpr int kMainTiles = TOPK / kTileKeys;      // 4
constexpr int kMaxTiles = kMainTiles + 1;         // 4 global + 1 window
static_assert(TOPK == kThreads, "one selected entry per thread in the set-up lookup");
static_assert(D == kThreads, "one output dimension per thread in the merges");
constexpr int kMaxH = CSA_MAX_HEADS;             // 64
constexpr float kLog2e = 1.4426950408889634f;
// The running max used for exp2 moves only when a tile's max exceeds it by
// more than this (log2 units): p <= 2^8, so P stays far inside fp16 range and
// the O^T accumulators are rarely rescaled.
constexpr float kRescaleLog2 = 8.0f;

struct AttnSmem {
  uint8_t k[kTileKeys * D * 2];        // 131072, 1024-aligned: kc*16384 + (key/8)*1024 + (key%8)*128
  uint8_t q[kMaxH * D * 2];            // 65536: kc*(H*128) + (h/8)*1024 + (h%8)*128
  uint8_t p[kTileKeys * 128];          // 16384: (key/8)*1024 + (key%8)*128, heads along the row
  int32_t ent_pg[TOPK];                // page of each selected entry, -1 when none
  uint8_t ent_slot[TOPK];
  float mu[kTileKeys];
  float red_max[4][kMaxH];             // per key-quarter partial max / sum of a tile
  float red_sum[4][kMaxH];
  float m_buf[2][kMaxH];               // running max (log2), two buffers flipped when it moves
  float m_fin[kMaxH];                  // the final running max per head
  float l_run[kMaxH];
  float m_out[kMaxH], l_out[kMaxH];    // a split's final (m, l), read by the cluster's merge
  float inv_l[kMaxH];
  uint32_t tail_last;                  // a tail row's CTA: it arrived last and merges the row
  uint64_t s_bar, pv_bar;
  uint32_t tmem_base;
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Four FP4 pairs (the bytes of w, low byte first) -> four f16x2; in each the
// low nibble (even dimension) lands in the low half.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// Two E4M3 pairs (the 16-bit halves of w) -> two f16x2, low byte -> low half.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t (&o)[2]) {
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "mov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h0;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
      : "=r"(o[0]), "=r"(o[1])
      : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t x, __half2 s) {
  const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&x), s);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// In-warp reduction of NV values per lane (NV = 4, 8, 16 or 32) across the 32
// lanes: recursive halving, then a butterfly over the remaining lane bits.
// Lane l ends with the reduction of value index (l >> (5 - log2 NV)).
template <int NV>
struct RedShift {
  static constexpr int v = NV == 32 ? 0 : (NV == 16 ? 1 : (NV == 8 ? 2 : 3));
};
template <int NV, bool kMax>
__device__ __forceinline__ float warp_reduce_many(float (&v)[NV], int lane) {
  int cnt = NV;
#pragma unroll
  for (int o = 16; o >= 1 && cnt > 1; o >>= 1) {
    const int half = cnt >> 1;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < NV / 2; ++i) {
      if (i < half) {
        const float send = upper ? v[i] : v[i + half];
        const float keep = upper ? v[i + half] : v[i];
        const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, o);
        v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
      }
    }
    cnt = half;
  }
  float x = v[0];
  constexpr int kShift = RedShift<NV>::v;
#pragma unroll
  for (int o = 1; o < (1 << kShift); o <<= 1) {
    const float y = __shfl_xor_sync(0xFFFFFFFFu, x, o);
    x = kMax ? fmaxf(x, y) : x + y;
  }
  return x;
}

// Gather role of a thread: warp w holds keys 8w..8w+7, lane = 8q + (key & 7).
// A thread takes the 16-byte chunks c16 = 4i + q of its key's row, so one
// warp-wide load covers 8 keys x 64 contiguous bytes (8 cache lines), and the
// eight lanes of a quarter-warp, which differ in key & 7, store to distinct
// swizzled banks.
struct RawMain {
  uint4 d[4];      // chunks c16 = q, 4+q, 8+q, 12+q of the 256 FP4 data bytes
  uint16_t sc[4];  // E4M3 scales of blocks 2*c16, 2*c16+1 for each chunk
  int valid;
};
struct RawWin {
  uint4 d[8];      // chunks c16 = 4i + q (i = 0..7) of the 512 E4M3 codes
  float ws;        // the token's fp32 scale
  int valid;
};

// Loads written as volatile asm stay where the program issues them, so the
// prefetch of the next tile is in flight while this one is processed.
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint16_t ldg_nc_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ldg_nc_f32(const void* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void gather_main(const AttnArgs& a, const AttnSmem& sm, int m, int key, int q,
                                            RawMain& g) {
  const int j = m * kTileKeys + key;
  const int pg = sm.ent_pg[j];
  g.valid = pg >= 0;
  if (pg >= 0) {
    const uint8_t* src = a.kv_pool + (size_t)pg * KV_PAGE;
    const int slot = sm.ent_slot[j];
    const uint8_t* dp = src + slot * 256 + 16 * q;
    const uint8_t* sp = src + KV_SCALE_OFF + slot * 32 + 2 * q;
#pragma unroll
    for (int i = 0; i < 4; ++i) g.d[i] = ldg_nc_v4(dp + 64 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) g.sc[i] = ldg_nc_u16(sp + 8 * i);
  }
}

__device__ __forceinline__ void gather_win(const AttnArgs& a, int b, int pos, int key, int q, RawWin& g) {
  const int p = max(0, pos - (WIN - 1)) + key;
  g.valid = p <= pos;
  if (p <= pos) {
    const size_t slot = (size_t)b * a.win_cap + (size_t)(p % a.win_cap);
    const uint8_t* dp = a.win_codes + slot * D + 16 * q;
#pragma unroll
    for (int i = 0; i < 8; ++i) g.d[i] = ldg_nc_v4(dp + 64 * i);
    g.ws = ldg_nc_f32(a.win_scale + slot);
  }
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16(uint16_t v) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
  return d;
}

// NVFP4 entry chunks -> fp16 K rows (e2m1 * E4M3 scale is exact in fp16).
__device__ __forceinline__ void dequant_main(const RawMain& g, AttnSmem& sm, int key, int q) {
  uint8_t* krow_base = sm.k + (key >> 3) * 1024;
  if (q == 0) sm.mu[key] = g.valid ? 1.0f : 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {                  // chunk c16 = 4i + q: dims 32*c16 .. +32
    const uint4 dv = g.valid ? g.d[i] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w4[4] = {dv.x, dv.y, dv.z, dv.w};
    const uint32_t sp = e4m3x2_to_f16(g.valid ? g.sc[i] : (uint16_t)0);
    const __half2 hs0 = __low2half2(*reinterpret_cast<const __half2*>(&sp));
    const __half2 hs1 = __high2half2(*reinterpret_cast<const __half2*>(&sp));
    uint32_t o[16];
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
      uint32_t f[4];
      e2m1x8_to_f16(w4[wd], f);
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) o[wd * 4 + bb] = hmul2_u32(f[bb], wd < 2 ? hs0 : hs1);
    }
    const int c16 = 4 * i + q;
    const int kc = c16 >> 1, ch0 = (c16 & 1) * 4;    // 64-dim atom, first 8-dim chunk
    uint8_t* dst = krow_base + kc * 16384;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(dst + swz128(key & 7, ch0 + c)) =
          make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
  }
}

// Rotate-half on the pair (a, b) = (dim 448 + j, dim 480 + j) of the last 64
// dims: a' = a*c - b*s, b' = b*c + a*s, each product and the sum rounded once
// (no fused multiply-add).  `mine` holds this thread's 16 values, `other` the
// partner's (the other half of the pairs); lower: this thread holds the a's.
__device__ __forceinline__ void rotate16(float (&mine)[16], const float (&other)[16], bool lower,
                                         const float* cs, const float* sn) {
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const float c = __ldg(cs + t), s = __ldg(sn + t);
    mine[t] = lower ? __fsub_rn(__fmul_rn(mine[t], c), __fmul_rn(other[t], s))
                    : __fadd_rn(__fmul_rn(mine[t], c), __fmul_rn(other[t], s));
  }
}

// Window token chunks: s = 2^e * mu, mu in [1, 2); codes * 2^e go to the
// fp16 K rows (exact), mu scales the logit and p.  With rotary tables the
// token's last 64 dims are rotated with its position's row first (in fp32,
// then rounded to fp16): lanes q and q ^ 2 of a key hold the two halves.
// rcos / rsin must be null in all lanes of a warp or in none.
__device__ __forceinline__ void dequant_win(const RawWin& g, AttnSmem& sm, int key, int q, const float* rcos,
                                            const float* rsin) {
  uint8_t* krow_base = sm.k + (key >> 3) * 1024;
  float pow2 = 0.0f, mu = 0.0f;
  if (g.valid && g.ws > 0.0f) {
    int ex;
    const float m = frexpf(g.ws, &ex);             // ws = m * 2^ex, m in [0.5, 1)
    mu = 2.0f * m;
    pow2 = ldexpf(1.0f, ex - 1);
  }
  if (q == 0) sm.mu[key] = g.valid ? mu : 0.0f;
  const bool fast = pow2 >= 6.103515625e-05f && pow2 <= 32768.0f;   // 2^e is a normal fp16
  const __half2 hp = __float2half2_rn(pow2);
#pragma unroll
  for (int i = 0; i < 8; ++i) {                  // chunk c16 = 4i + q: 16 codes = dims 16*c16 .. +16
    const uint4 dv = g.valid ? g.d[i] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w4[4] = {dv.x, dv.y, dv.z, dv.w};
    uint32_t o[8];
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
      uint32_t f[2];
      e4m3x4_to_f16(w4[wd], f);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (fast) {
          o[wd * 2 + hh] = hmul2_u32(f[hh], hp);
        } else {
          const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&f[hh]));
          const __half2 v = __floats2half2_rn(x.x * pow2, x.y * pow2);
          o[wd * 2 + hh] = *reinterpret_cast<const uint32_t*>(&v);
        }
      }
    }
    if (i == 7 && rcos != nullptr) {             // dims 448 + 16q .. +15: the rotated part
      float mine[16], other[16];
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        uint32_t f[2];
        e4m3x4_to_f16(w4[wd], f);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&f[hh]));
          mine[4 * wd + 2 * hh] = x.x * pow2;      // exact: an E4M3 value times a power of two
          mine[4 * wd + 2 * hh + 1] = x.y * pow2;
        }
      }
#pragma unroll
      for (int t = 0; t < 16; ++t) other[t] = __shfl_xor_sync(0xFFFFFFFFu, mine[t], 16);
      rotate16(mine, other, q < 2, rcos + 16 * (q & 1), rsin + 16 * (q & 1));
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const __half2 v = __floats2half2_rn(mine[2 * t], mine[2 * t + 1]);
        o[t] = *reinterpret_cast<const uint32_t*>(&v);
      }
    }
    const int c16 = 4 * i + q;
    const int kc = c16 >> 2, ch0 = (c16 & 3) * 2;
    uint8_t* dst = krow_base + kc * 16384;
    *reinterpret_cast<uint4*>(dst + swz128(key & 7, ch0)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(dst + swz128(key & 7, ch0 + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// Barrier over the four warps that share one head group (ids 1..8).
__device__ __forceinline__ void group_sync(int id) {
  asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}
// The same barrier, also OR-ing a flag over the four warps: every thread of
// the head group gets the same answer, so all take the same branch after it.
__device__ __forceinline__ bool group_sync_or(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, float (&v)[N]) {
  if constexpr (N % 16 == 0) {
#pragma unroll
    for (int c = 0; c < N; c += 16) {
      uint32_t u[16];
      tmem_ld16(taddr + c, u);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) v[c + i] = __uint_as_float(u[i]);
    }
  } else {
#pragma unroll
    for (int c = 0; c < N; c += 4) {
      uint32_t u[4];
      tmem_ld4(taddr + c, u);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 4; ++i) v[c + i] = __uint_as_float(u[i]);
    }
  }
}

template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const float (&v)[N]) {
  if constexpr (N % 16 == 0) {
#pragma unroll
    for (int c = 0; c < N; c += 16) {
      uint32_t u[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(v[c + i]);
      tmem_st16(taddr + c, u);
    }
  } else {
#pragma unroll
    for (int c = 0; c < N; c += 4) {
      uint32_t u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) u[i] = __float_as_uint(v[c + i]);
      tmem_st4(taddr + c, u);
    }
  }
}

// Tile order within a row: the window first (when present), then the
// selected entries' tiles in ascending order.  A CTA takes the contiguous
// tile range [t_beg, t_end) of its split.
template <int H>
__global__ void __launch_bounds__(kThreads, 1) k_sparse_attn(AttnArgs a) {
  constexpr int HH = H / 4;                       // heads per thread in the softmax
  extern __shared__ uint8_t smem_raw[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  // row and split: rows before tail_row0 (all rows without a tail split) take
  // a.splits CTAs each; a tail row takes tail_splits CTAs that merge through
  // the workspace
  const bool tail = a.tail_splits > 1 && (int)blockIdx.x >= a.tail_row0;
  const int kt = (int)blockIdx.x - a.tail_row0;          // a tail CTA's partial
  const int splits = tail ? a.tail_splits : a.splits;
  const int r = tail ? a.tail_row0 + kt / splits : (int)blockIdx.x / splits;
  const int split = tail ? kt % splits : (int)blockIdx.x % splits;

  const int b = __ldg(a.row_req + r);
  const int pos = __ldg(a.row_pos + r);
  const bool rope = a.rope_cos != nullptr;
  // with rotary tables a row needs a table row for its position
  const bool row_ok = (b >= 0 && b < a.num_requests && pos >= 0) && (!rope || pos < a.rope_rows);
  if (!row_ok && tid == 0) raise_flag(a.status, CSA_FLAG_ROW_INVALID);
  const int n = row_ok ? (pos + 1) / a.P : 0;
  const int nsel = min(n, TOPK);
  const int gtiles = (nsel + kTileKeys - 1) / kTileKeys;
  const int hw = ((a.win_codes != nullptr) && row_ok) ? 1 : 0;   // window tile present
  const int ntiles = gtiles + hw;
  const int tper = (ntiles + splits - 1) / splits;
  const int t_beg = min(ntiles, split * tper), t_end = min(ntiles, t_beg + tper);
  const bool win_here = hw && t_beg == 0 && t_end > 0;
  const int m_beg = max(t_beg - hw, 0), m_end = max(t_end - hw, 0);   // main tiles [m_beg, m_end)

  // ---- prologue, overlapping the previous kernel's tail when chained after
  // the top-k of the same call: barriers and TMEM, then everything that does
  // not read the selection -- Q, and the whole window tile (gather,
  // dequantise, S, softmax, PV issue) -- and only then the wait for the
  // top-k.  The call's inputs were complete before its first kernel started;
  // the window ring and the cache, which the step's append writes, were
  // complete before this kernel could start (in a step the score kernel lets
  // its dependents start only after its own wait, which follows the append).
  pdl_trigger();
  if (tid == 0) {
    mbar_init(&sm.s_bar, 1);
    mbar_init(&sm.pv_bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, 512);

  const int key = 8 * warp + (lane & 7), gq = lane >> 3;      // gather role (see RawMain)
  RawWin wraw;
  RawMain cur, nxt;
  wraw.valid = 0;
  cur.valid = 0;
  if (win_here) gather_win(a, b, pos, key, gq, wraw);
  constexpr int kQChunks = H * 64 / kThreads;     // 16-byte chunks of Q per thread
  uint4 qv[kQChunks];
  const uint16_t* qr = a.q + (size_t)r * H * D;
#pragma unroll
  for (int i = 0; i < kQChunks; ++i) {
    const int c = tid + i * kThreads, h = c >> 6, ch = c & 63;
    qv[i] = __ldg(reinterpret_cast<const uint4*>(qr + (size_t)h * D + ch * 8));
  }
  // Q: bf16 -> fp16, K-major 128B swizzle.  With rotary tables the last 64
  // dims of every head are rotated with the row's table row first (fp32, then
  // rounded to fp16): chunks 56..59 hold the a's, 60..63 the b's, lane ^ 4.
  const float* qcos = (rope && row_ok) ? a.rope_cos + (size_t)pos * 32 : nullptr;
  const float* qsin = (rope && row_ok) ? a.rope_sin + (size_t)pos * 32 : nullptr;
#pragma unroll
  for (int i = 0; i < kQChunks; ++i) {
    const int c = tid + i * kThreads, h = c >> 6, ch = c & 63, kc = ch >> 3;
    const uint32_t w[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
    uint32_t o[4];
    float f[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
    if (rope) {
      float g[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) g[k] = __shfl_xor_sync(0xFFFFFFFFu, f[k], 4);
      if (ch >= 56 && qcos != nullptr) {
        const int j0 = (ch & 3) * 8;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float cc = __ldg(qcos + j0 + k), ss = __ldg(qsin + j0 + k);
          f[k] = ch < 60 ? __fsub_rn(__fmul_rn(f[k], cc), __fmul_rn(g[k], ss))
                         : __fadd_rn(__fmul_rn(f[k], cc), __fmul_rn(g[k], ss));
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 hv = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
      o[k] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    *reinterpret_cast<uint4*>(sm.q + kc * (H * 128) + (h >> 3) * 1024 + swz128(h & 7, ch & 7)) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (tid < H) {
    sm.m_buf[0][tid] = -INFINITY;
    sm.m_buf[1][tid] = -INFINITY;
    sm.l_run[tid] = 0.0f;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t tS = tmem, tO = tmem + 64;      // S^T: H cols; O^T chunk c at 64 + 64c
  const float scale_log2 = a.softmax_scale * kLog2e;

  const int q4 = warp & 3, hsel = warp >> 2;                  // TMEM role: lane quarter, head group
  const int mykey = 32 * q4 + lane;
  const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
  const int myh = hsel * HH + (lane < HH ? lane : 0);         // head owned by this lane (lane < HH)
  bool ok = true;
  // base descriptors; each MMA adds a constant (byte offset >> 4) to the address field
  const uint64_t dK = smem_desc(smem_u32(sm.k), 16, 1024, kSwizzle128B);
  const uint64_t dQ = smem_desc(smem_u32(sm.q), 16, 1024, kSwizzle128B);
  const uint64_t dV = smem_desc(smem_u32(sm.k), 16384, 1024, kSwizzle128B);
  const uint64_t dP = smem_desc(smem_u32(sm.p), 8192, 1024, kSwizzle128B);

  // Softmax state: the running max per head in sm.m_buf[mcur] (the same for
  // the four warps of a head group, which flip mcur together), and this
  // thread's partial sums of p over its keys for its HH heads.
  int mcur = 0;
  float lpart[HH];
#pragma unroll
  for (int i = 0; i < HH; ++i) lpart[i] = 0.0f;

  // S^T, softmax, P, rescale, PV for the tile now in sm.k.
  auto compute = [&](int it, bool is_win) -> bool {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t id = idesc_f16(128, H, 0, 0);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        mma_f16(tS, dK + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2),
                dQ + (uint64_t)((ks >> 2) * (H * 8) + (ks & 3) * 2), id, ks > 0 ? 1u : 0u);
      }
      tc_commit(&sm.s_bar);
    }
    __syncwarp();
    // every thread takes the same branch, so no barrier below is left short
    if (__syncthreads_or(!mbar_wait(&sm.s_bar, it & 1))) {
      if (tid == 0) raise_flag(a.status, CSA_FLAG_TIMEOUT);
      return false;
    }
    tc_fence_after();
    // ---- softmax over this tile (log2 domain) ----
    float lg[HH];
    tmem_ld_n<HH>(tS + lane_off + hsel * HH, lg);
    // a global key is valid when it was gathered (mu = 1); a window key when
    // its position is inside the window (an all-zero token has mu = 0 and
    // contributes logit 0 and value 0, as its dequantised vector is zero)
    const float mu_k = sm.mu[mykey];
    const bool key_ok = is_win ? (max(0, pos - (WIN - 1)) + mykey) <= pos : mu_k != 0.0f;
    const float f = scale_log2 * (is_win ? mu_k : 1.0f);
#pragma unroll
    for (int i = 0; i < HH; ++i) lg[i] = key_ok ? lg[i] * f : -INFINITY;
    // The running max moves only when a logit of the tile exceeds it by more
    // than 2^8 (p stays <= 2^8, far inside fp16).  The head group agrees on
    // that with one barrier; usually nothing moves, and then no max or sum is
    // reduced here at all: each thread adds its own p to its partial sums,
    // which are reduced once after the last tile.
    const float* mr = sm.m_buf[mcur] + hsel * HH;
    bool need = false;
#pragma unroll
    for (int i = 0; i < HH; ++i) need |= lg[i] > mr[i] + kRescaleLog2;
    need = group_sync_or(1 + hsel, need);
    float mi[HH];
    if (need) {
      float tmp[HH];
#pragma unroll
      for (int i = 0; i < HH; ++i) tmp[i] = lg[i];
      constexpr int kShift = RedShift<HH>::v;
      {
        const float mx = warp_reduce_many<HH, true>(tmp, lane);
        if ((lane & ((1 << kShift) - 1)) == 0) sm.red_max[q4][hsel * HH + (lane >> kShift)] = mx;
      }
      group_sync(5 + hsel);
      // lane i < HH owns head hsel*HH + i: its new running max and correction
      float mnew, alpha;
      {
        const float tmax = fmaxf(fmaxf(sm.red_max[0][myh], sm.red_max[1][myh]),
                                 fmaxf(sm.red_max[2][myh], sm.red_max[3][myh]));
        const float mold = sm.m_buf[mcur][myh];
        mnew = (mold == -INFINITY || tmax > mold + kRescaleLog2) ? tmax : mold;
        alpha = (mold == -INFINITY) ? 0.0f : (mnew == mold ? 1.0f : exp2f(mold - mnew));
        if (q4 == 0 && lane < HH) sm.m_buf[mcur ^ 1][myh] = mnew;
      }
      bool moved = false;
#pragma unroll
      for (int i = 0; i < HH; ++i) {
        mi[i] = __shfl_sync(0xFFFFFFFFu, mnew, i);
        const float al = __shfl_sync(0xFFFFFFFFu, alpha, i);
        lpart[i] *= al;
        moved |= al != 1.0f;
      }
      // rescale this warp's lanes of the O^T columns of its heads whose max moved
      if (it > 0 && moved) {
        float al[HH];
#pragma unroll
        for (int i = 0; i < HH; ++i) al[i] = __shfl_sync(0xFFFFFFFFu, alpha, i);
#pragma unroll 1
        for (int dc = 0; dc < D / 128; ++dc) {
          float v[HH];
          const uint32_t ta = tO + lane_off + dc * 64 + hsel * HH;
          tmem_ld_n<HH>(ta, v);
#pragma unroll
          for (int i = 0; i < HH; ++i) v[i] *= al[i];
          tmem_st_n<HH>(ta, v);
        }
        tmem_st_wait();
      }
      mcur ^= 1;
    } else {
#pragma unroll
      for (int i = 0; i < HH; ++i) mi[i] = mr[i];
    }
    // p = exp2(l - m); P'^T = p * mu (window) as fp16, heads along the 128-byte row
    {
      const float fm = is_win ? mu_k : 1.0f;
      uint32_t packed[HH / 2];
#pragma unroll
      for (int i = 0; i < HH; i += 2) {
        const float p0 = (lg[i] == -INFINITY) ? 0.0f : exp2f(lg[i] - mi[i]);
        const float p1 = (lg[i + 1] == -INFINITY) ? 0.0f : exp2f(lg[i + 1] - mi[i + 1]);
        lpart[i] += p0;
        lpart[i + 1] += p1;
        const __half2 hv = __floats2half2_rn(p0 * fm, p1 * fm);
        packed[i / 2] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      uint8_t* prow = sm.p + (mykey >> 3) * 1024;
      if constexpr (HH >= 8) {
#pragma unroll
        for (int c = 0; c < HH / 8; ++c) {
          const int chunk = (hsel * HH) / 8 + c;
          *reinterpret_cast<uint4*>(prow + swz128(mykey & 7, chunk)) =
              make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        }
      } else {                                        // 4 heads = half a 16-byte chunk
        const int chunk = (hsel * HH) / 8;
        *reinterpret_cast<uint2*>(prow + swz128(mykey & 7, chunk) + 8 * (hsel & 1)) =
            make_uint2(packed[0], packed[1]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- O^T += V^T P^T ----
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t id = idesc_f16(128, H, 1, 1);
      const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll
      for (int dc = 0; dc < D / 128; ++dc) {
#pragma unroll
        for (int ks = 0; ks < kTileKeys / 16; ++ks) {
          mma_f16(tO + dc * 64, dV + (uint64_t)(dc * 2048 + ks * 128), dP + (uint64_t)(ks * 128), id,
                  ks > 0 ? 1u : acc0);
        }
      }
      tc_commit(&sm.pv_bar);
    }
    __syncwarp();
    return true;
  };

  int it = 0;
  if (win_here) {
    // ---------------- the window tile (before the wait) ----------------
    {
      // this thread's window token position; a key past the row's position is
      // empty (zero) and uses the row's own table row.  Whether to rotate is
      // the same for the whole CTA: the rotation exchanges values between lanes.
      const int p = min(pos, max(0, pos - (WIN - 1)) + key);
      const bool rot = rope && row_ok;
      dequant_win(wraw, sm, key, gq, rot ? a.rope_cos + (size_t)p * 32 : nullptr,
                  rot ? a.rope_sin + (size_t)p * 32 : nullptr);
    }
    ok = compute(0, true);
    it = 1;
  }
  pdl_wait();                    // the selected indices are ready from here on

  // ---- the selected entries: looked up (index, then page) by all threads at
  // once and their bytes prefetched into L2, so the per-tile gathers hit L2
  const int j = tid;                              // TOPK == kThreads: one selected entry per thread
  const bool jin = j < nsel && j >= m_beg * kTileKeys && j < m_end * kTileKeys;
  int e = jin ? __ldg((a.plan_in ? a.plan_in : a.topk) + (size_t)r * TOPK + j) : -1;
  {
    int pg = -1, slot = 0;
    if (e >= 0 && a.plan_in) {                    // a resolved entry: page * 64 + slot
      if ((e >> 6) >= a.num_pages) raise_flag(a.status, CSA_FLAG_PAGE_OOB);
      else { pg = e >> 6; slot = e & (PAGE - 1); }
    } else if (e >= 0) {
      if (e >= n || e / PAGE >= a.max_pages) {
        raise_flag(a.status, CSA_FLAG_TOPK_OOB);
      } else {
        const int p = __ldg(a.page_table + (size_t)b * a.max_pages + e / PAGE);
        if (p < 0 || p >= a.num_pages) raise_flag(a.status, CSA_FLAG_PAGE_OOB);
        else { pg = p; slot = e % PAGE; }
      }
    }
    // the plan: every slot of the row written once (its tile's CTA, or split
    // 0 for the padding past the selection)
    if (a.plan_out && (jin || (split == 0 && j >= nsel)))
      a.plan_out[(size_t)r * TOPK + j] = pg >= 0 ? pg * PAGE + slot : -1;
    if (pg >= 0) {
      const uint8_t* src = a.kv_pool + (size_t)pg * KV_PAGE;
      prefetch_l2(src + slot * 256, 256);
      prefetch_l2(src + KV_SCALE_OFF + slot * 32, 32);
    }
    sm.ent_pg[j] = pg;
    sm.ent_slot[j] = (uint8_t)slot;
  }
  __syncthreads();                                // entry table visible
  if (m_beg < m_end) gather_main(a, sm, m_beg, key, gq, cur);
  for (int m = m_beg; m < m_end && ok; ++m, ++it) {
    nxt.valid = 0;
    if (m + 1 < m_end) gather_main(a, sm, m + 1, key, gq, nxt);
    if (__syncthreads_or(it > 0 && !mbar_wait(&sm.pv_bar, (it - 1) & 1))) {
      if (tid == 0) raise_flag(a.status, CSA_FLAG_TIMEOUT);
      ok = false;
      break;
    }
    // ---------------- dequantise this tile into sm.k ----------------
    dequant_main(cur, sm, key, gq);
    ok = compute(it, false);
    cur = nxt;
  }
  const int done = it;
  if (ok && done > 0) {
    if (!mbar_wait(&sm.pv_bar, (done - 1) & 1)) {
      raise_flag(a.status, CSA_FLAG_TIMEOUT);
      ok = false;
    }
  }
  // ---- the sums of p over all keys per head: the threads' partial sums reduced once
  {
    constexpr int kShift = RedShift<HH>::v;
    float tmp[HH];
#pragma unroll
    for (int i = 0; i < HH; ++i) tmp[i] = lpart[i];
    const float sum = warp_reduce_many<HH, false>(tmp, lane);
    if ((lane & ((1 << kShift) - 1)) == 0) sm.red_sum[q4][hsel * HH + (lane >> kShift)] = sum;
    group_sync(1 + hsel);
    if (q4 == 0 && lane < HH) {
      sm.l_run[myh] = (sm.red_sum[0][myh] + sm.red_sum[1][myh]) + (sm.red_sum[2][myh] + sm.red_sum[3][myh]);
      sm.m_fin[myh] = sm.m_buf[mcur][myh];
    }
  }
  tc_fence_after();
  __syncthreads();
  // ---------------- epilogue ----------------
  // thread: dims d = 128*hsel + 32*q4 + lane (O^T chunk hsel, TMEM lane quarter q4)
  const bool have = ok && done > 0;
  const float* m_fin = sm.m_fin;
  const int d = 128 * hsel + 32 * q4 + lane;
  const uint32_t obase = tO + lane_off + hsel * 64;
  if (splits == 1) {
    // O[h][d] = O^T[d][h] / l[h] as bf16, straight to global memory: a warp
    // holds 32 consecutive dimensions of a head, 64 contiguous bytes per store
    if (tid < H) {
      const float l = sm.l_run[tid];
      sm.inv_l[tid] = (have && l > 0.0f) ? 1.0f / l : 0.0f;
    }
    __syncthreads();
    uint16_t* orow = a.out + (size_t)r * H * D + d;
    for (int h0 = 0; h0 < H; h0 += 16) {
      uint32_t v[16];
      if (have) {
        tmem_ld16(obase + h0, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const __nv_bfloat16 o = __float2bfloat16_rn(__uint_as_float(v[i]) * sm.inv_l[h0 + i]);
        orow[(size_t)(h0 + i) * D] = *reinterpret_cast<const uint16_t*>(&o);
      }
    }
    if (a.lse && tid < H) {
      const float l = sm.l_run[tid];
      a.lse[(size_t)r * H + tid] = (have && l > 0.0f) ? (m_fin[tid] + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
  } else if (tail) {
    // a tail row's split: its unnormalised O [H][512] and (m, l) go to the
    // workspace; the row's CTA that arrives last merges the row's partials by
    // log-sum-exp (the weights of the cluster merge below) and writes the row
    const int S = splits;
    const int ntail = (int)gridDim.x - a.tail_row0;
    float* pm = a.part + (size_t)ntail * H * D;            // [ntail][2][H]: m, then l
    {
      float* po = a.part + (size_t)kt * H * D;
      for (int h0 = 0; h0 < H; h0 += 16) {
        uint32_t v[16];
        if (have) {
          tmem_ld16(obase + h0, v);
          tmem_ld_wait();
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) __stcg(po + (size_t)(h0 + i) * D + d, have ? __uint_as_float(v[i]) : 0.0f);
      }
      if (tid < H) {
        __stcg(pm + (size_t)kt * 2 * H + tid, have ? m_fin[tid] : -INFINITY);
        __stcg(pm + (size_t)kt * 2 * H + H + tid, have ? sm.l_run[tid] : 0.0f);
      }
    }
    __threadfence();                               // this CTA's partial is visible device-wide
    __syncthreads();
    if (tid == 0) {
      const uint32_t prev = atomicAdd(a.row_done + (r - a.tail_row0), 1u);
      sm.tail_last = prev == (uint32_t)(S - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (sm.tail_last) {
      __threadfence();
      const int q0 = kt - split;                   // the row's first partial
      float* wq = reinterpret_cast<float*>(sm.p);  // [S][H] merge weights (P is free after the last PV)
      if (tid < H) {
        float mq[kMaxTiles], lq[kMaxTiles];
#pragma unroll
        for (int q = 0; q < kMaxTiles; ++q) {
          mq[q] = q < S ? __ldcg(pm + (size_t)(q0 + q) * 2 * H + tid) : -INFINITY;
          lq[q] = q < S ? __ldcg(pm + (size_t)(q0 + q) * 2 * H + H + tid) : 0.0f;
        }
        float M = -INFINITY, L = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxTiles; ++q) M = fmaxf(M, mq[q]);
#pragma unroll
        for (int q = 0; q < kMaxTiles; ++q) {
          mq[q] = mq[q] == -INFINITY ? 0.0f : exp2f(mq[q] - M);
          L += mq[q] * lq[q];
        }
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxTiles; ++q)
          if (q < S) wq[q * H + tid] = mq[q] * inv;
        if (a.lse) a.lse[(size_t)r * H + tid] = L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
      }
      __syncthreads();
      // O[h][d] = sum_q w_q[h] O_q[h][d], thread tid: dim tid (D == kThreads)
      const float* pq = a.part + (size_t)q0 * H * D + tid;
      constexpr int kHG = 16;                      // heads whose loads go out together
      for (int h0 = 0; h0 < H; h0 += kHG) {
        float v[kHG][kMaxTiles];
#pragma unroll
        for (int u = 0; u < kHG; ++u)
#pragma unroll
          for (int q = 0; q < kMaxTiles; ++q)
            v[u][q] = q < S ? __ldcg(pq + (size_t)q * H * D + (size_t)(h0 + u) * D) : 0.0f;
#pragma unroll
        for (int u = 0; u < kHG; ++u) {
          float acc = 0.0f;
#pragma unroll
          for (int q = 0; q < kMaxTiles; ++q)
            if (q < S) acc += wq[q * H + h0 + u] * v[u][q];
          const __nv_bfloat16 o = __float2bfloat16_rn(acc);
          a.out[((size_t)r * H + h0 + u) * D + tid] = *reinterpret_cast<const uint16_t*>(&o);
        }
      }
      if (tid == 0) a.row_done[r - a.tail_row0] = 0u;   // zero again for the next call
    }
  } else {
    // split partials, merged inside the row's cluster: O [H][512] unnormalised
    // (fp32, in the key tile's buffer, free after the last PV) and (m, l)
    cg::cluster_group cluster = cg::this_cluster();
    float* ostage = reinterpret_cast<float*>(sm.k);
    for (int h0 = 0; h0 < H; h0 += 16) {
      uint32_t v[16];
      if (have) {
        tmem_ld16(obase + h0, v);
        tmem_ld_wait();
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) ostage[(h0 + i) * D + d] = have ? __uint_as_float(v[i]) : 0.0f;
    }
    if (tid < H) {
      sm.m_out[tid] = have ? m_fin[tid] : -INFINITY;
      sm.l_out[tid] = have ? sm.l_run[tid] : 0.0f;
    }
    cluster.sync();                                // every split's partials are published
    // this CTA merges heads split, split + S, ...: first every (head, split)
    // pair's (m, l) in one parallel round of remote loads, then per head the
    // weights w_q = 2^(m_q - M) / sum_q 2^(m_q - M) l_q, then O = sum_q w_q O_q
    const int S = a.splits;
    const int nh = (H - split + S - 1) / S;
    float (*mq_s)[kMaxTiles] = reinterpret_cast<float (*)[kMaxTiles]>(&sm.red_max[0][0]);   // [nh][S]
    float (*lq_s)[kMaxTiles] = reinterpret_cast<float (*)[kMaxTiles]>(&sm.red_sum[0][0]);
    if (tid < nh * kMaxTiles) {
      const int i = tid / kMaxTiles, q = tid % kMaxTiles;
      float m = -INFINITY, l = 0.0f;
      if (q < S) {
        const AttnSmem* rs = cluster.map_shared_rank(&sm, q);
        m = rs->m_out[split + i * S];
        l = rs->l_out[split + i * S];
      }
      mq_s[i][q] = m;
      lq_s[i][q] = l;
    }
    __syncthreads();
    if (tid < nh) {
      float M = -INFINITY, L = 0.0f;
#pragma unroll
      for (int q = 0; q < kMaxTiles; ++q) M = fmaxf(M, mq_s[tid][q]);
      float wq[kMaxTiles];
#pragma unroll
      for (int q = 0; q < kMaxTiles; ++q) {
        wq[q] = mq_s[tid][q] == -INFINITY ? 0.0f : exp2f(mq_s[tid][q] - M);
        L += wq[q] * lq_s[tid][q];
      }
      const float inv = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
      for (int q = 0; q < kMaxTiles; ++q) mq_s[tid][q] = wq[q] * inv;   // the row's own entries only
      if (a.lse)
        a.lse[(size_t)r * H + split + tid * S] = L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    const float* ob[kMaxTiles];                    // every split's O, thread tid: dim tid (D == kThreads)
#pragma unroll
    for (int q = 0; q < kMaxTiles; ++q)
      ob[q] = reinterpret_cast<const float*>(cluster.map_shared_rank(&sm, q < S ? q : 0)->k) + tid;
    constexpr int kHG = 4;                         // heads whose remote loads go out together
    for (int i0 = 0; i0 < nh; i0 += kHG) {
      float v[kHG][kMaxTiles];
#pragma unroll
      for (int u = 0; u < kHG; ++u)
#pragma unroll
        for (int q = 0; q < kMaxTiles; ++q)
          v[u][q] = (i0 + u < nh && q < S) ? ob[q][(split + (i0 + u) * S) * D] : 0.0f;
#pragma unroll
      for (int u = 0; u < kHG; ++u) {
        if (i0 + u >= nh) break;
        float acc = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxTiles; ++q) acc += mq_s[i0 + u][q] * v[u][q];
        const __nv_bfloat16 o = __float2bfloat16_rn(acc);
        a.out[((size_t)r * H + split + (i0 + u) * S) * D + tid] = *reinterpret_cast<const uint16_t*>(&o);
      }
    }
    cluster.sync();                                // no CTA leaves while another reads its partials
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

constexpr int kMaxDevices = 64;

// Clusters of s CTAs (one CTA per SM) that the device holds at once.  A GPC
// holds whole clusters, so s times this can fall short of the SM count.
// Queried once per (device, s); 0 when the query fails.
template <int H>
int clusters_resident(int s, size_t smem) {
  static std::atomic<int> known[kMaxDevices][kMaxTiles + 1];   // value + 1; 0 = not yet asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) {
    const int v = known[dev][s].load(std::memory_order_relaxed);
    if (v > 0) return v - 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = s;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_sparse_attn<H>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  if (dev >= 0 && dev < kMaxDevices) known[dev][s].store(n + 1, std::memory_order_relaxed);
  return n;
}

template <int H>
cudaError_t launch_h(const AttnArgs& args, Order order, cudaStream_t stream) {
  const size_t smem = sizeof(AttnSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_sparse_attn<H>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // fewer splits where the rows' clusters would not all be resident at once
  AttnArgs a = args;
  while (a.splits > 1 && a.num_rows > clusters_resident<H>(a.splits, smem)) --a.splits;
  if (a.splits > 1) a.tail_splits = 1;
  if (a.splits == 1) {
    const int grid = a.tail_splits > 1 ? a.tail_row0 + (a.num_rows - a.tail_row0) * a.tail_splits : a.num_rows;
    return launch_kernel(order, k_sparse_attn<H>, dim3(grid), dim3(kThreads), smem, stream, a);
  }
  // a row's splits form one cluster, which merges their partials
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_rows * a.splits, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1 + order_attr(order, attr + 1);
  return cudaLaunchKernelEx(&cfg, k_sparse_attn<H>, a);
}

}  // namespace

int32_t attn_choose_splits(int32_t num_rows, int num_sms) {
  if (num_rows <= 0) return 1;
  int s = num_sms / num_rows;
  return s < 1 ? 1 : (s > kMaxTiles ? kMaxTiles : s);
}

int32_t attn_tail_plan(int32_t num_rows, int num_sms, int32_t* tail_row0) {
  *tail_row0 = num_rows;
  if (num_sms <= 0 || num_rows <= num_sms) return 1;
  const int rem = num_rows % num_sms;
  if (rem == 0) return 1;
  int s = num_sms / rem;
  s = s > kMaxTiles ? kMaxTiles : s;
  if (s < 2) return 1;
  *tail_row0 = num_rows - rem;
  return s;
}

namespace {
constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
// The tail partials' bytes: O of every tail CTA, then its (m, l).
size_t tail_part_bytes(size_t ctas, int32_t H) {
  return align256(ctas * (size_t)H * D * sizeof(float) + ctas * 2 * (size_t)H * sizeof(float));
}
}  // namespace

size_t attn_tail_ws_bytes(int32_t num_rows, int32_t H, int num_sms) {
  int32_t row0 = 0;
  const int32_t s = attn_tail_plan(num_rows, num_sms, &row0);
  if (s < 2) return 0;
  return align256((size_t)(num_rows - row0) * sizeof(uint32_t)) + tail_part_bytes((size_t)(num_rows - row0) * s, H);
}

void attn_tail_setup(AttnArgs& a, void* base, size_t bytes, int num_sms) {
  a.tail_row0 = a.num_rows;
  a.tail_splits = 1;
  a.part = nullptr;
  a.row_done = nullptr;
  if (a.splits != 1 || base == nullptr) return;
  int32_t row0 = 0;
  const int32_t s = attn_tail_plan(a.num_rows, num_sms, &row0);
  if (s < 2 || bytes < attn_tail_ws_bytes(a.num_rows, a.H, num_sms)) return;
  // the counters first, then the partials
  uint8_t* p = static_cast<uint8_t*>(base);
  a.tail_row0 = row0;
  a.tail_splits = s;
  a.row_done = reinterpret_cast<uint32_t*>(p);
  a.part = reinterpret_cast<float*>(p + align256((size_t)(a.num_rows - row0) * sizeof(uint32_t)));
}

cudaError_t launch_sparse_attn(const AttnArgs& a, Order order, cudaStream_t stream) {
  if (a.num_rows <= 0) return cudaSuccess;
  switch (a.H) {
    case 16: return launch_h<16>(a, order, stream);
    case 32: return launch_h<32>(a, order, stream);
    case 64: return launch_h<64>(a, order, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csa
