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
// Per CTA: one row and a contiguous run of its 128-key tiles (tiles 0..3 =
// the selected entries in ascending order, the last tile = the window).  Each
// tile is gathered and dequantised to fp16 into one shared-memory buffer
// [128 keys x 512 dims] (128-byte swizzle), which serves as
//   the K-major A operand of  S^T = K Q^T        (M = 128 keys, N = H heads)
//   and the MN-major A operand of O^T += V^T P^T (M = 128 dims x 4, N = H).
// Keys = values = the latent (MQA).  Window keys are stored as e4m3 * 2^e
// (exact in fp16) with the rest of their fp32 scale, mu in [1, 2), applied to
// the logit and to p.  Online softmax across tiles in the log2 domain; the
// O^T accumulators live in TMEM and are rescaled when a head's max grows.
// With several CTAs per row, partial (O, m, l) go to the workspace and a merge
// kernel combines them by log-sum-exp.
//
// Latency: every selected entry's page is resolved once, up front, by all
// threads together; the raw FP4/FP8 bytes of tile t+1 are loaded into
// registers while tile t is dequantised and multiplied, so the HBM gather of
// one tile overlaps the tensor-core and softmax work of the previous one.
// Dequantisation uses the packed e2m1x2 / e4m3x2 -> f16x2 conversions.
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

constexpr int kThreads = 512;
constexpr int kTileKeys = 128;
constexpr int kMainTiles = TOPK / kTileKeys;      // 4
constexpr int kMaxTiles = kMainTiles + 1;         // 4 global + 1 window
constexpr int kMaxH = CSA_MAX_HEADS;             // 64
constexpr float kLog2e = 1.4426950408889634f;

struct AttnSmem {
  uint8_t k[kTileKeys * D * 2];        // 131072, 1024-aligned: kc*16384 + (key/8)*1024 + (key%8)*128
  uint8_t q[kMaxH * D * 2];            // 65536: kc*(H*128) + (h/8)*1024 + (h%8)*128
  uint8_t p[kTileKeys * 128];          // 16384: (key/8)*1024 + (key%8)*128, heads along the row
  int32_t ent_pg[TOPK];                // page of each selected entry, -1 when none
  uint8_t ent_slot[TOPK];
  float mu[kTileKeys];
  float red[4][kMaxH];                 // per-quarter partial max / sum
  float m_run[kMaxH], l_run[kMaxH], alpha[kMaxH];
  uint64_t s_bar, pv_bar;
  uint32_t tmem_base;
  int32_t rescale;
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

// Raw bytes of one key's quarter (128 dims) of a tile, in registers.
struct Raw {
  uint4 d[8];      // main entry: d[0..3] = 64 FP4 bytes; window: 128 E4M3 codes
  uint2 sc;        // main entry: the 8 E4M3 block scales of these 128 dims
  float ws;        // window token: fp32 scale
  int valid;
};

__device__ __forceinline__ void gather(const AttnArgs& a, const AttnSmem& sm, int r, int b, int pos,
                                       int t, bool is_win, int key, int part, Raw& g) {
  if (!is_win) {
    const int j = t * kTileKeys + key;
    const int pg = sm.ent_pg[j];
    g.valid = pg >= 0;
    if (pg >= 0) {
      const uint8_t* src = a.kv_pool + (size_t)pg * KV_PAGE;
      const int slot = sm.ent_slot[j];
      const uint4* dp = reinterpret_cast<const uint4*>(src + slot * 256 + 64 * part);
#pragma unroll
      for (int i = 0; i < 4; ++i) g.d[i] = __ldg(dp + i);
      g.sc = __ldg(reinterpret_cast<const uint2*>(src + KV_SCALE_OFF + slot * 32 + 8 * part));
    }
  } else {
    const int p = max(0, pos - (WIN - 1)) + key;
    g.valid = p <= pos;
    if (p <= pos) {
      const size_t slot = (size_t)b * a.win_cap + (size_t)(p % a.win_cap);
      const uint4* dp = reinterpret_cast<const uint4*>(a.win_codes + slot * D + 128 * part);
#pragma unroll
      for (int i = 0; i < 8; ++i) g.d[i] = __ldg(dp + i);
      g.ws = __ldg(a.win_scale + slot);
    }
  }
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1) k_sparse_attn(AttnArgs a) {
  constexpr int HH = H / 4;                       // heads per thread in the softmax
  extern __shared__ uint8_t smem_raw[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  const int r = blockIdx.x / a.splits, split = blockIdx.x % a.splits;

  const int b = __ldg(a.row_req + r);
  const int pos = __ldg(a.row_pos + r);
  const bool row_ok = (b >= 0 && b < a.num_requests && pos >= 0);
  if (!row_ok && tid == 0) raise_flag(a.status, CSA_FLAG_ROW_INVALID);
  const int n = row_ok ? (pos + 1) / a.P : 0;
  const int nsel = min(n, TOPK);
  const int gtiles = (nsel + kTileKeys - 1) / kTileKeys;
  const bool has_win = (a.win_codes != nullptr) && row_ok;
  const int ntiles = gtiles + (has_win ? 1 : 0);
  const int tper = (ntiles + a.splits - 1) / a.splits;
  const int t_beg = min(ntiles, split * tper), t_end = min(ntiles, t_beg + tper);

  // ---- setup: entry pages, barriers, TMEM, Q (bf16 -> fp16, K-major 128B swizzle)
  {
    const int j = tid;                            // TOPK == kThreads
    int pg = -1, slot = 0;
    if (j < nsel && j >= t_beg * kTileKeys && j < min(t_end, gtiles) * kTileKeys) {
      const int e = __ldg(a.topk + (size_t)r * TOPK + j);
      if (e >= 0) {
        if (e >= n || e / PAGE >= a.max_pages) {
          raise_flag(a.status, CSA_FLAG_TOPK_OOB);
        } else {
          const int p = __ldg(a.page_table + (size_t)b * a.max_pages + e / PAGE);
          if (p < 0 || p >= a.num_pages) raise_flag(a.status, CSA_FLAG_PAGE_OOB);
          else { pg = p; slot = e % PAGE; }
        }
      }
    }
    sm.ent_pg[j] = pg;
    sm.ent_slot[j] = (uint8_t)slot;
  }
  if (tid < H) {
    sm.m_run[tid] = -INFINITY;
    sm.l_run[tid] = 0.0f;
  }
  if (tid == 0) {
    mbar_init(&sm.s_bar, 1);
    mbar_init(&sm.pv_bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, 512);
  {
    const uint16_t* qr = a.q + (size_t)r * H * D;
    for (int c = tid; c < H * 64; c += kThreads) {     // 16-byte chunks of 8 dims
      const int h = c >> 6, ch = c & 63, kc = ch >> 3;
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(qr + (size_t)h * D + ch * 8));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 hv = __floats2half2_rn(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
        o[i] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      *reinterpret_cast<uint4*>(sm.q + kc * (H * 128) + (h >> 3) * 1024 + swz128(h & 7, ch & 7)) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t tS = tmem, tO = tmem + 64;      // S^T: H cols; O^T chunk c at 64 + 64c
  const float scale_log2 = a.softmax_scale * kLog2e;

  const int key = tid & (kTileKeys - 1), part = tid >> 7;    // gather role: dims 128*part..+128
  const int q4 = warp & 3, hsel = warp >> 2;                  // TMEM role: lane quarter, head quarter
  const int mykey = 32 * q4 + lane;
  bool ok = true;

  Raw cur, nxt;
  cur.valid = 0;
  if (t_beg < t_end) gather(a, sm, r, b, pos, t_beg, has_win && t_beg == ntiles - 1, key, part, cur);

  for (int t = t_beg; t < t_end && ok; ++t) {
    const int it = t - t_beg;
    const bool is_win = has_win && (t == ntiles - 1);
    nxt.valid = 0;
    if (t + 1 < t_end) gather(a, sm, r, b, pos, t + 1, has_win && t + 1 == ntiles - 1, key, part, nxt);
    if (it > 0 && !mbar_wait(&sm.pv_bar, (it - 1) & 1)) { raise_flag(a.status, CSA_FLAG_TIMEOUT); ok = false; break; }
    // ---------------- dequantise this tile into sm.k ----------------
    uint8_t* krow_base = sm.k + (key >> 3) * 1024;
    if (!is_win) {
      if (part == 0) sm.mu[key] = cur.valid ? 1.0f : 0.0f;
      const uint32_t sw[2] = {cur.valid ? cur.sc.x : 0u, cur.valid ? cur.sc.y : 0u};
#pragma unroll
      for (int i = 0; i < 4; ++i) {                  // 32 dims, scale blocks 2i and 2i+1
        const uint4 dv = cur.valid ? cur.d[i] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w4[4] = {dv.x, dv.y, dv.z, dv.w};
        uint32_t s2[2];
        e4m3x4_to_f16(sw[i >> 1], s2);
        const uint32_t sp = s2[i & 1];
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
        const int dim0 = 128 * part + 32 * i;          // 32 dims = 4 chunks of 8
        const int kc = dim0 >> 6, ch0 = (dim0 & 63) >> 3;
        uint8_t* dst = krow_base + kc * 16384;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(dst + swz128(key & 7, ch0 + c)) =
              make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
      }
    } else {
      // s = 2^e * mu, mu in [1, 2): the codes are scaled by 2^e (exact in fp16)
      float pow2 = 0.0f, mu = 0.0f;
      if (cur.valid && cur.ws > 0.0f) {
        int ex;
        const float m = frexpf(cur.ws, &ex);           // ws = m * 2^ex, m in [0.5, 1)
        mu = 2.0f * m;
        pow2 = ldexpf(1.0f, ex - 1);
      }
      if (part == 0) sm.mu[key] = cur.valid ? mu : 0.0f;
      const bool fast = pow2 >= 6.103515625e-05f && pow2 <= 32768.0f;   // 2^e is a normal fp16
      const __half2 hp = __float2half2_rn(pow2);
#pragma unroll
      for (int i = 0; i < 8; ++i) {                  // 16 codes = 16 dims = 2 chunks
        const uint4 dv = cur.valid ? cur.d[i] : make_uint4(0u, 0u, 0u, 0u);
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
        const int dim0 = 128 * part + 16 * i;
        const int kc = dim0 >> 6, ch0 = (dim0 & 63) >> 3;
        uint8_t* dst = krow_base + kc * 16384;
        *reinterpret_cast<uint4*>(dst + swz128(key & 7, ch0)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(dst + swz128(key & 7, ch0 + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---------------- S^T = K Q^T ----------------
    if (tid == 0) {
      tc_fence_after();
      const uint32_t kb = smem_u32(sm.k), qb = smem_u32(sm.q);
#pragma unroll 4
      for (int ks = 0; ks < D / 16; ++ks) {
        mma_f16(tS, smem_desc(kb + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, kSwizzle128B),
                smem_desc(qb + (ks >> 2) * (H * 128) + (ks & 3) * 32, 16, 1024, kSwizzle128B),
                idesc_f16(128, H, 0, 0), ks > 0 ? 1u : 0u);
      }
      tc_commit(&sm.s_bar);
    }
    __syncwarp();
    if (!mbar_wait(&sm.s_bar, it & 1)) { raise_flag(a.status, CSA_FLAG_TIMEOUT); ok = false; break; }
    tc_fence_after();
    // ---------------- softmax over this tile (log2 domain) ----------------
    float lg[HH];
    {
      const uint32_t base = tS + ((uint32_t)(32 * q4) << 16) + hsel * HH;
      if constexpr (HH % 16 == 0) {
#pragma unroll
        for (int c = 0; c < HH; c += 16) {
          uint32_t v[16];
          tmem_ld16(base + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) lg[c + i] = __uint_as_float(v[i]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < HH; c += 4) {
          uint32_t v[4];
          tmem_ld4(base + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 4; ++i) lg[c + i] = __uint_as_float(v[i]);
        }
      }
    }
    // a global key is valid when it was gathered (mu = 1); a window key when
    // its position is inside the window (an all-zero token has mu = 0 and
    // contributes logit 0 and value 0, as its dequantised vector is zero)
    const float mu_k = sm.mu[mykey];
    const bool key_ok = is_win ? (max(0, pos - (WIN - 1)) + mykey) <= pos : mu_k != 0.0f;
#pragma unroll
    for (int i = 0; i < HH; ++i) lg[i] = key_ok ? lg[i] * (scale_log2 * (is_win ? mu_k : 1.0f)) : -INFINITY;
    float tmp[HH];
#pragma unroll
    for (int i = 0; i < HH; ++i) tmp[i] = lg[i];
    constexpr int kShift = RedShift<HH>::v;
    {
      const float mx = warp_reduce_many<HH, true>(tmp, lane);
      if ((lane & ((1 << kShift) - 1)) == 0) sm.red[q4][hsel * HH + (lane >> kShift)] = mx;
    }
    __syncthreads();
    if (tid < H) {
      const float tmax = fmaxf(fmaxf(sm.red[0][tid], sm.red[1][tid]), fmaxf(sm.red[2][tid], sm.red[3][tid]));
      const float mold = sm.m_run[tid];
      const float mnew = fmaxf(mold, tmax);
      sm.alpha[tid] = (mold == -INFINITY) ? 0.0f : exp2f(mold - mnew);
      sm.m_run[tid] = mnew;
    }
    if (tid == 0) sm.rescale = 0;
    __syncthreads();
    if (tid < H && it > 0 && sm.alpha[tid] != 1.0f) sm.rescale = 1;
    // p = exp2(l - m); P'^T = p * mu (window) as fp16, heads along the 128-byte row
    {
      uint32_t packed[HH / 2];
#pragma unroll
      for (int i = 0; i < HH; i += 2) {
        const float m0 = sm.m_run[hsel * HH + i], m1 = sm.m_run[hsel * HH + i + 1];
        const float p0 = (lg[i] == -INFINITY) ? 0.0f : exp2f(lg[i] - m0);
        const float p1 = (lg[i + 1] == -INFINITY) ? 0.0f : exp2f(lg[i + 1] - m1);
        tmp[i] = p0;
        tmp[i + 1] = p1;
        const float f = is_win ? mu_k : 1.0f;
        const __half2 hv = __floats2half2_rn(p0 * f, p1 * f);
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
    {
      const float sum = warp_reduce_many<HH, false>(tmp, lane);
      __syncthreads();   // everyone is done reading sm.red (max) above
      if ((lane & ((1 << kShift) - 1)) == 0) sm.red[q4][hsel * HH + (lane >> kShift)] = sum;
    }
    __syncthreads();
    if (tid < H) {
      const float ts = (sm.red[0][tid] + sm.red[1][tid]) + (sm.red[2][tid] + sm.red[3][tid]);
      sm.l_run[tid] = sm.alpha[tid] * sm.l_run[tid] + ts;
    }
    // rescale the O^T accumulators of heads whose running max grew
    if (sm.rescale) {
      tc_fence_after();
      const uint32_t base = tO + ((uint32_t)(32 * q4) << 16) + hsel * 64;
      if constexpr (H % 16 == 0) {
#pragma unroll 1
        for (int h0 = 0; h0 < H; h0 += 16) {
          uint32_t v[16];
          tmem_ld16(base + h0, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * sm.alpha[h0 + i]);
          tmem_st16(base + h0, v);
        }
      }
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---------------- O^T += V^T P^T ----------------
    if (tid == 0) {
      tc_fence_after();
      const uint32_t kb = smem_u32(sm.k), pb = smem_u32(sm.p);
      for (int dc = 0; dc < D / 128; ++dc) {
#pragma unroll
        for (int ks = 0; ks < kTileKeys / 16; ++ks) {
          mma_f16(tO + dc * 64, smem_desc(kb + dc * 32768 + ks * 2048, 16384, 1024, kSwizzle128B),
                  smem_desc(pb + ks * 2048, 8192, 1024, kSwizzle128B), idesc_f16(128, H, 1, 1),
                  (it > 0 || ks > 0) ? 1u : 0u);
        }
      }
      tc_commit(&sm.pv_bar);
    }
    __syncwarp();
    cur = nxt;
  }
  const int done = t_end - t_beg;
  if (ok && done > 0) {
    if (!mbar_wait(&sm.pv_bar, (done - 1) & 1)) {
      raise_flag(a.status, CSA_FLAG_TIMEOUT);
      ok = false;
    }
  }
  tc_fence_after();
  __syncthreads();
  // ---------------- epilogue ----------------
  // thread: dims d = 128*hsel + 32*q4 + lane (O^T chunk hsel, TMEM lane quarter q4)
  const bool have = ok && done > 0;
  const int d = 128 * hsel + 32 * q4 + lane;
  const uint32_t obase = tO + ((uint32_t)(32 * q4) << 16) + hsel * 64;
  if (a.splits == 1) {
    for (int h0 = 0; h0 < H; h0 += 16) {
      uint32_t v[16];
      if (have) {
        tmem_ld16(obase + h0, v);
        tmem_ld_wait();
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int h = h0 + i;
        const float l = sm.l_run[h];
        const float o = (have && l > 0.0f) ? __uint_as_float(v[i]) / l : 0.0f;
        const __nv_bfloat16 ob = __float2bfloat16_rn(o);
        a.out[((size_t)r * H + h) * D + d] = *reinterpret_cast<const uint16_t*>(&ob);
      }
    }
    if (a.lse && tid < H) {
      const float l = sm.l_run[tid];
      a.lse[(size_t)r * H + tid] = (have && l > 0.0f) ? (sm.m_run[tid] + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
  } else {
    // partial: O [H][512] unnormalised, then m (log2) [H], l [H]
    float* part_out = a.part + ((size_t)r * a.splits + split) * (size_t)H * (D + 2);
    for (int h0 = 0; h0 < H; h0 += 16) {
      uint32_t v[16];
      if (have) {
        tmem_ld16(obase + h0, v);
        tmem_ld_wait();
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) part_out[(size_t)(h0 + i) * D + d] = have ? __uint_as_float(v[i]) : 0.0f;
    }
    if (tid < H) {
      part_out[(size_t)H * D + tid] = have ? sm.m_run[tid] : -INFINITY;
      part_out[(size_t)H * D + H + tid] = have ? sm.l_run[tid] : 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Log-sum-exp merge of the split partials: one block per (row, head).
__global__ void __launch_bounds__(128) k_attn_merge(AttnArgs a) {
  const int r = blockIdx.x / a.H, h = blockIdx.x % a.H;
  const int H = a.H, S = a.splits;
  const float* base = a.part + (size_t)r * S * H * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, base[(size_t)s * H * (D + 2) + (size_t)H * D + h]);
  float L = 0.0f;
  float wts[kMaxTiles];
  for (int s = 0; s < S; ++s) {
    const float ms = base[(size_t)s * H * (D + 2) + (size_t)H * D + h];
    const float ls = base[(size_t)s * H * (D + 2) + (size_t)H * D + H + h];
    wts[s] = (ms == -INFINITY) ? 0.0f : exp2f(ms - M);
    L += wts[s] * ls;
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.0f;
    for (int s = 0; s < S; ++s) acc += wts[s] * base[(size_t)s * H * (D + 2) + (size_t)h * D + d];
    const float o = L > 0.0f ? acc / L : 0.0f;
    const __nv_bfloat16 ob = __float2bfloat16_rn(o);
    a.out[((size_t)r * H + h) * D + d] = *reinterpret_cast<const uint16_t*>(&ob);
  }
  if (threadIdx.x == 0 && a.lse)
    a.lse[(size_t)r * H + h] = (L > 0.0f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

template <int H>
cudaError_t launch_h(const AttnArgs& a, cudaStream_t stream) {
  const size_t smem = sizeof(AttnSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_sparse_attn<H>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_sparse_attn<H><<<a.num_rows * a.splits, kThreads, smem, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  k_attn_merge<<<a.num_rows * a.H, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t attn_partial_bytes(int32_t num_rows, int32_t n_heads, int32_t splits) {
  if (splits <= 1) return 0;
  return sizeof(float) * (size_t)num_rows * splits * n_heads * (D + 2);
}

int32_t attn_choose_splits(int32_t num_rows, int num_sms) {
  if (num_rows <= 0) return 1;
  int s = num_sms / num_rows;
  return s < 1 ? 1 : (s > kMaxTiles ? kMaxTiles : s);
}

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream) {
  if (a.num_rows <= 0) return cudaSuccess;
  switch (a.H) {
    case 16: return launch_h<16>(a, stream);
    case 32: return launch_h<32>(a, stream);
    case 64: return launch_h<64>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csa
