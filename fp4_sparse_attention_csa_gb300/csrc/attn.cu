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
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

constexpr int kThreads = 256;
constexpr int kTileKeys = 128;
constexpr int kMaxTiles = TOPK / kTileKeys + 1;   // 4 global + 1 window
constexpr int kMaxH = CSA_MAX_HEADS;             // 64
constexpr float kLog2e = 1.4426950408889634f;

struct AttnSmem {
  uint8_t k[kTileKeys * D * 2];        // 131072, 1024-aligned: kc*16384 + (key/8)*1024 + (key%8)*128
  uint8_t q[kMaxH * D * 2];            // 65536: kc*(H*128) + (h/8)*1024 + (h%8)*128
  uint8_t p[kTileKeys * 128];          // 16384: (key/8)*1024 + (key%8)*128, heads along the row
  __half2 e2m1_pair[256];              // byte -> (lo nibble, hi nibble) values
  float e4m3_tab[256];
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

// In-warp reduction of NV values per lane (NV = 8, 16 or 32) across the 32
// lanes: recursive halving, then a butterfly over the remaining lane bits.
// Lane l ends with the reduction of value index (l >> (5 - log2 NV)).
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
  // lanes that share the value index: reduce over the low lane bits
  constexpr int kShift = (NV == 32) ? 0 : (NV == 16 ? 1 : 2);
#pragma unroll
  for (int o = 1; o < (1 << kShift); o <<= 1) {
    const float y = __shfl_xor_sync(0xFFFFFFFFu, x, o);
    x = kMax ? fmaxf(x, y) : x + y;
  }
  return x;
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1) k_sparse_attn(AttnArgs a) {
  constexpr int HH = H / 2;                       // heads per thread in the softmax
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

  // ---- setup: tables, barriers, TMEM, Q (bf16 -> fp16, K-major 128B swizzle)
  {
    const uint32_t lo = tid & 15, hi = tid >> 4;
    sm.e2m1_pair[tid] = __floats2half2_rn(e2m1_value(lo), e2m1_value(hi));
    sm.e4m3_tab[tid] = e4m3_value((uint32_t)tid);
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

  const int key = tid & (kTileKeys - 1), khalf = tid >> 7;   // gather role
  const int q4 = warp & 3, hsel = warp >> 2;                  // TMEM role: lane quarter, head half
  const int mykey = 32 * q4 + lane;
  bool ok = true;

  for (int t = t_beg; t < t_end && ok; ++t) {
    const int it = t - t_beg;
    if (it > 0 && !mbar_wait(&sm.pv_bar, (it - 1) & 1)) { raise_flag(a.status, CSA_FLAG_TIMEOUT); ok = false; break; }
    // ---------------- gather + dequantise this tile into sm.k ----------------
    const bool is_win = has_win && (t == ntiles - 1);
    uint8_t* krow_base = sm.k + (key >> 3) * 1024;
    if (!is_win) {
      const int j = t * kTileKeys + key;
      int e = (j < nsel) ? __ldg(a.topk + (size_t)r * TOPK + j) : -1;
      const uint8_t* src = nullptr;
      if (e >= 0) {
        if (e >= n || e / PAGE >= a.max_pages) {
          raise_flag(a.status, CSA_FLAG_TOPK_OOB);
        } else {
          const int pg = __ldg(a.page_table + (size_t)b * a.max_pages + e / PAGE);
          if (pg < 0 || pg >= a.num_pages) raise_flag(a.status, CSA_FLAG_PAGE_OOB);
          else src = a.kv_pool + (size_t)pg * KV_PAGE;
        }
      }
      if (khalf == 0) sm.mu[key] = src ? 1.0f : 0.0f;
      uint4 data[8], sc;
      if (src) {
        const uint4* dp = reinterpret_cast<const uint4*>(src + (e % PAGE) * 256 + khalf * 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) data[i] = __ldg(dp + i);
        sc = __ldg(reinterpret_cast<const uint4*>(src + KV_SCALE_OFF + (e % PAGE) * 32 + khalf * 16));
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) data[i] = make_uint4(0u, 0u, 0u, 0u);
        sc = make_uint4(0u, 0u, 0u, 0u);
      }
      const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
      // 128 data bytes = 256 dims = 4 atom columns of 64 dims; 16 B of data = 32 dims = 2 scale blocks
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t w4[4] = {data[i].x, data[i].y, data[i].z, data[i].w};
        // data[i] covers dims 256*khalf + 32*i .. +32, scale blocks 2i, 2i+1
        const uint32_t s0 = (scw[(2 * i) >> 2] >> (8 * ((2 * i) & 3))) & 0xFFu;
        const uint32_t s1 = (scw[(2 * i + 1) >> 2] >> (8 * ((2 * i + 1) & 3))) & 0xFFu;
        const __half2 hs0 = __float2half2_rn(sm.e4m3_tab[s0]);
        const __half2 hs1 = __float2half2_rn(sm.e4m3_tab[s1]);
        uint32_t o[16];
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          const __half2 hs = (wd < 2) ? hs0 : hs1;
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const __half2 v = __hmul2(sm.e2m1_pair[(w4[wd] >> (8 * bb)) & 0xFFu], hs);
            o[wd * 4 + bb] = *reinterpret_cast<const uint32_t*>(&v);
          }
        }
        const int dim0 = 256 * khalf + 32 * i;          // 32 dims = 4 chunks of 8
        const int kc = dim0 >> 6, ch0 = (dim0 & 63) >> 3;
        uint8_t* dst = krow_base + kc * 16384;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(dst + swz128(key & 7, ch0 + c)) =
              make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
      }
    } else {
      const int lo_pos = max(0, pos - (WIN - 1));
      const int p = lo_pos + key;
      const bool valid = p <= pos;
      uint4 data[16];
      float s = 0.0f;
      if (valid) {
        const size_t slot = (size_t)b * a.win_cap + (size_t)(p % a.win_cap);
        const uint4* dp = reinterpret_cast<const uint4*>(a.win_codes + slot * D + khalf * 256);
#pragma unroll
        for (int i = 0; i < 16; ++i) data[i] = __ldg(dp + i);
        s = __ldg(a.win_scale + slot);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) data[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      // s = 2^e * mu, mu in [1, 2): the codes are scaled by 2^e (exact in fp16)
      float pow2 = 0.0f, mu = 0.0f;
      if (s > 0.0f) {
        pow2 = __uint_as_float(__float_as_uint(s) & 0x7F800000u);
        mu = s / pow2;
      }
      if (khalf == 0) sm.mu[key] = valid ? mu : 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {       // 16 codes = 16 dims = 2 chunks
        const uint32_t w4[4] = {data[i].x, data[i].y, data[i].z, data[i].w};
        uint32_t o[8];
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t c0 = (w4[wd] >> (16 * hh)) & 0xFFu, c1 = (w4[wd] >> (16 * hh + 8)) & 0xFFu;
            const __half2 v = __floats2half2_rn(sm.e4m3_tab[c0] * pow2, sm.e4m3_tab[c1] * pow2);
            o[wd * 2 + hh] = *reinterpret_cast<const uint32_t*>(&v);
          }
        }
        const int dim0 = 256 * khalf + 16 * i;
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
#pragma unroll
      for (int c = 0; c < HH; c += 16) {
        uint32_t v[16];
        if constexpr (HH >= 16) {
          tmem_ld16(base + c, v);
        } else {
          uint32_t v4[4];
          tmem_ld4(base + c, v4);
          uint32_t v4b[4];
          tmem_ld4(base + c + 4, v4b);
#pragma unroll
          for (int i = 0; i < 4; ++i) { v[i] = v4[i]; v[4 + i] = v4b[i]; }
        }
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c + i < HH) lg[c + i] = __uint_as_float(v[i]);
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
    {
      const float mx = warp_reduce_many<HH, true>(tmp, lane);
      constexpr int kShift = (HH == 32) ? 0 : (HH == 16 ? 1 : 2);
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
#pragma unroll
      for (int c = 0; c < HH / 8; ++c) {
        const int chunk = (hsel * HH) / 8 + c;
        *reinterpret_cast<uint4*>(prow + swz128(mykey & 7, chunk)) =
            make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
      }
    }
    {
      const float sum = warp_reduce_many<HH, false>(tmp, lane);
      constexpr int kShift = (HH == 32) ? 0 : (HH == 16 ? 1 : 2);
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
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int chunk = 2 * hsel + cc;
        const uint32_t base = tO + ((uint32_t)(32 * q4) << 16) + chunk * 64;
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
  // thread: dims d = chunk*128 + 32*q4 + lane for chunks 2*hsel, 2*hsel+1
  const bool have = ok && done > 0;
  if (a.splits == 1) {
    for (int cc = 0; cc < 2; ++cc) {
      const int chunk = 2 * hsel + cc;
      const int d = chunk * 128 + 32 * q4 + lane;
      const uint32_t base = tO + ((uint32_t)(32 * q4) << 16) + chunk * 64;
      for (int h0 = 0; h0 < H; h0 += 16) {
        uint32_t v[16];
        if (have) {
          tmem_ld16(base + h0, v);
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
    }
    if (a.lse && tid < H) {
      const float l = sm.l_run[tid];
      a.lse[(size_t)r * H + tid] = (have && l > 0.0f) ? (sm.m_run[tid] + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
  } else {
    // partial: O [H][512] unnormalised, then m (log2) [H], l [H]
    float* part = a.part + ((size_t)r * a.splits + split) * (size_t)H * (D + 2);
    for (int cc = 0; cc < 2; ++cc) {
      const int chunk = 2 * hsel + cc;
      const int d = chunk * 128 + 32 * q4 + lane;
      const uint32_t base = tO + ((uint32_t)(32 * q4) << 16) + chunk * 64;
      for (int h0 = 0; h0 < H; h0 += 16) {
        uint32_t v[16];
        if (have) {
          tmem_ld16(base + h0, v);
          tmem_ld_wait();
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) part[(size_t)(h0 + i) * D + d] = have ? __uint_as_float(v[i]) : 0.0f;
      }
    }
    if (tid < H) {
      part[(size_t)H * D + tid] = have ? sm.m_run[tid] : -INFINITY;
      part[(size_t)H * D + H + tid] = have ? sm.l_run[tid] : 0.0f;
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
