// csa_append: fused pair pooling + FP4 quantisation + paged cache write, and
// the FP8 window write, for the new tokens of a decode / verify step.
//
// [SGL] "DeepSeek-V4.1 Flash on SGLang: from 35 to 873 tokens/s",
//   "Architecture changes and KV cache compression": three global caches pool
//   every two tokens into one entry, the last keeps one entry per token; the
//   entries are FP4, 288 B main KV and 68 B indexer K.
//   "DSpark adaptation and optimization": pair pooling, quantisation and the
//   main-KV write are one kernel, reused for index-K; within a request the
//   previous token is read directly and only the first row needs the saved one.
// [VLLM] "DeepSeek-V4.1-Flash runs 5.3x faster on vLLM...", "SWA bounded
//   replay": the window is uncompressed FP8 over the most recent 128 positions.
//
// One warp per new token.  Lane l owns latent elements 16l..16l+15 (exactly
// one NVFP4 block) and key elements 4l..4l+3 (8 lanes per MXFP4 block).
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

constexpr int kWarps = 8;

// kReadOnly: the source is not written by this kernel (then the read-only
// data path may be used); the pending buffer is read and written in place.
template <bool kReadOnly = true>
__device__ __forceinline__ void load_bf16x16(const uint16_t* src, float (&x)[16]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  const uint4 a = kReadOnly ? __ldg(s) : s[0], b = kReadOnly ? __ldg(s + 1) : s[1];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <bool kReadOnly = true>
__device__ __forceinline__ void load_bf16x4(const uint16_t* src, float (&y)[4]) {
  const uint2* s = reinterpret_cast<const uint2*>(src);
  const uint2 a = kReadOnly ? __ldg(s) : s[0];
  y[0] = __uint_as_float(a.x << 16);
  y[1] = __uint_as_float(a.x & 0xFFFF0000u);
  y[2] = __uint_as_float(a.y << 16);
  y[3] = __uint_as_float(a.y & 0xFFFF0000u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

constexpr int kOffStage = 4096;      // token offsets staged in shared memory

// RMSNorm of a vector spread over the warp, K values per lane (lane l holds
// elements K*l .. K*l+K-1): each lane sums its squares left to right, the 32
// partial sums are combined at lane distance 16, 8, 4, 2, 1 (every lane ends
// with the same sum), then v = (v * r) * gamma with r = 1 / sqrt(ss/dim + eps),
// each step rounded to fp32.
template <int K>
__device__ __forceinline__ void rms_norm(float (&v)[K], const float* gamma, float eps, float inv_dim) {
  float p = 0.0f;
#pragma unroll
  for (int i = 0; i < K; ++i) p = __fadd_rn(p, __fmul_rn(v[i], v[i]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xFFFFFFFFu, p, o));
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(p, inv_dim), eps)));
#pragma unroll
  for (int i = 0; i < K; ++i) v[i] = __fmul_rn(__fmul_rn(v[i], r), __ldg(gamma + i));
}

// Rotate-half RoPE on the last 64 elements of a warp-spread vector, K values
// per lane: the first half (a) sits in lanes [lo, lo + 32/K), the second half
// (b) in the next 32/K lanes, partner = lane xor (32/K).  a' = a*c - b*s,
// b' = b*c + a*s for pair j (products rounded, then the sum).
template <int K>
__device__ __forceinline__ void rope_last64(float (&v)[K], const float* cs, const float* sn, int lane) {
  constexpr int kHalfLanes = 32 / K;              // lanes holding one 32-element half
  constexpr int kLo = 32 - 2 * kHalfLanes;        // first lane of the rotary part
  float other[K];
#pragma unroll
  for (int i = 0; i < K; ++i) other[i] = __shfl_xor_sync(0xFFFFFFFFu, v[i], kHalfLanes);
  if (lane >= kLo) {
    const int jb = K * ((lane - kLo) % kHalfLanes);
    const bool first = lane < kLo + kHalfLanes;
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const float c = __ldg(cs + jb + i), s = __ldg(sn + jb + i);
      v[i] = first ? __fsub_rn(__fmul_rn(v[i], c), __fmul_rn(other[i], s))
                   : __fadd_rn(__fmul_rn(v[i], c), __fmul_rn(other[i], s));
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32) k_append(AppendArgs a) {
  pdl_trigger();                 // csa_step's score prep may start beside it (it reads nothing written here)
  // request lookup table: tok_off staged once per block (one coalesced read
  // instead of a chain of dependent global loads per token)
  __shared__ int32_t s_off[kOffStage + 1];
  const bool staged = a.num_requests + 1 <= kOffStage + 1;
  if (staged)
    for (int i = threadIdx.x; i <= a.num_requests; i += blockDim.x) s_off[i] = __ldg(a.tok_off + i);
  __syncthreads();
  const int t = blockIdx.x * kWarps + warp_id();
  if (t >= a.total_tokens) return;
  const int lane = lane_id();
  // The token's rows, and the previous token's (its pair partner when both are
  // in this call), go out before anything that waits on the request lookup:
  // they depend on t alone.
  float x[16], y[4], xq[16], yq[4];
  load_bf16x16(a.kv_in + (size_t)t * D + lane * 16, x);
  load_bf16x4(a.idx_in + (size_t)t * DI + lane * 4, y);
  if (a.P == 2 && t > 0) {
    load_bf16x16(a.kv_in + (size_t)(t - 1) * D + lane * 16, xq);
    load_bf16x4(a.idx_in + (size_t)(t - 1) * DI + lane * 4, yq);
  }

  // request of token t: the largest b with tok_off[b] <= t
  int lo = 0, hi = a.num_requests - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int v = staged ? s_off[mid] : __ldg(a.tok_off + mid);
    if (v <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int t0 = staged ? s_off[b] : __ldg(a.tok_off + b);
  const int T = (staged ? s_off[b + 1] : __ldg(a.tok_off + b + 1)) - t0;
  const int j = t - t0;
  if (j < 0 || j >= T) {
    if (lane == 0) raise_flag(a.status, CSA_FLAG_APPEND);
    return;
  }
  const int p0 = __ldg(a.pos0 + b);
  const int p = p0 + j;
  if (p0 < 0 || p < 0) {
    if (lane == 0) raise_flag(a.status, CSA_FLAG_APPEND);
    return;
  }

  // ---- FP8 window slot of this token: scale = amax / 448, codes = E4M3(x / scale).
  // Only the last win_cap tokens of the request in this call are written: an
  // older token's slot is taken by a newer one of the same call, and writing
  // both would race.
  if (a.win_codes != nullptr && j >= T - a.win_cap) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = warp_max(amax);
    const size_t slot = (size_t)b * a.win_cap + (size_t)(p % a.win_cap);
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
    float s = 0.0f;
    if (amax != 0.0f) {
      s = __fdiv_rn(amax, 448.0f);
#pragma unroll
      for (int i = 0; i < 16; ++i) packed[i >> 2] |= e4m3_rne_sat(__fdiv_rn(x[i], s)) << (8 * (i & 3));
    }
    *reinterpret_cast<uint4*>(a.win_codes + slot * D + lane * 16) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if (lane == 0) a.win_scale[slot] = s;
  }

  // ---- cache entry completed by this token
  if (p % a.P == a.P - 1) {
    const int e = p / a.P;
    if (a.P == 2) {
      // the pair partner: the request's pending token, or the previous token
      if (j == 0) {
        load_bf16x16<false>(a.pending + (size_t)b * (D + DI) + lane * 16, xq);
        load_bf16x4<false>(a.pending + (size_t)b * (D + DI) + D + lane * 4, yq);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = (xq[i] + x[i]) * 0.5f;
#pragma unroll
      for (int i = 0; i < 4; ++i) y[i] = (yq[i] + y[i]) * 0.5f;
    }
    // ---- compressor steps on the pooled entry (csa_append_compress)
    bool write_entry = true;
    if (a.kv_gamma) rms_norm<16>(x, a.kv_gamma + lane * 16, a.eps, 1.0f / 512.0f);
    if (a.idx_gamma) rms_norm<4>(y, a.idx_gamma + lane * 4, a.eps, 1.0f / 128.0f);
    if (a.rope_cos) {
      if (p >= a.rope_rows) {      // p: the position of the entry's last token
        if (lane == 0) raise_flag(a.status, CSA_FLAG_APPEND);
        write_entry = false;
      } else {
        const float* cs = a.rope_cos + (size_t)p * 32;
        const float* sn = a.rope_sin + (size_t)p * 32;
        rope_last64<16>(x, cs, sn, lane);
        rope_last64<4>(y, cs, sn, lane);
      }
    }
    const int lp = e / PAGE, slot = e % PAGE;
    int page = -1;
    if (lp < a.max_pages) page = __ldg(a.page_table + (size_t)b * a.max_pages + lp);
    if (page < 0 || page >= a.num_pages) {
      if (lane == 0) raise_flag(a.status, CSA_FLAG_PAGE_OOB);
    } else if (write_entry) {
      // NVFP4 block (this lane's 16 values): S = E4M3(amax/6), codes = e2m1(x/s)
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
      const uint32_t S = e4m3_rne_sat(__fdiv_rn(amax, 6.0f));
      const float s = e4m3_value(S);
      uint32_t lo32 = 0u, hi32 = 0u;
      if (s != 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) lo32 |= e2m1_rne(__fdiv_rn(x[i], s)) << (4 * i);
#pragma unroll
        for (int i = 0; i < 8; ++i) hi32 |= e2m1_rne(__fdiv_rn(x[8 + i], s)) << (4 * i);
      }
      uint8_t* kvp = a.kv_pool + (size_t)page * KV_PAGE;
      *reinterpret_cast<uint2*>(kvp + slot * 256 + lane * 8) = make_uint2(lo32, hi32);
      kvp[KV_SCALE_OFF + slot * 32 + lane] = (uint8_t)S;

      // MXFP4 block of 32 = lanes 8k..8k+7: scale 2^E, E = floor(log2 amax) - 2
      float am = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 4));
      const uint32_t E8 = e8m0_block_code(am);
      uint32_t codes = 0u;
      if (am != 0.0f) {
        const float inv = e8m0_inv_scale(E8);
#pragma unroll
        for (int i = 0; i < 4; ++i) codes |= e2m1_rne(y[i] * inv) << (4 * i);
      }
      uint8_t* ixp = a.idx_pool + (size_t)page * IDX_PAGE;
      *reinterpret_cast<uint16_t*>(ixp + idx_data_off(slot, 2 * lane)) = (uint16_t)codes;
      if ((lane & 7) == 0) ixp[idx_scale_off(slot, lane >> 3)] = (uint8_t)E8;
    }
  }

  // ---- pending token: written by the warp of the request's first new token,
  // after its own read of the old pending token (so in-place is safe).
  if (a.P == 2 && j == 0 && ((p0 + T - 1) & 1) == 0) {
    __syncwarp();
    const size_t tl = (size_t)t0 + T - 1;
    const uint4* skv = reinterpret_cast<const uint4*>(a.kv_in + tl * D);
    const uint4* six = reinterpret_cast<const uint4*>(a.idx_in + tl * DI);
    uint4* dst = reinterpret_cast<uint4*>(a.pending + (size_t)b * (D + DI));
    dst[lane] = __ldg(skv + lane);
    dst[32 + lane] = __ldg(skv + 32 + lane);
    if (lane < 16) dst[64 + lane] = __ldg(six + lane);
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
  if (a.total_tokens <= 0) return cudaSuccess;
  const int blocks = (a.total_tokens + kWarps - 1) / kWarps;
  k_append<<<blocks, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace csa
