/*
 * CPU oracle for the CSA decode path -- TEST INFRASTRUCTURE ONLY (see
 * csa_oracle.h for the sources, the precision rules and the pin status).
 *
 * Plain scalar C, fp32, no SIMD, no fast-math, built with -ffp-contract=off.
 * Every step follows the definitions in the order they are stated; nothing
 * is blocked, fused or reordered.
 */
#include "csa_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---- format constants, restated (not shared with the CUDA library) -----
 * [SGL] "Architecture changes and KV cache compression": a main-KV entry is
 * 288 bytes and an indexer-K entry 68 bytes.  Main KV = 512 e2m1 values
 * (256 B) + one E4M3 scale per 16 values (32 B); indexer K = 128 e2m1 values
 * (64 B) + one E8M0 scale per 32 values (4 B).  Pages hold 64 entries:
 *   main-KV page 18432 B: entry e data at 256*e, scales at 16384 + 32*e
 *   indexer page  4352 B: 8 groups of 544 B, group g = entries 8g..8g+7:
 *     data byte k (0..63) of entry 8g+r at 544*g + 128*(k/16) + 16*r + k%16,
 *     scale byte b (0..3) of entry 8g+r at 544*g + 512 + 4*r + b.
 * Element 2j sits in the low nibble of byte j, element 2j+1 in the high one. */
#define OR_D            512
#define OR_DI           128
#define OR_PAGE         64
#define OR_KV_PAGE      18432
#define OR_KV_SCALE_OFF 16384
#define OR_IDX_PAGE     4352
#define OR_IDX_GROUP    544

/* byte offsets of an indexer entry's data byte k / scale byte b in its page */
static int64_t idx_data_off(int64_t slot, int k) {
  return OR_IDX_GROUP * (slot / 8) + 128 * (k / 16) + 16 * (slot % 8) + k % 16;
}
static int64_t idx_scale_off(int64_t slot, int b) {
  return OR_IDX_GROUP * (slot / 8) + 512 + 4 * (slot % 8) + b;
}
#define OR_TOPK         512
#define OR_WINDOW       128

/* ======================================================================
 * Element codes ([OCP] MX v1.0 and OCP FP8)
 * ====================================================================== */

/* E2M1 magnitudes for codes 0..7; bit 3 of the code is the sign. */
static const float E2M1_MAG[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float or_e2m1_decode(uint8_t code) {
  float m = E2M1_MAG[code & 7];
  return (code & 8) ? -m : m;
}

/* Round to nearest grid value; a tie between two neighbours goes to the one
 * with the even code (round-half-to-even on the 3-bit magnitude).  Values
 * beyond 6 land on 6 (the nearest grid point), i.e. saturation.  The sign bit
 * is copied from the input, so a negative value that rounds to zero gives
 * code 0x8.  Distances are taken in double, where they are exact. */
uint8_t or_e2m1_encode(float v) {
  uint8_t sign = signbit(v) ? 8 : 0;
  double a = fabs((double)v);
  int best = 0;
  for (int k = 1; k < 8; ++k) {
    double dk = fabs(a - (double)E2M1_MAG[k]);
    double db = fabs(a - (double)E2M1_MAG[best]);
    if (dk < db || (dk == db && (k % 2) == 0)) best = k;
  }
  return (uint8_t)(sign | best);
}

/* E4M3 "fn": sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent
 * field 0 holds subnormals m * 2^-9; S.1111.111 is NaN; no infinities. */
float or_e4m3_decode(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  float v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexpf((float)m, -9);
  else        v = ldexpf(1.0f + (float)m / 8.0f, e - 7);
  return s ? -v : v;
}

/* Nearest finite E4M3 value, ties to the even code, |v| >= 448 -> 448.
 * Magnitude codes 0..126 are monotone in value, so a binary search finds the
 * neighbours.  Sign copied from the input (negative underflow -> 0x80). */
uint8_t or_e4m3_encode(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0;
  double a = fabs((double)v);
  int mag;
  if (a >= 448.0) {
    mag = 126;
  } else {
    int lo = 0, hi = 126;          /* largest code whose value is <= a */
    while (lo < hi) {
      int mid = (lo + hi + 1) / 2;
      if ((double)or_e4m3_decode((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
    }
    double dl = a - (double)or_e4m3_decode((uint8_t)lo);
    double dh = (double)or_e4m3_decode((uint8_t)(lo + 1)) - a;
    if (dl < dh) mag = lo;
    else if (dh < dl) mag = lo + 1;
    else mag = (lo % 2 == 0) ? lo : lo + 1;
  }
  return (uint8_t)(sign | mag);
}

/* E8M0: 2^(code-127); code 255 is NaN. */
float or_e8m0_decode(uint8_t code) {
  if (code == 255) return NAN;
  return ldexpf(1.0f, (int)code - 127);
}

/* [OCP] MX v1.0 scale rule for an FP4 (E2M1, emax = 2) element type:
 * E = floor(log2(amax)) - 2, clamped to the E8M0 range, code = E + 127.
 * frexp gives amax = m * 2^e with m in [0.5, 1), so floor(log2 amax) = e - 1.
 * amax == 0 gives code 0. */
uint8_t or_e8m0_block_code(float amax) {
  if (amax == 0.0f) return 0;
  int e;
  (void)frexpf(amax, &e);
  int E = (e - 1) - 2;
  if (E < -127) E = -127;
  if (E > 127) E = 127;
  return (uint8_t)(E + 127);
}

float or_bf16_to_f32(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ======================================================================
 * Block quantisers
 * ====================================================================== */

/* NVFP4 (16 values, one E4M3 scale): s_f = amax / 6 (IEEE division),
 * S = E4M3(s_f), s = decode(S); code_i = e2m1(x_i / s); s == 0 -> all 0. */
void or_nvfp4_block(const float* x16, uint8_t* codes16, uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x16[i]));
  float sf = amax / 6.0f;
  uint8_t S = or_e4m3_encode(sf);
  float s = or_e4m3_decode(S);
  *scale = S;
  for (int i = 0; i < 16; ++i) codes16[i] = (s == 0.0f) ? 0 : or_e2m1_encode(x16[i] / s);
}

/* MXFP4 (32 values, one E8M0 scale), [OCP] MX v1.0 conversion: the scale
 * is 2^E with E from the block's amax; each element is x * 2^-E (exact)
 * rounded to E2M1 with saturation.  amax == 0 -> scale code 0, codes 0. */
void or_mxfp4_block(const float* x32, uint8_t* codes32, uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x32[i]));
  uint8_t code = or_e8m0_block_code(amax);
  *scale = code;
  if (amax == 0.0f) {
    for (int i = 0; i < 32; ++i) codes32[i] = 0;
    return;
  }
  int E = (int)code - 127;
  for (int i = 0; i < 32; ++i) codes32[i] = or_e2m1_encode(ldexpf(x32[i], -E));
}

static void pack_nibbles(const uint8_t* codes, int n, uint8_t* out) {
  for (int j = 0; j < n / 2; ++j)
    out[j] = (uint8_t)((codes[2 * j] & 15) | ((codes[2 * j + 1] & 15) << 4));
}

static uint8_t nibble(const uint8_t* data, int k) {
  uint8_t byte = data[k / 2];
  return (k % 2 == 0) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4);
}

void or_quant_main_entry(const float* x512, uint8_t* data256, uint8_t* scale32) {
  uint8_t codes[OR_D];
  for (int b = 0; b < OR_D / 16; ++b) or_nvfp4_block(x512 + 16 * b, codes + 16 * b, scale32 + b);
  pack_nibbles(codes, OR_D, data256);
}

void or_quant_idx_entry(const float* y128, uint8_t* data64, uint8_t* scale4) {
  uint8_t codes[OR_DI];
  for (int b = 0; b < OR_DI / 32; ++b) or_mxfp4_block(y128 + 32 * b, codes + 32 * b, scale4 + b);
  pack_nibbles(codes, OR_DI, data64);
}

/* [VLLM] "SWA bounded replay": the local window is uncompressed FP8 over the
 * most recent 128 positions.  One fp32 scale per token: scale = amax / 448,
 * codes = E4M3(x / scale); amax == 0 gives scale 0 and codes 0. */
void or_quant_window_token(const float* x512, uint8_t* codes512, float* scale) {
  float amax = 0.0f;
  for (int i = 0; i < OR_D; ++i) amax = fmaxf(amax, fabsf(x512[i]));
  if (amax == 0.0f) {
    *scale = 0.0f;
    for (int i = 0; i < OR_D; ++i) codes512[i] = 0;
    return;
  }
  float s = amax / 448.0f;
  *scale = s;
  for (int i = 0; i < OR_D; ++i) codes512[i] = or_e4m3_encode(x512[i] / s);
}

/* ======================================================================
 * Append: pair pooling + quantisation + cache write
 * [SGL] "Architecture changes and KV cache compression" (three caches pool
 * every two tokens into one entry, the last keeps one entry per token) and
 * "DSpark adaptation and optimization" (pair pooling, quantisation and the
 * main-KV write fused; within a request the previous token is read directly,
 * only the first new token needs the saved one).
 * Entry e = floor(p / P) is written when its last token (p % P == P-1)
 * arrives; x = (t_{2e} + t_{2e+1}) * 0.5 in fp32 for P = 2, x = t for P = 1.
 * An unpaired last token is saved to pending_out.
 * ====================================================================== */

static void load_token(const uint16_t* kv_in, const uint16_t* idx_in, int64_t t,
                       float* x512, float* y128) {
  for (int d = 0; d < OR_D; ++d) x512[d] = or_bf16_to_f32(kv_in[t * OR_D + d]);
  for (int d = 0; d < OR_DI; ++d) y128[d] = or_bf16_to_f32(idx_in[t * OR_DI + d]);
}

/* ======================================================================
 * Compressor steps on a pooled entry ([SGL] "DSpark adaptation and
 * optimization": pooling, RMSNorm, RoPE and quantisation fused in one step,
 * reused for the indexer key).  The pages name the steps but give neither the
 * weights nor a rotary convention; the readings used here:
 *   RMSNorm   v_i = (v_i * r) * gamma_i, r = 1 / sqrt(ms + eps), ms = ss / dim,
 *             every product, sum, square root and quotient rounded to fp32
 *             once (IEEE, no fused multiply-add).  ss, the sum of squares, is
 *             taken in one fixed order: the vector is cut into 32 contiguous
 *             parts of dim/32 values, each part summed left to right, then the
 *             32 part sums are combined pairwise at distance 16, 8, 4, 2, 1
 *             (s_l <- s_l + s_(l xor d)).  Every sum of this tree is the same
 *             in all 32 positions, so the tree defines one value.
 *   RoPE      rotate-half on the last 64 dims: for j < 32, with a = v[dim-64+j],
 *             b = v[dim-32+j], c = cos[j], s = sin[j]:
 *             a' = a*c - b*s,  b' = b*c + a*s  (products rounded, then the sum).
 * ====================================================================== */
void or_compress_vec(float* v, int dim, const float* gamma, float eps, const float* cos32,
                     const float* sin32) {
  if (gamma != NULL) {
    const int k = dim / 32;
    float part[32], next[32];
    for (int l = 0; l < 32; ++l) {
      float p = 0.0f;
      for (int i = 0; i < k; ++i) {
        const float sq = v[l * k + i] * v[l * k + i];
        p = p + sq;
      }
      part[l] = p;
    }
    for (int d = 16; d >= 1; d >>= 1) {
      for (int l = 0; l < 32; ++l) next[l] = part[l] + part[l ^ d];
      memcpy(part, next, sizeof(part));
    }
    const float ms = part[0] * (1.0f / (float)dim);      /* dim is a power of two: exact */
    const float den = sqrtf(ms + eps);
    const float r = 1.0f / den;
    for (int i = 0; i < dim; ++i) {
      const float t = v[i] * r;
      v[i] = t * gamma[i];
    }
  }
  if (cos32 != NULL && sin32 != NULL) {
    for (int j = 0; j < 32; ++j) {
      const float a = v[dim - 64 + j], b = v[dim - 32 + j];
      const float ac = a * cos32[j], bs = b * sin32[j], bc = b * cos32[j], as = a * sin32[j];
      v[dim - 64 + j] = ac - bs;
      v[dim - 32 + j] = bc + as;
    }
  }
}

int or_append(const or_cache_t* c, const int32_t* pos0, const int32_t* tok_off,
              const uint16_t* kv_in, const uint16_t* idx_in,
              const uint16_t* pending_in, uint16_t* pending_out) {
  return or_append_compress(c, pos0, tok_off, kv_in, idx_in, pending_in, pending_out, NULL);
}

int or_append_compress(const or_cache_t* c, const int32_t* pos0, const int32_t* tok_off,
                       const uint16_t* kv_in, const uint16_t* idx_in,
                       const uint16_t* pending_in, uint16_t* pending_out, const or_compress_t* cmp) {
  int status = 0;
  const int P = c->pool_ratio;
  float x[OR_D], y[OR_DI], xp[OR_D], yp[OR_DI];
  for (int b = 0; b < c->num_requests; ++b) {
    int64_t t0 = tok_off[b], T = (int64_t)tok_off[b + 1] - tok_off[b];
    uint16_t saved[OR_D + OR_DI];
    int have_saved = 0;
    if (P == 2 && T > 0 && (pos0[b] % 2) == 1) {          /* read before any write */
      memcpy(saved, pending_in + (int64_t)b * (OR_D + OR_DI), sizeof(saved));
      have_saved = 1;
    }
    for (int64_t j = 0; j < T; ++j) {
      int64_t p = (int64_t)pos0[b] + j, t = t0 + j;
      load_token(kv_in, idx_in, t, x, y);
      if (c->win_codes != NULL) {
        int64_t slot = (int64_t)b * c->win_cap + p % c->win_cap;
        or_quant_window_token(x, c->win_codes + slot * OR_D, c->win_scale + slot);
      }
      if (p % P != P - 1) continue;
      int64_t e = p / P;
      if (P == 2) {
        if (j == 0) {
          if (!have_saved) { status = -2; continue; }
          for (int d = 0; d < OR_D; ++d) xp[d] = or_bf16_to_f32(saved[d]);
          for (int d = 0; d < OR_DI; ++d) yp[d] = or_bf16_to_f32(saved[OR_D + d]);
        } else {
          load_token(kv_in, idx_in, t - 1, xp, yp);
        }
        for (int d = 0; d < OR_D; ++d) x[d] = (xp[d] + x[d]) * 0.5f;
        for (int d = 0; d < OR_DI; ++d) y[d] = (yp[d] + y[d]) * 0.5f;
      }
      int64_t lp = e / OR_PAGE, slot = e % OR_PAGE;
      if (lp >= c->max_pages_per_req) { status = -1; continue; }
      int32_t page = c->page_table[(int64_t)b * c->max_pages_per_req + lp];
      if (page < 0 || page >= c->num_pages) { status = -1; continue; }
      if (cmp != NULL) {
        const int64_t rp = e * P + (P - 1);          /* position of the entry's last token */
        const float* cs = NULL;
        const float* sn = NULL;
        if (cmp->rope_cos != NULL && cmp->rope_sin != NULL) {
          if (rp >= cmp->rope_rows) { status = -3; continue; }
          cs = cmp->rope_cos + rp * 32;
          sn = cmp->rope_sin + rp * 32;
        }
        or_compress_vec(x, OR_D, cmp->kv_gamma, cmp->eps, cs, sn);
        or_compress_vec(y, OR_DI, cmp->idx_gamma, cmp->eps, cs, sn);
      }
      uint8_t* kvp = c->kv_pool + (int64_t)page * OR_KV_PAGE;
      uint8_t* ixp = c->idx_pool + (int64_t)page * OR_IDX_PAGE;
      or_quant_main_entry(x, kvp + slot * 256, kvp + OR_KV_SCALE_OFF + slot * 32);
      uint8_t idata[64], iscale[4];
      or_quant_idx_entry(y, idata, iscale);
      for (int k = 0; k < 64; ++k) ixp[idx_data_off(slot, k)] = idata[k];
      for (int b2 = 0; b2 < 4; ++b2) ixp[idx_scale_off(slot, b2)] = iscale[b2];
    }
    if (P == 2 && T > 0 && ((pos0[b] + T - 1) % 2) == 0) {
      uint16_t* dst = pending_out + (int64_t)b * (OR_D + OR_DI);
      int64_t t = t0 + T - 1;
      memcpy(dst, kv_in + t * OR_D, OR_D * sizeof(uint16_t));
      memcpy(dst + OR_D, idx_in + t * OR_DI, OR_DI * sizeof(uint16_t));
    }
  }
  return status;
}

/* ======================================================================
 * Indexer score
 * score(i) = sum_h w_h * relu(q_h . k_i) over the FP4 indexer cache, with
 * q_h quantised to MXFP4 per head (a block-scaled FP4 product needs FP4 on
 * both sides).  [SGL] "Architecture changes..." (CSA2 scores the indexer K
 * so that only the top 512 global positions take part in attention).
 * dot = sequential fp32 sum over d; score = sequential fp32 sum over h.
 * A row at position t sees entries e < floor((t+1)/P) (complete entries).
 * ====================================================================== */

static int32_t row_visible(int32_t pos, int32_t P) { return (pos + 1) / P; }

static void dequant_idx_entry(const or_cache_t* c, int32_t req, int32_t e, float* k128) {
  int32_t page = c->page_table[(int64_t)req * c->max_pages_per_req + e / OR_PAGE];
  const uint8_t* ixp = c->idx_pool + (int64_t)page * OR_IDX_PAGE;
  uint8_t data[64], sc[4];
  for (int k = 0; k < 64; ++k) data[k] = ixp[idx_data_off(e % OR_PAGE, k)];
  for (int b = 0; b < 4; ++b) sc[b] = ixp[idx_scale_off(e % OR_PAGE, b)];
  for (int d = 0; d < OR_DI; ++d) k128[d] = or_e2m1_decode(nibble(data, d)) * or_e8m0_decode(sc[d / 32]);
}

static void quant_dequant_q_idx(const uint16_t* q128, float* qhat) {
  float qf[OR_DI];
  uint8_t codes[32], sc;
  for (int d = 0; d < OR_DI; ++d) qf[d] = or_bf16_to_f32(q128[d]);
  for (int b = 0; b < OR_DI / 32; ++b) {
    or_mxfp4_block(qf + 32 * b, codes, &sc);
    for (int i = 0; i < 32; ++i) qhat[32 * b + i] = or_e2m1_decode(codes[i]) * or_e8m0_decode(sc);
  }
}

static void score_one_row(const or_cache_t* c, int32_t req, int32_t pos, int32_t Hi,
                          const uint16_t* q_idx_row, const float* w_row, float* out) {
  int32_t n = row_visible(pos, c->pool_ratio);
  float* qhat = (float*)malloc(sizeof(float) * (size_t)Hi * OR_DI);
  float k[OR_DI];
  for (int h = 0; h < Hi; ++h) quant_dequant_q_idx(q_idx_row + (int64_t)h * OR_DI, qhat + (int64_t)h * OR_DI);
  for (int32_t i = 0; i < n; ++i) {
    dequant_idx_entry(c, req, i, k);
    float score = 0.0f;
    for (int h = 0; h < Hi; ++h) {
      float dot = 0.0f;
      for (int d = 0; d < OR_DI; ++d) dot = dot + qhat[(int64_t)h * OR_DI + d] * k[d];
      float r = dot > 0.0f ? dot : 0.0f;
      score = score + w_row[h] * r;
    }
    out[i] = score;
  }
  free(qhat);
}

void or_index_score(const or_cache_t* c, int32_t num_rows, const int32_t* row_req,
                    const int32_t* row_pos, int32_t n_idx_heads,
                    const uint16_t* q_idx, const float* w, float* scores, int64_t ld) {
  for (int32_t r = 0; r < num_rows; ++r)
    score_one_row(c, row_req[r], row_pos[r], n_idx_heads,
                  q_idx + (int64_t)r * n_idx_heads * OR_DI, w + (int64_t)r * n_idx_heads,
                  scores + (int64_t)r * ld);
}

/* ======================================================================
 * Exact top-512: sort by (score descending, index ascending), keep the first
 * min(512, n), return them in ascending index order padded with -1.
 * [SGL] "Architecture changes...": only the top 512 global positions take
 * part in attention; ties go to the lower index.
 * ====================================================================== */

typedef struct { float s; int32_t i; } or_pair_t;

static int cmp_pair(const void* a, const void* b) {
  const or_pair_t* x = (const or_pair_t*)a;
  const or_pair_t* y = (const or_pair_t*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->i < y->i) ? -1 : (x->i > y->i);
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

void or_topk_row(const float* scores, int32_t n, int32_t* out512) {
  int32_t k = n < OR_TOPK ? n : OR_TOPK;
  if (n > 0) {
    or_pair_t* v = (or_pair_t*)malloc(sizeof(or_pair_t) * (size_t)n);
    for (int32_t i = 0; i < n; ++i) { v[i].s = scores[i]; v[i].i = i; }
    qsort(v, (size_t)n, sizeof(or_pair_t), cmp_pair);
    for (int32_t j = 0; j < k; ++j) out512[j] = v[j].i;
    free(v);
    qsort(out512, (size_t)k, sizeof(int32_t), cmp_i32);
  }
  for (int32_t j = k; j < OR_TOPK; ++j) out512[j] = -1;
}

/* ======================================================================
 * Two-level candidate filter (NEXT f-2; [SGL] "Architecture changes and KV
 * cache compression": CSA2 narrows the indexer's search before the top 512;
 * "DSpark adaptation and optimization": chosen candidate blocks expand
 * straight into a token mask).  The pages give no block size or block score;
 * the reading used here:
 *   1. a block is a page of 64 entries, block b = entries 64b .. 64b+63 (< n);
 *   2. its score is the largest score among its entries;
 *   3. the blocks are ordered by (block score descending, block index
 *      ascending) and the first `blocks` of them are kept;
 *   4. the candidates are the entries of the kept blocks; among them the 512
 *      largest by (score descending, index ascending) are returned in
 *      ascending index order, padded with -1.
 * ====================================================================== */
void or_topk_two_level(const float* scores, int32_t n, int32_t blocks, int32_t* out512) {
  const int32_t nb = (n + OR_PAGE - 1) / OR_PAGE;
  or_pair_t* bs = (or_pair_t*)malloc(sizeof(or_pair_t) * (size_t)(nb > 0 ? nb : 1));
  for (int32_t b = 0; b < nb; ++b) {
    float m = scores[(int64_t)b * OR_PAGE];
    for (int32_t i = b * OR_PAGE + 1; i < n && i < (b + 1) * OR_PAGE; ++i)
      if (scores[i] > m) m = scores[i];
    bs[b].s = m;
    bs[b].i = b;
  }
  qsort(bs, (size_t)nb, sizeof(or_pair_t), cmp_pair);
  const int32_t kept = blocks < nb ? (blocks > 0 ? blocks : 0) : nb;
  /* a mask of the kept blocks, then the candidates in ascending index order */
  uint8_t* keep = (uint8_t*)calloc((size_t)(nb > 0 ? nb : 1), 1);
  for (int32_t j = 0; j < kept; ++j) keep[bs[j].i] = 1;
  float* cand = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  int32_t* cidx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  int32_t m = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (keep[i / OR_PAGE]) { cand[m] = scores[i]; cidx[m] = i; ++m; }
  }
  int32_t sel[OR_TOPK];
  or_topk_row(cand, m, sel);                      /* positions within the candidate list */
  for (int32_t j = 0; j < OR_TOPK; ++j) out512[j] = sel[j] >= 0 ? cidx[sel[j]] : -1;
  free(bs); free(keep); free(cand); free(cidx);
}

/* ======================================================================
 * Sparse MQA attention over the selected entries and the FP8 window.
 * Keys = values = the dequantised 512-d latent (shared by all heads):
 *   global entry: e2m1 * E4M3 block scale;  window token: E4M3 * fp32 scale.
 * For each head: l_j = scale * (q . k_j); m = max l; p_j = exp(l_j - m);
 * Z = sum p; o = (sum_j p_j v_j) / Z; lse = m + log(Z).
 * Key order: global entries ascending, then window positions ascending.
 * [SGL] "Architecture changes..." (top 512 global positions) and [VLLM]
 * "SWA bounded replay" (FP8 window over the most recent 128 positions).
 * ====================================================================== */

static void dequant_main_entry(const or_cache_t* c, int32_t req, int32_t e, float* v512) {
  int32_t page = c->page_table[(int64_t)req * c->max_pages_per_req + e / OR_PAGE];
  const uint8_t* kvp = c->kv_pool + (int64_t)page * OR_KV_PAGE;
  const uint8_t* data = kvp + (e % OR_PAGE) * 256;
  const uint8_t* sc = kvp + OR_KV_SCALE_OFF + (e % OR_PAGE) * 32;
  for (int d = 0; d < OR_D; ++d) v512[d] = or_e2m1_decode(nibble(data, d)) * or_e4m3_decode(sc[d / 16]);
}

/* The rotary reading for attention (no counterpart printed on the pages beyond
 * "Q RoPE merged into the attention-buffer write", [SGL] "DSpark adaptation
 * and optimization"): the same rotate-half as the compressor step above, on
 * the last 64 dims, with table row = position.  The query of a row at
 * position t is rotated with row t; a window token at position p, whose ring
 * slot holds it raw, is rotated with row p before it serves as key and value
 * (keys = values = the latent); the global entries were rotated when they
 * were appended and are used as stored.  rope_cos == NULL: no rotation. */
int or_attention_row_rope(const or_cache_t* c, int32_t req, int32_t pos,
                          const int32_t* topk512, int32_t n_heads, const uint16_t* q_row,
                          float softmax_scale, const float* rope_cos, const float* rope_sin,
                          int32_t rope_rows, float* out, float* lse);

void or_attention_row(const or_cache_t* c, int32_t req, int32_t pos,
                      const int32_t* topk512, int32_t n_heads, const uint16_t* q_row,
                      float softmax_scale, float* out, float* lse) {
  (void)or_attention_row_rope(c, req, pos, topk512, n_heads, q_row, softmax_scale, NULL, NULL, 0, out, lse);
}

int or_attention_row_rope(const or_cache_t* c, int32_t req, int32_t pos,
                          const int32_t* topk512, int32_t n_heads, const uint16_t* q_row,
                          float softmax_scale, const float* rope_cos, const float* rope_sin,
                          int32_t rope_rows, float* out, float* lse) {
  const int rope = rope_cos != NULL && rope_sin != NULL;
  if (rope && (pos < 0 || pos >= rope_rows)) {      /* no table row for this position */
    for (int64_t i = 0; i < (int64_t)n_heads * OR_D; ++i) out[i] = 0.0f;
    if (lse) for (int h = 0; h < n_heads; ++h) lse[h] = -INFINITY;
    return -1;
  }
  int32_t n = row_visible(pos, c->pool_ratio);
  int32_t nk = 0;
  float* keys = (float*)malloc(sizeof(float) * (size_t)(OR_TOPK + OR_WINDOW) * OR_D);
  for (int j = 0; j < OR_TOPK; ++j) {
    int32_t e = topk512[j];
    if (e < 0 || e >= n) continue;
    dequant_main_entry(c, req, e, keys + (int64_t)nk * OR_D);
    ++nk;
  }
  if (c->win_codes != NULL) {
    int32_t lo = pos - (OR_WINDOW - 1) > 0 ? pos - (OR_WINDOW - 1) : 0;
    for (int32_t p = lo; p <= pos; ++p) {
      int64_t slot = (int64_t)req * c->win_cap + p % c->win_cap;
      const uint8_t* codes = c->win_codes + slot * OR_D;
      float s = c->win_scale[slot];
      for (int d = 0; d < OR_D; ++d) keys[(int64_t)nk * OR_D + d] = or_e4m3_decode(codes[d]) * s;
      if (rope)
        or_compress_vec(keys + (int64_t)nk * OR_D, OR_D, NULL, 0.0f, rope_cos + (int64_t)p * 32,
                        rope_sin + (int64_t)p * 32);
      ++nk;
    }
  }
  float* logit = (float*)malloc(sizeof(float) * (size_t)(nk > 0 ? nk : 1));
  float q[OR_D];
  for (int h = 0; h < n_heads; ++h) {
    float* o = out + (int64_t)h * OR_D;
    for (int d = 0; d < OR_D; ++d) q[d] = or_bf16_to_f32(q_row[(int64_t)h * OR_D + d]);
    if (rope) or_compress_vec(q, OR_D, NULL, 0.0f, rope_cos + (int64_t)pos * 32, rope_sin + (int64_t)pos * 32);
    if (nk == 0) {
      for (int d = 0; d < OR_D; ++d) o[d] = 0.0f;
      if (lse) lse[h] = -INFINITY;
      continue;
    }
    float m = -INFINITY;
    for (int32_t j = 0; j < nk; ++j) {
      float dot = 0.0f;
      for (int d = 0; d < OR_D; ++d) dot = dot + q[d] * keys[(int64_t)j * OR_D + d];
      logit[j] = softmax_scale * dot;
      if (logit[j] > m) m = logit[j];
    }
    float Z = 0.0f;
    for (int32_t j = 0; j < nk; ++j) {
      logit[j] = expf(logit[j] - m);            /* p_j, stored in place */
      Z = Z + logit[j];
    }
    for (int d = 0; d < OR_D; ++d) {
      float acc = 0.0f;
      for (int32_t j = 0; j < nk; ++j) acc = acc + logit[j] * keys[(int64_t)j * OR_D + d];
      o[d] = acc / Z;
    }
    if (lse) lse[h] = m + logf(Z);
  }
  free(logit);
  free(keys);
  return 0;
}

/* ======================================================================
 * Whole decode step, rows split over POSIX threads.
 * ====================================================================== */

typedef struct {
  const or_cache_t* c;
  int32_t num_rows, tid, nthreads, Hi, H;
  const int32_t *row_req, *row_pos;
  const uint16_t *q_idx, *q;
  const float* w;
  float softmax_scale;
  float *out, *lse, *scores;
  int32_t* topk;
  int64_t ld;
} or_job_t;

static void* decode_worker(void* arg) {
  or_job_t* j = (or_job_t*)arg;
  int32_t tk[OR_TOPK];
  for (int32_t r = j->tid; r < j->num_rows; r += j->nthreads) {
    float* sc = j->scores + (int64_t)r * j->ld;
    score_one_row(j->c, j->row_req[r], j->row_pos[r], j->Hi,
                  j->q_idx + (int64_t)r * j->Hi * OR_DI, j->w + (int64_t)r * j->Hi, sc);
    or_topk_row(sc, row_visible(j->row_pos[r], j->c->pool_ratio), tk);
    if (j->topk) memcpy(j->topk + (int64_t)r * OR_TOPK, tk, sizeof(tk));
    or_attention_row(j->c, j->row_req[r], j->row_pos[r], tk, j->H,
                     j->q + (int64_t)r * j->H * OR_D, j->softmax_scale,
                     j->out + (int64_t)r * j->H * OR_D, j->lse ? j->lse + (int64_t)r * j->H : NULL);
  }
  return NULL;
}

void or_decode(const or_cache_t* c, int32_t num_rows, const int32_t* row_req,
               const int32_t* row_pos, int32_t n_idx_heads, const uint16_t* q_idx,
               const float* w, int32_t n_heads, const uint16_t* q, float softmax_scale,
               float* out, float* lse, int32_t* topk_out, float* scores_ws, int64_t ld,
               int32_t threads) {
  if (threads < 1) threads = 1;
  or_job_t* jobs = (or_job_t*)calloc((size_t)threads, sizeof(or_job_t));
  pthread_t* tids = (pthread_t*)calloc((size_t)threads, sizeof(pthread_t));
  for (int t = 0; t < threads; ++t) {
    or_job_t j = {c, num_rows, t, threads, n_idx_heads, n_heads, row_req, row_pos,
                  q_idx, q, w, softmax_scale, out, lse, scores_ws, topk_out, ld};
    jobs[t] = j;
  }
  if (threads == 1) {
    decode_worker(&jobs[0]);
  } else {
    for (int t = 0; t < threads; ++t) pthread_create(&tids[t], NULL, decode_worker, &jobs[t]);
    for (int t = 0; t < threads; ++t) pthread_join(tids[t], NULL);
  }
  free(tids);
  free(jobs);
}
