/*
 * CPU oracle for the CSA decode path -- TEST INFRASTRUCTURE ONLY.
 *
 * This header and csa_oracle.c are a plain, slow, scalar restatement of what
 * the decode path computes.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or constant with the CUDA library: every constant below is restated
 * here from the format description, not included from the library.
 *
 * Sources (web pages; cited by title and section):
 *  [SGL]  "DeepSeek-V4.1 Flash on SGLang: from 35 to 873 tokens/s",
 *         sections "Architecture changes and KV cache compression",
 *         "Small-operator fusion and GEMV", "DSpark adaptation and optimization".
 *  [VLLM] "DeepSeek-V4.1-Flash runs 5.3x faster on vLLM after three weeks of
 *         optimization", sections "The architecture behind the jump",
 *         "SWA bounded replay, or how to skip half the model".
 *  [KT]   ktransformers issue "Support for Deepseek V4.1 Flash" (comments on
 *         the SM120 sparse-MLA precision routes and the V4 KV layout).
 *  [OCP]  OCP Microscaling (MX) Formats Specification v1.0 (E2M1, E8M0 and
 *         the MX block-scale rule) and the OCP 8-bit floating point
 *         specification (E4M3 "fn": bias 7, max 448, no infinities).
 *
 * Floating point: fp32 throughout, compiled with -ffp-contract=off and no
 * fast-math, so every add and multiply below rounds exactly once, in the
 * order written.
 *
 * Parity status: every function here is pinned by a CPU test (code tables,
 * RNE tie points, brute-force quantiser search, closed forms, dense attention
 * in fp64, append order invariance); none is "parity unpinned".
 */
#ifndef CSA_ORACLE_H
#define CSA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- element codes ([OCP]) ------------------------------------------- */
float   or_e2m1_decode(uint8_t code);          /* 4-bit code, bit 3 = sign      */
uint8_t or_e2m1_encode(float v);               /* RNE to the grid, saturate ±6  */
float   or_e4m3_decode(uint8_t code);          /* NaN for S.1111.111            */
uint8_t or_e4m3_encode(float v);               /* RNE, saturate to ±448         */
float   or_e8m0_decode(uint8_t code);          /* 2^(code-127); 255 = NaN       */
uint8_t or_e8m0_block_code(float amax);        /* MX rule: floor(log2 amax) - 2 */

/* ---- block quantisers -------------------------------------------------- */
/* NVFP4 block of 16: one E4M3 scale, 16 e2m1 codes (one per byte, unpacked) */
void or_nvfp4_block(const float* x16, uint8_t* codes16, uint8_t* scale);
/* MXFP4 block of 32: one E8M0 scale, 32 e2m1 codes (unpacked)               */
void or_mxfp4_block(const float* x32, uint8_t* codes32, uint8_t* scale);

/* One main-KV entry: 512 values -> 256 packed bytes + 32 E4M3 scales (288 B) */
void or_quant_main_entry(const float* x512, uint8_t* data256, uint8_t* scale32);
/* One indexer-K entry: 128 values -> 64 packed bytes + 4 E8M0 scales (68 B)  */
void or_quant_idx_entry(const float* y128, uint8_t* data64, uint8_t* scale4);
/* One window token: 512 values -> 512 E4M3 codes + fp32 scale amax/448       */
void or_quant_window_token(const float* x512, uint8_t* codes512, float* scale);

/* bf16 bits -> fp32 (exact) */
float or_bf16_to_f32(uint16_t bits);

/* ---- cache description --------------------------------------------------
 * Pools hold num_pages pages.  Main-KV page = 18432 B, indexer page = 4352 B
 * (see csa_oracle.c for the byte layout).  page_table[b*max_pages + j] is the
 * physical page of request b's logical page j; both pools use the same id. */
typedef struct {
  uint8_t*       kv_pool;
  uint8_t*       idx_pool;
  const int32_t* page_table;
  int32_t        num_pages, num_requests, max_pages_per_req, pool_ratio;
  uint8_t*       win_codes;   /* [num_requests, win_cap, 512] or NULL */
  float*         win_scale;   /* [num_requests, win_cap]              */
  int32_t        win_cap;
} or_cache_t;

/* Append new tokens (pool, quantise, write).  Returns 0, or a negative value
 * when a page index is out of range (nothing is written for that entry).
 * pending_in / pending_out: bf16 [num_requests, 640] (512 latent + 128 key). */
int or_append(const or_cache_t* c, const int32_t* pos0, const int32_t* tok_off,
              const uint16_t* kv_in, const uint16_t* idx_in,
              const uint16_t* pending_in, uint16_t* pending_out);

/* The compressor's normalisation and rotary steps, applied to each pooled
 * entry before quantisation ([SGL] "DSpark adaptation and optimization":
 * pair pooling, RMSNorm, RoPE, quantisation and the cache write are one fused
 * step, reused for the indexer key).  Any pointer may be NULL (step skipped).
 * rope_cos / rope_sin: [rope_rows, 32] for the 32 frequency pairs of the last
 * 64 dims of each vector, indexed by the position of the entry's last token. */
typedef struct {
  const float* kv_gamma;    /* [512] */
  const float* idx_gamma;   /* [128] */
  float        eps;
  const float* rope_cos;
  const float* rope_sin;
  int32_t      rope_rows;
} or_compress_t;

/* RMSNorm (sum of squares in the fixed order documented in csa_oracle.c),
 * then rotate-half RoPE on the last 64 dims, in place.  dim: 512 or 128. */
void or_compress_vec(float* v, int dim, const float* gamma, float eps, const float* cos32,
                     const float* sin32);

/* or_append with the compressor steps (cmp may be NULL: plain or_append).
 * Returns -3 when an entry's position is beyond the rotary tables. */
int or_append_compress(const or_cache_t* c, const int32_t* pos0, const int32_t* tok_off,
                       const uint16_t* kv_in, const uint16_t* idx_in,
                       const uint16_t* pending_in, uint16_t* pending_out, const or_compress_t* cmp);

/* Indexer scores for rows: scores[r*ld + i] for i < n(r) = (pos+1)/P. */
void or_index_score(const or_cache_t* c, int32_t num_rows, const int32_t* row_req,
                    const int32_t* row_pos, int32_t n_idx_heads,
                    const uint16_t* q_idx, const float* w, float* scores, int64_t ld);

/* Exact top-512 of scores[0..n): ascending index order, padded with -1. */
void or_topk_row(const float* scores, int32_t n, int32_t* out512);

/* Two-level candidate filter: blocks of 64 entries scored by their largest
 * score, the first `blocks` by (block score desc, block index asc) kept, then
 * the exact top-512 among their entries (ascending, -1 padded). */
void or_topk_two_level(const float* scores, int32_t n, int32_t blocks, int32_t* out512);

/* Sparse MQA attention for one row: keys = the selected global entries
 * (ascending) followed by the window positions max(0,t-127)..t. */
void or_attention_row(const or_cache_t* c, int32_t req, int32_t pos,
                      const int32_t* topk512, int32_t n_heads, const uint16_t* q_row,
                      float softmax_scale, float* out /*[H,512]*/, float* lse /*[H]*/);

/* or_attention_row with the query and the window tokens rotated (rotate-half
 * on the last 64 dims, as or_compress_vec, with rope_cos/rope_sin row = the
 * position: t for the query, p for a window token, which is rotated as key
 * and value alike); global entries are used as stored.  NULL tables: no
 * rotation.  Returns -1 (zero output, lse -inf) when t >= rope_rows. */
int or_attention_row_rope(const or_cache_t* c, int32_t req, int32_t pos,
                          const int32_t* topk512, int32_t n_heads, const uint16_t* q_row,
                          float softmax_scale, const float* rope_cos, const float* rope_sin,
                          int32_t rope_rows, float* out /*[H,512]*/, float* lse /*[H]*/);

/* Whole decode step for all rows (score -> top-512 -> attention), split over
 * `threads` POSIX threads by row.  scores_ws: [num_rows, ld] scratch. */
void or_decode(const or_cache_t* c, int32_t num_rows, const int32_t* row_req,
               const int32_t* row_pos, int32_t n_idx_heads, const uint16_t* q_idx,
               const float* w, int32_t n_heads, const uint16_t* q, float softmax_scale,
               float* out, float* lse, int32_t* topk_out, float* scores_ws, int64_t ld,
               int32_t threads);

#ifdef __cplusplus
}
#endif
#endif
