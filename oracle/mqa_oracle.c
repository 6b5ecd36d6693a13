/*
 * mqa_oracle.c -- plain, slow, fp64 CPU oracle for the incremental decode step of
 * Multi-Query / Grouped-Query Attention (KV-cache append + grouped attention).
 *
 * THIS IS TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the test suite, the package's
 * smoke check and the benchmark's CPU-baseline leg may load it. It shares no code, header,
 * table or helper with the CUDA library: it is written directly from the definitions on the
 * source pages, with no blocking, fusion or reordering beyond what those definitions state.
 *
 * Sources (web pages on MQA/GQA; cited by page title and section):
 *   [GQA-MQA] "分组查询注意力（GQA）与多查询注意力（MQA）深度实战" (ybb.press)
 *       §一  KV_bytes = 2 x num_layers x num_kv_heads x seq_len x head_dim x dtype_bytes
 *       §四  g = num_kv_heads, the h query heads split evenly into g groups
 *       §五  j = i // (h/g);  score_{i,t} = Q_i . K_{j,t} / sqrt(d_h);
 *            alpha_{i,t} = softmax_t(score_{i,t});  O_i = sum_t alpha_{i,t} V_{j,t}
 *       §八  the reference module writes the new token's K/V rows into the cache at the
 *            current position, then attends over every cached row up to and including it
 *   [MQA-CSDN] nanhubrain.csdn.net MQA decoding article, §2.2: the decode step concatenates the
 *            new K/V row onto the cache along the sequence axis, then takes logits of every
 *            query head against the (shared) keys.
 *   [MQA-ENC] "多查詢注意力" (compassingai.com), section "KV Cache 結構與視訊記憶體佔用對比".
 *   [MQA-CSDN] §3.3 and [GQA-MQA] §十 item 12: serving stacks (vLLM PagedAttention) keep the
 *            cache in fixed blocks of 16 tokens found through a per-sequence block table.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - attention covers rows 0 .. L_b-1 of sequence b, where L_b (seq_lens[b]) already counts the
 *     token appended in this step;
 *   - heads of one group are contiguous: query head i uses KV head i / (h/g);
 *   - the caller passes the scale (the pages use 1/sqrt(d_h));
 *   - a length outside 1..n_max is an error: that sequence's output is all zeros and the call
 *     returns ORACLE_ERR_BOUNDS;
 *   - the "scores minus their maximum" form of softmax is the definition written out; the
 *     maximum cancels exactly in exact arithmetic.
 *
 * Storage conventions (chosen to match the library's memory layout so that the same buffers can
 * be handed to both, never to share code):
 *   q        [b][h][d_h]            bf16 bit patterns (uint16_t) or double
 *   k_cache  [b][g][n_max][d_h]     idem
 *   v_cache  [b][g][n_max][d_h]     idem
 *   out      [b][h][d_h]            double
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_INVALID_ARG 1
#define ORACLE_ERR_BOUNDS 4

/* ------------------------------------------------------------------------------------------ */
/* KV-cache size: [GQA-MQA] §一 and §七; [MQA-ENC] KV Cache section.                          */
/* ------------------------------------------------------------------------------------------ */
uint64_t oracle_kv_cache_bytes(uint64_t num_layers, uint64_t num_kv_heads, uint64_t seq_len,
                               uint64_t head_dim, uint64_t dtype_bytes) {
  /* factor 2: one K and one V tensor per layer */
  return 2u * num_layers * num_kv_heads * seq_len * head_dim * dtype_bytes;
}

/* ------------------------------------------------------------------------------------------ */
/* bfloat16 <-> double, written from the bfloat16 bit layout: 1 sign bit, 8 exponent bits     */
/* (bias 127), 7 fraction bits.                                                               */
/* ------------------------------------------------------------------------------------------ */
double oracle_bf16_to_double(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int expo = (bits >> 7) & 0xFF;
  int frac = bits & 0x7F;
  double mag;
  if (expo == 0xFF) {
    mag = frac ? NAN : INFINITY;
  } else if (expo == 0) {
    /* subnormal: frac * 2^(1 - 127 - 7) */
    mag = ldexp((double)frac, -133);
  } else {
    /* normal: (1 + frac/128) * 2^(expo - 127) = (128 + frac) * 2^(expo - 134) */
    mag = ldexp((double)(128 + frac), expo - 134);
  }
  return sign ? -mag : mag;
}

/* Round a double to the nearest bfloat16, ties to even. Returns the bit pattern. */
uint16_t oracle_double_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isinf(a)) return sign | 0x7F80;
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);           /* a = m * 2^e2, m in [0.5, 1)  =>  a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;          /* a in [2^E, 2^(E+1)) */
  /* spacing of the bf16 grid around a: 2^(E-7) for normals, 2^-133 below 2^-126 */
  int spacing_exp = (E < -126) ? -133 : (E - 7);
  double units = ldexp(a, -spacing_exp);   /* exact: scaling by a power of two */
  double r = floor(units);
  double rem = units - r;
  if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  double v = ldexp(r, spacing_exp);
  /* largest finite bf16 is (2 - 2^-7) * 2^127; anything that rounds past it is infinite */
  if (v >= ldexp(1.0, 128)) return sign | 0x7F80;
  if (v < ldexp(1.0, -126)) {
    /* subnormal (or rounded up to the smallest normal, which the same formula encodes) */
    return sign | (uint16_t)ldexp(v, 133);
  }
  int ev;
  frexp(v, &ev);
  int Ev = ev - 1;         /* v in [2^Ev, 2^(Ev+1)) */
  uint16_t frac = (uint16_t)(ldexp(v, 7 - Ev) - 128.0);
  return sign | (uint16_t)((Ev + 127) << 7) | frac;
}

/* ------------------------------------------------------------------------------------------ */
/* fp8 E4M3 (the OCP 8-bit format with 4 exponent bits and no infinities) <-> double, written  */
/* from its bit layout: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits. Exponent field */
/* 15 with fraction 7 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448; exponent    */
/* field 0 holds the subnormals frac/8 * 2^-6. Quantized caches ([GQA-MQA] §十 item 7 and      */
/* [MQA-CSDN] §4.3 on quantizing K/V at low bit widths; the format and scaling are this        */
/* build's reading, see the design notes).                                                    */
/* ------------------------------------------------------------------------------------------ */
double oracle_e4m3_to_double(uint8_t code) {
  int sign = (code >> 7) & 1;
  int expo = (code >> 3) & 0xF;
  int frac = code & 0x7;
  double mag;
  if (expo == 0xF && frac == 0x7) {
    mag = NAN;
  } else if (expo == 0) {
    mag = ldexp((double)frac, -9);                  /* frac/8 * 2^-6 */
  } else {
    mag = ldexp((double)(8 + frac), expo - 7 - 3);  /* (1 + frac/8) * 2^(expo - 7) */
  }
  return sign ? -mag : mag;
}

/* Round a double to the nearest E4M3 value, ties to even; magnitudes beyond 448 saturate to   */
/* +-448 (the largest finite value), NaN gives 0x7F. Returns the code.                         */
uint8_t oracle_double_to_e4m3(double x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);
  int E = e2 - 1;                              /* a in [2^E, 2^(E+1)) */
  int spacing_exp = (E < -6) ? -9 : (E - 3);   /* grid step: 2^-9 below 2^-6, else 2^(E-3) */
  double units = ldexp(a, -spacing_exp);
  double r = floor(units);
  double rem = units - r;
  if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) == 1.0)) r += 1.0;   /* ties to the even code */
  double v = ldexp(r, spacing_exp);
  if (v == 0.0) return sign;
  if (v < ldexp(1.0, -6)) return sign | (uint8_t)r;   /* subnormal: the code is the fraction */
  int ev;
  frexp(v, &ev);
  int Ev = ev - 1;                             /* v in [2^Ev, 2^(Ev+1)), Ev in [-6, 8] */
  uint8_t frac = (uint8_t)(ldexp(v, 3 - Ev) - 8.0);
  return sign | (uint8_t)((Ev + 7) << 3) | frac;
}

/* Quantized append: row pos[b] of every KV head j receives the codes                          */
/*     e4m3( float(k_new[b][j][d]) / k_scale )   (and v_new with v_scale),                     */
/* the division done once in binary32 (IEEE, rounded to nearest), then rounded to E4M3 as      */
/* above. A position outside [0, n_max) skips that sequence and reports ORACLE_ERR_BOUNDS.     */
int oracle_kv_append_fp8(const uint16_t* k_new, const uint16_t* v_new, uint8_t* k_cache,
                         uint8_t* v_cache, const int32_t* pos, int b, int g, int d_h, int n_max,
                         float k_scale, float v_scale) {
  if (!k_new || !v_new || !k_cache || !v_cache || !pos) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || g <= 0 || d_h <= 0 || n_max <= 0) return ORACLE_ERR_INVALID_ARG;
  if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || isinf(k_scale) || isinf(v_scale))
    return ORACLE_ERR_INVALID_ARG;
  int status = ORACLE_OK;
  for (int bi = 0; bi < b; ++bi) {
    const int p = pos[bi];
    if (p < 0 || p >= n_max) { status = ORACLE_ERR_BOUNDS; continue; }
    for (int j = 0; j < g; ++j) {
      const size_t src = ((size_t)bi * g + j) * (size_t)d_h;
      const size_t row = ((size_t)bi * g + j) * (size_t)n_max + (size_t)p;
      const size_t dst = row * (size_t)d_h;
      for (int d = 0; d < d_h; ++d) {
        volatile float kq = (float)oracle_bf16_to_double(k_new[src + d]) / k_scale;
        volatile float vq = (float)oracle_bf16_to_double(v_new[src + d]) / v_scale;
        k_cache[dst + d] = oracle_double_to_e4m3((double)kq);
        v_cache[dst + d] = oracle_double_to_e4m3((double)vq);
      }
    }
  }
  return status;
}

/* Dequantize: out[i] = e4m3(codes[i]) * scale, in double (exact: a 4-bit significand times a  */
/* binary32 scale).                                                                            */
int oracle_dequantize_e4m3(const uint8_t* codes, size_t n, double scale, double* out) {
  if (!codes || !out) return ORACLE_ERR_INVALID_ARG;
  for (size_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_double(codes[i]) * scale;
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* KV append: [GQA-MQA] §八 (cache_k[:, start:start+T] = k with T = 1);                      */
/* [MQA-CSDN] §2.2 (concat along the sequence axis). Bit copy of one row per (b, KV head).    */
/* ------------------------------------------------------------------------------------------ */
int oracle_kv_append(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_cache,
                     uint16_t* v_cache, const int32_t* pos, int b, int g, int d_h, int n_max) {
  if (!k_new || !v_new || !k_cache || !v_cache || !pos) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || g <= 0 || d_h <= 0 || n_max <= 0) return ORACLE_ERR_INVALID_ARG;
  int status = ORACLE_OK;
  for (int bi = 0; bi < b; ++bi) {
    int p = pos[bi];
    if (p < 0 || p >= n_max) { status = ORACLE_ERR_BOUNDS; continue; }
    for (int j = 0; j < g; ++j) {
      size_t src = ((size_t)bi * g + j) * (size_t)d_h;
      size_t dst = (((size_t)bi * g + j) * (size_t)n_max + (size_t)p) * (size_t)d_h;
      memcpy(k_cache + dst, k_new + src, (size_t)d_h * sizeof(uint16_t));
      memcpy(v_cache + dst, v_new + src, (size_t)d_h * sizeof(uint16_t));
    }
  }
  return status;
}

/* ------------------------------------------------------------------------------------------ */
/* Paged cache ([MQA-CSDN] §3.3; [GQA-MQA] §十 item 12). Reading: a pool of pages               */
/* [num_pages][g][page_size][d_h], and for sequence b a table of max_pages page indices; the    */
/* sequence's row t of KV head j is row t % page_size of KV head j in page                      */
/* table[b][t / page_size]. Attention over a paged cache is attention over the rows this map   */
/* gives, so the oracle gathers them into the contiguous layout and attends there.              */
/* ------------------------------------------------------------------------------------------ */
int oracle_gather_pages(const uint16_t* pool, const int32_t* table, int b, int g, int d_h,
                        int page_size, int max_pages, int num_pages, uint16_t* cache) {
  if (!pool || !table || !cache) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || g <= 0 || d_h <= 0 || page_size <= 0 || max_pages <= 0 || num_pages <= 0)
    return ORACLE_ERR_INVALID_ARG;
  const int n_max = max_pages * page_size;
  int status = ORACLE_OK;
  for (int bi = 0; bi < b; ++bi)
    for (int j = 0; j < g; ++j)
      for (int t = 0; t < n_max; ++t) {
        uint16_t* dst = cache + (((size_t)bi * g + j) * (size_t)n_max + (size_t)t) * (size_t)d_h;
        const int page = table[(size_t)bi * max_pages + t / page_size];
        if (page < 0 || page >= num_pages) {
          status = ORACLE_ERR_BOUNDS;
          memset(dst, 0, (size_t)d_h * sizeof(uint16_t));
          continue;
        }
        const uint16_t* src = pool + (((size_t)page * g + j) * (size_t)page_size +
                                      (size_t)(t % page_size)) * (size_t)d_h;
        memcpy(dst, src, (size_t)d_h * sizeof(uint16_t));
      }
  return status;
}

/* The append through the table: row pos[b] of sequence b's KV head j <- k_new[b][j] (and V). */
int oracle_kv_append_paged(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_pool,
                           uint16_t* v_pool, const int32_t* pos, const int32_t* table, int b,
                           int g, int d_h, int page_size, int max_pages, int num_pages) {
  if (!k_new || !v_new || !k_pool || !v_pool || !pos || !table) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || g <= 0 || d_h <= 0 || page_size <= 0 || max_pages <= 0 || num_pages <= 0)
    return ORACLE_ERR_INVALID_ARG;
  int status = ORACLE_OK;
  for (int bi = 0; bi < b; ++bi) {
    const int p = pos[bi];
    if (p < 0 || p >= max_pages * page_size) { status = ORACLE_ERR_BOUNDS; continue; }
    const int page = table[(size_t)bi * max_pages + p / page_size];
    if (page < 0 || page >= num_pages) { status = ORACLE_ERR_BOUNDS; continue; }
    for (int j = 0; j < g; ++j) {
      size_t src = ((size_t)bi * g + j) * (size_t)d_h;
      size_t dst = (((size_t)page * g + j) * (size_t)page_size + (size_t)(p % page_size)) *
                   (size_t)d_h;
      memcpy(k_pool + dst, k_new + src, (size_t)d_h * sizeof(uint16_t));
      memcpy(v_pool + dst, v_new + src, (size_t)d_h * sizeof(uint16_t));
    }
  }
  return status;
}

/* The same gather for a pool of one-byte E4M3 codes (fp8 caches): rows of out-of-range pages   */
/* come back as code 0 (the value 0) and the call reports ORACLE_ERR_BOUNDS.                    */
int oracle_gather_pages_u8(const uint8_t* pool, const int32_t* table, int b, int g, int d_h,
                           int page_size, int max_pages, int num_pages, uint8_t* cache) {
  if (!pool || !table || !cache) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || g <= 0 || d_h <= 0 || page_size <= 0 || max_pages <= 0 || num_pages <= 0)
    return ORACLE_ERR_INVALID_ARG;
  const int n_max = max_pages * page_size;
  int status = ORACLE_OK;
  for (int bi = 0; bi < b; ++bi)
    for (int j = 0; j < g; ++j)
      for (int t = 0; t < n_max; ++t) {
        uint8_t* dst = cache + (((size_t)bi * g + j) * (size_t)n_max + (size_t)t) * (size_t)d_h;
        const int pg = table[(size_t)bi * max_pages + (t / page_size)];
        if (pg < 0 || pg >= num_pages) {
          status = ORACLE_ERR_BOUNDS;
          memset(dst, 0, (size_t)d_h);
          continue;
        }
        const size_t in_page = (size_t)(t % page_size);
        memcpy(dst, pool + (((size_t)pg * g + j) * (size_t)page_size + in_page) * (size_t)d_h,
               (size_t)d_h);
      }
  return status;
}

/* Several tokens through the table ([GQA-MQA] §八 with T new tokens; [MQA-CSDN] §3.3 paging):  */
/* token t of sequence b goes to row pos[b] + t, i.e. row (pos[b] + t) % page_size of KV head j */
/* in page table[b][(pos[b] + t) / page_size]. A sequence whose rows pos .. pos + T - 1 are not */
/* all in [0, max_pages * page_size) is skipped; a row whose page index is out of range is      */
/* skipped alone (the sequence's other rows are written); both report ORACLE_ERR_BOUNDS.       */
int oracle_kv_append_paged_multi(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_pool,
                                 uint16_t* v_pool, const int32_t* pos, const int32_t* table,
                                 int b, int T, int g, int d_h, int page_size, int max_pages,
                                 int num_pages) {
  if (!k_new || !v_new || !k_pool || !v_pool || !pos || !table) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || T <= 0 || g <= 0 || d_h <= 0 || page_size <= 0 || max_pages <= 0 ||
      num_pages <= 0)
    return ORACLE_ERR_INVALID_ARG;
  int status = ORACLE_OK;
  for (int bi = 0; bi < b; ++bi) {
    const int p0 = pos[bi];
    if (p0 < 0 || (long long)p0 + T > (long long)max_pages * page_size) {
      status = ORACLE_ERR_BOUNDS;
      continue;
    }
    for (int t = 0; t < T; ++t) {
      const int p = p0 + t;
      const int page = table[(size_t)bi * max_pages + p / page_size];
      if (page < 0 || page >= num_pages) { status = ORACLE_ERR_BOUNDS; continue; }
      const size_t row_in_page = (size_t)(p % page_size);
      for (int j = 0; j < g; ++j) {
        const size_t src = (((size_t)bi * T + t) * g + j) * (size_t)d_h;
        const size_t dst = (((size_t)page * g + j) * (size_t)page_size + row_in_page) *
                           (size_t)d_h;
        memcpy(k_pool + dst, k_new + src, (size_t)d_h * sizeof(uint16_t));
        memcpy(v_pool + dst, v_new + src, (size_t)d_h * sizeof(uint16_t));
      }
    }
  }
  return status;
}

/* The quantized append through the table: the codes of oracle_kv_append_fp8                   */
/* (e4m3(float(x) / scale), the division once in binary32) at the row oracle_kv_append_paged    */
/* writes. A bad position or page skips the sequence and reports ORACLE_ERR_BOUNDS.             */
int oracle_kv_append_paged_fp8(const uint16_t* k_new, const uint16_t* v_new, uint8_t* k_pool,
                               uint8_t* v_pool, const int32_t* pos, const int32_t* table, int b,
                               int g, int d_h, int page_size, int max_pages, int num_pages,
                               float k_scale, float v_scale) {
  if (!k_new || !v_new || !k_pool || !v_pool || !pos || !table) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || g <= 0 || d_h <= 0 || page_size <= 0 || max_pages <= 0 || num_pages <= 0)
    return ORACLE_ERR_INVALID_ARG;
  if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || isinf(k_scale) || isinf(v_scale))
    return ORACLE_ERR_INVALID_ARG;
  int status = ORACLE_OK;
  for (int bi = 0; bi < b; ++bi) {
    const int p = pos[bi];
    if (p < 0 || p >= max_pages * page_size) { status = ORACLE_ERR_BOUNDS; continue; }
    const int page = table[(size_t)bi * max_pages + p / page_size];
    if (page < 0 || page >= num_pages) { status = ORACLE_ERR_BOUNDS; continue; }
    const size_t prow = (size_t)(p % page_size);
    for (int j = 0; j < g; ++j) {
      const size_t src = ((size_t)bi * g + j) * (size_t)d_h;
      const size_t dst = (((size_t)page * g + j) * (size_t)page_size + prow) * (size_t)d_h;
      for (int d = 0; d < d_h; ++d) {
        const float kx = (float)oracle_bf16_to_double(k_new[src + d]);
        const float vx = (float)oracle_bf16_to_double(v_new[src + d]);
        volatile float kq = kx / k_scale;
        volatile float vq = vx / v_scale;
        k_pool[dst + d] = oracle_double_to_e4m3((double)kq);
        v_pool[dst + d] = oracle_double_to_e4m3((double)vq);
      }
    }
  }
  return status;
}

/* ------------------------------------------------------------------------------------------ */
/* Grouped decode attention: [GQA-MQA] §五.                                                   */
/* ------------------------------------------------------------------------------------------ */
enum { KIND_BF16 = 0, KIND_F64 = 1 };

static inline double load_elem(const void* base, size_t idx, int kind) {
  if (kind == KIND_F64) return ((const double*)base)[idx];
  return oracle_bf16_to_double(((const uint16_t*)base)[idx]);
}

/* Softmax-weighted sum over rows t in [t_begin, t_end) for one (sequence, query head).
 * Writes m = max score, l = sum_t exp(score_t - m), o[d] = sum_t exp(score_t - m) V[t][d].
 * An empty range gives m = -inf, l = 0, o = 0. */
static void attend_range(const void* q, const void* k_cache, const void* v_cache, int kind,
                         int bi, int i, int h, int g, int d_h, int n_max, double scale,
                         int t_begin, int t_end, double* scores, double* m_out, double* l_out,
                         double* o_out) {
  int group_size = h / g;
  int j = i / group_size;                      /* §五: j = i // (h/g) */
  size_t q_off = ((size_t)bi * h + i) * (size_t)d_h;
  size_t kv_off = ((size_t)bi * g + j) * (size_t)n_max * (size_t)d_h;

  for (int d = 0; d < d_h; ++d) o_out[d] = 0.0;
  if (t_end <= t_begin) { *m_out = -INFINITY; *l_out = 0.0; return; }

  /* score_{i,t} = scale * sum_d Q_i[d] K_{j,t}[d] */
  double m = -INFINITY;
  for (int t = t_begin; t < t_end; ++t) {
    double s = 0.0;
    for (int d = 0; d < d_h; ++d)
      s += load_elem(q, q_off + d, kind) * load_elem(k_cache, kv_off + (size_t)t * d_h + d, kind);
    s *= scale;
    scores[t - t_begin] = s;
    if (s > m) m = s;
  }
  /* weights exp(s - m), their sum, and the weighted sum of value rows */
  double l = 0.0;
  for (int t = t_begin; t < t_end; ++t) {
    double w = exp(scores[t - t_begin] - m);
    l += w;
    for (int d = 0; d < d_h; ++d)
      o_out[d] += w * load_elem(v_cache, kv_off + (size_t)t * d_h + d, kind);
  }
  *m_out = m;
  *l_out = l;
}

static int check_attention_args(const void* q, const void* k, const void* v, const int32_t* lens,
                                 const double* out, int b, int h, int g, int d_h, int n_max) {
  if (!q || !k || !v || !lens || !out) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || h <= 0 || g <= 0 || d_h <= 0 || n_max <= 0) return ORACLE_ERR_INVALID_ARG;
  if (h % g != 0) return ORACLE_ERR_INVALID_ARG;  /* §十 item 1: heads split evenly */
  return ORACLE_OK;
}

static int attention_full(const void* q, const void* k_cache, const void* v_cache, int kind,
                          const int32_t* seq_lens, double* out, int b, int h, int g, int d_h,
                          int n_max, double scale, int threads) {
  int st = check_attention_args(q, k_cache, v_cache, seq_lens, out, b, h, g, d_h, n_max);
  if (st) return st;
  int bad = 0;
  for (int bi = 0; bi < b; ++bi)
    if (seq_lens[bi] < 1 || seq_lens[bi] > n_max) bad = 1;
#ifdef _OPENMP
  if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel num_threads(threads)
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)n_max);
    double* acc = (double*)malloc(sizeof(double) * (size_t)d_h);
#ifdef _OPENMP
#pragma omp for collapse(2) schedule(dynamic, 1)
#endif
    for (int bi = 0; bi < b; ++bi) {
      for (int i = 0; i < h; ++i) {
        double* o = out + ((size_t)bi * h + i) * (size_t)d_h;
        int L = seq_lens[bi];
        if (L < 1 || L > n_max) {
          for (int d = 0; d < d_h; ++d) o[d] = 0.0;
          continue;
        }
        double m, l;
        attend_range(q, k_cache, v_cache, kind, bi, i, h, g, d_h, n_max, scale, 0, L, scores,
                     &m, &l, acc);
        /* O_i = sum_t alpha_{i,t} V_{j,t},  alpha = exp(s - m) / l */
        for (int d = 0; d < d_h; ++d) o[d] = acc[d] / l;
      }
    }
    free(scores);
    free(acc);
  }
  return bad ? ORACLE_ERR_BOUNDS : ORACLE_OK;
}

int oracle_decode_attention_bf16(const uint16_t* q, const uint16_t* k_cache,
                                 const uint16_t* v_cache, const int32_t* seq_lens, double* out,
                                 int b, int h, int g, int d_h, int n_max, double scale,
                                 int threads) {
  return attention_full(q, k_cache, v_cache, KIND_BF16, seq_lens, out, b, h, g, d_h, n_max,
                        scale, threads);
}

int oracle_decode_attention_f64(const double* q, const double* k_cache, const double* v_cache,
                                const int32_t* seq_lens, double* out, int b, int h, int g,
                                int d_h, int n_max, double scale, int threads) {
  return attention_full(q, k_cache, v_cache, KIND_F64, seq_lens, out, b, h, g, d_h, n_max,
                        scale, threads);
}

/* ------------------------------------------------------------------------------------------ */
/* Several new tokens per sequence ([GQA-MQA] §八: forward(x, start) appends T rows at          */
/* start .. start+T-1 and attends over the first start+T rows; §十 item 10: the causal mask     */
/* still applies per query position when K/V are shared). Query token t of sequence b sits at  */
/* row L_b - T + t, where L_b = seq_lens[b] counts all T new rows, and attends rows             */
/* 0 .. L_b - T + t: the first L_b - T + 1 + t rows.                                           */
/* q and out are [b][T][h][d_h]; k_new, v_new [b][T][g][d_h].                                  */
/* ------------------------------------------------------------------------------------------ */
int oracle_kv_append_multi(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_cache,
                           uint16_t* v_cache, const int32_t* pos, int b, int T, int g, int d_h,
                           int n_max) {
  if (!k_new || !v_new || !k_cache || !v_cache || !pos) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || T <= 0 || g <= 0 || d_h <= 0 || n_max <= 0) return ORACLE_ERR_INVALID_ARG;
  int status = ORACLE_OK;
  for (int bi = 0; bi < b; ++bi) {
    const int p0 = pos[bi];
    if (p0 < 0 || (long long)p0 + T > n_max) { status = ORACLE_ERR_BOUNDS; continue; }
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < g; ++j) {
        const size_t src = (((size_t)bi * T + t) * g + j) * (size_t)d_h;
        const size_t row = ((size_t)bi * g + j) * (size_t)n_max + (size_t)(p0 + t);
        memcpy(k_cache + row * (size_t)d_h, k_new + src, (size_t)d_h * sizeof(uint16_t));
        memcpy(v_cache + row * (size_t)d_h, v_new + src, (size_t)d_h * sizeof(uint16_t));
      }
  }
  return status;
}

int oracle_decode_attention_multi_bf16(const uint16_t* q, const uint16_t* k_cache,
                                       const uint16_t* v_cache, const int32_t* seq_lens,
                                       double* out, int b, int T, int h, int g, int d_h,
                                       int n_max, double scale, int threads) {
  if (!q || !k_cache || !v_cache || !seq_lens || !out) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || T <= 0 || h <= 0 || g <= 0 || d_h <= 0 || n_max <= 0 || h % g)
    return ORACLE_ERR_INVALID_ARG;
  int bad = 0;
  for (int bi = 0; bi < b; ++bi)
    if (seq_lens[bi] < T || seq_lens[bi] > n_max) bad = 1;
#ifdef _OPENMP
  if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel num_threads(threads)
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)n_max);
    double* qf = (double*)malloc(sizeof(double) * (size_t)d_h);
#ifdef _OPENMP
#pragma omp for collapse(3) schedule(dynamic, 1)
#endif
    for (int bi = 0; bi < b; ++bi) {
      for (int tq = 0; tq < T; ++tq) {
        for (int i = 0; i < h; ++i) {
          const size_t row_off = (((size_t)bi * T + tq) * h + i) * (size_t)d_h;
          double* o = out + row_off;
          for (int d = 0; d < d_h; ++d) o[d] = 0.0;
          const int Lb = seq_lens[bi];
          if (Lb < T || Lb > n_max) continue;
          const int visible = Lb - T + 1 + tq;             /* causal: rows 0 .. Lb - T + tq */
          const int j = i / (h / g);                       /* §五: j = i // (h/g) */
          const size_t kv_off = ((size_t)bi * g + j) * (size_t)n_max * (size_t)d_h;
          for (int d = 0; d < d_h; ++d) qf[d] = oracle_bf16_to_double(q[row_off + d]);
          double m = -INFINITY;
          for (int t = 0; t < visible; ++t) {
            double s = 0.0;
            for (int d = 0; d < d_h; ++d)
              s += qf[d] * oracle_bf16_to_double(k_cache[kv_off + (size_t)t * d_h + d]);
            scores[t] = scale * s;
            if (scores[t] > m) m = scores[t];
          }
          double l = 0.0;
          for (int t = 0; t < visible; ++t) {
            const double w = exp(scores[t] - m);
            l += w;
            for (int d = 0; d < d_h; ++d)
              o[d] += w * oracle_bf16_to_double(v_cache[kv_off + (size_t)t * d_h + d]);
          }
          for (int d = 0; d < d_h; ++d) o[d] /= l;
        }
      }
    }
    free(scores);
    free(qf);
  }
  return bad ? ORACLE_ERR_BOUNDS : ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Split-sequence partials and their log-sum-exp merge. The pages do not describe splitting;  */
/* this is the identity  softmax over a union of ranges = exp-weighted combination of the     */
/* per-range softmax states, used to check that splitting a sequence changes nothing.         */
/* ------------------------------------------------------------------------------------------ */
int oracle_attention_partial_f64(const double* q, const double* k_cache, const double* v_cache,
                                 int b, int h, int g, int d_h, int n_max, double scale,
                                 int t_begin, int t_end, double* m_out, double* l_out,
                                 double* o_out) {
  if (!q || !k_cache || !v_cache || !m_out || !l_out || !o_out) return ORACLE_ERR_INVALID_ARG;
  if (b <= 0 || h <= 0 || g <= 0 || d_h <= 0 || n_max <= 0 || h % g) return ORACLE_ERR_INVALID_ARG;
  if (t_begin < 0 || t_end > n_max) return ORACLE_ERR_BOUNDS;
  double* scores = (double*)malloc(sizeof(double) * (size_t)n_max);
  for (int bi = 0; bi < b; ++bi)
    for (int i = 0; i < h; ++i) {
      size_t r = (size_t)bi * h + i;
      attend_range(q, k_cache, v_cache, KIND_F64, bi, i, h, g, d_h, n_max, scale, t_begin, t_end,
                   scores, &m_out[r], &l_out[r], &o_out[r * (size_t)d_h]);
    }
  free(scores);
  return ORACLE_OK;
}

/* Merge S partial states (m_s, l_s, o_s[d]) of one row:
 *   M = max_s m_s,  out[d] = sum_s exp(m_s - M) o_s[d] / sum_s exp(m_s - M) l_s.
 * Empty partials (m = -inf) carry zero weight. */
int oracle_lse_merge(const double* m, const double* l, const double* o, int S, int d_h,
                     double* out) {
  if (!m || !l || !o || !out || S <= 0 || d_h <= 0) return ORACLE_ERR_INVALID_ARG;
  double M = -INFINITY;
  for (int s = 0; s < S; ++s)
    if (m[s] > M) M = m[s];
  for (int d = 0; d < d_h; ++d) out[d] = 0.0;
  if (M == -INFINITY) return ORACLE_ERR_BOUNDS;   /* every range empty: no softmax exists */
  double denom = 0.0;
  for (int s = 0; s < S; ++s) {
    if (m[s] == -INFINITY) continue;
    double w = exp(m[s] - M);
    denom += w * l[s];
    for (int d = 0; d < d_h; ++d) out[d] += w * o[(size_t)s * d_h + d];
  }
  for (int d = 0; d < d_h; ++d) out[d] /= denom;
  return ORACLE_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
