/*
 * pkv_oracle.c — fp64 CPU oracle of the PagedAttention decode path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do. It shares no code, header, table or helper with the CUDA path.
 *
 * What it follows (page title, then section):
 *   [VM]  "PagedAttention: the KV cache was the bottleneck all along",
 *         "Virtual memory for attention": fixed-size blocks of K/V for a fixed
 *         number of tokens; a per-sequence block table maps logical block
 *         positions to physical blocks; attention reads K/V from the scattered
 *         blocks; shared blocks are copied only when a sharer diverges.
 *   [ABS] "Efficient Memory Management for Large Language Model Serving with
 *         PagedAttention", "From the abstract": PagedAttention computes
 *         attention (paging changes where K/V live, not what is computed).
 *
 * The attention result is therefore the plain definition of scaled
 * dot-product attention of one query over the sequence's earlier tokens,
 * evaluated in double precision after decoding each stored element exactly
 * from its bit pattern. Paging only decides where token t of a sequence is
 * read from; this oracle walks the block table one token at a time.
 *
 * Build: plain C99, -ffp-contract=off so that x86 and Arm round identically.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* ---- element decoding, from the storage formats' definitions ------------ */

/* IEEE 754 binary16: sign(1) exponent(5, bias 15) fraction(10). */
double orc_decode_f16(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1f;
  int f = bits & 0x3ff;
  double mag;
  if (e == 0)
    mag = ldexp((double)f, -24); /* subnormal: f * 2^(1-15-10) */
  else if (e == 31)
    mag = f ? NAN : INFINITY;
  else
    mag = ldexp((double)(f + 1024), e - 25); /* (1.f) * 2^(e-15), as an integer times 2^-10 */
  return sign ? -mag : mag;
}

/* bfloat16: sign(1) exponent(8, bias 127) fraction(7). */
double orc_decode_bf16(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 7) & 0xff;
  int f = bits & 0x7f;
  double mag;
  if (e == 0)
    mag = ldexp((double)f, -133); /* subnormal: f * 2^(1-127-7) */
  else if (e == 255)
    mag = f ? NAN : INFINITY;
  else
    mag = ldexp((double)(f + 128), e - 134); /* (1.f) * 2^(e-127) */
  return sign ? -mag : mag;
}

/* IEEE 754 binary32: sign(1) exponent(8, bias 127) fraction(23). */
double orc_decode_f32(uint32_t bits) {
  int sign = (int)((bits >> 31) & 1u);
  int e = (int)((bits >> 23) & 0xffu);
  uint32_t f = bits & 0x7fffffu;
  double mag;
  if (e == 0)
    mag = ldexp((double)f, -149); /* subnormal: f * 2^(1-127-23) */
  else if (e == 255)
    mag = f ? NAN : INFINITY;
  else
    mag = ldexp((double)(f + 0x800000u), e - 150);
  return sign ? -mag : mag;
}

static int elem_bytes(int dtype) {
  return dtype == ORC_F32 ? 4 : (dtype == ORC_F16 || dtype == ORC_BF16) ? 2 : 0;
}

/* Element `idx` of an array of `dtype`, as a double. */
static double elem(const void* base, size_t idx, int dtype) {
  if (dtype == ORC_F32) {
    uint32_t u;
    memcpy(&u, (const unsigned char*)base + idx * 4, 4);
    return orc_decode_f32(u);
  }
  uint16_t h;
  memcpy(&h, (const unsigned char*)base + idx * 2, 2);
  return dtype == ORC_F16 ? orc_decode_f16(h) : orc_decode_bf16(h);
}

/* ---- softmax-weighted sum over an explicit list of tokens --------------- */

/* Given logits x[0..n) and a way to read V row t, write
 *   out[d] = sum_t exp(x_t - m) * V_t[d] / sum_t exp(x_t - m),  m = max_t x_t
 * (subtracting m is an exact identity of softmax that keeps exp finite).
 * x is scratch: it is overwritten with the weights exp(x_t - m). */
typedef struct {
  const void* v;     /* value storage */
  const size_t* row; /* element offset of token t's row */
  int dtype;
} vrows;

static void softmax_combine(double* out, double* x, int n, vrows V, int head_dim) {
  double m = -INFINITY, z = 0.0;
  for (int t = 0; t < n; ++t)
    if (x[t] > m) m = x[t];
  for (int t = 0; t < n; ++t) {
    x[t] = exp(x[t] - m);
    z += x[t];
  }
  for (int d = 0; d < head_dim; ++d) {
    double acc = 0.0;
    for (int t = 0; t < n; ++t) acc += x[t] * elem(V.v, V.row[t] + (size_t)d, V.dtype);
    out[d] = acc / z;
  }
}

static double dot_rows(const void* a, size_t a_off, const void* b, size_t b_off, int n, int dtype) {
  double acc = 0.0;
  for (int d = 0; d < n; ++d) acc += elem(a, a_off + (size_t)d, dtype) * elem(b, b_off + (size_t)d, dtype);
  return acc;
}

/* ---- paged decode attention ------------------------------------------- */

/*
 * out[s][h][d] (double) for s in [seq_begin, seq_end), every head h.
 * Cache layout [num_blocks][num_kv_heads][block_size][head_dim]; token t of
 * sequence s lives in physical block block_tables[s][t / block_size], row
 * t % block_size ([VM]: block table = logical-to-physical map). Query head h
 * reads kv head h / (num_heads / num_kv_heads).
 * Returns 0, or a negative code for a bad argument / out-of-range block id.
 */
int orc_paged_attention(double* out, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                        int head_dim, int block_size, int num_blocks, int dtype, double scale,
                        int seq_begin, int seq_end) {
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return -1;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return -2;
  if (head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || !elem_bytes(dtype)) return -3;
  if (seq_begin < 0 || seq_end > num_seqs || seq_begin > seq_end) return -4;
  const int group = num_heads / num_kv_heads;
  int max_len = 0;
  for (int s = seq_begin; s < seq_end; ++s) {
    if (context_lens[s] < 0 || context_lens[s] > max_blocks_per_seq * block_size) return -5;
    if (context_lens[s] > max_len) max_len = context_lens[s];
  }
  double* x = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
  size_t* row = (size_t*)malloc(sizeof(size_t) * (size_t)(max_len > 0 ? max_len : 1));
  if (!x || !row) {
    free(x);
    free(row);
    return -6;
  }
  int rc = 0;
  for (int s = seq_begin; s < seq_end && rc == 0; ++s) {
    const int L = context_lens[s];
    for (int h = 0; h < num_heads; ++h) {
      const int g = h / group;
      double* o = out + ((size_t)s * num_heads + h) * head_dim;
      if (L == 0) {
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        continue;
      }
      const size_t q_off = ((size_t)s * num_heads + h) * head_dim;
      for (int t = 0; t < L; ++t) {
        const int32_t p = block_tables[(size_t)s * max_blocks_per_seq + t / block_size];
        if (p < 0 || p >= num_blocks) {
          rc = -7;
          break;
        }
        row[t] = (((size_t)p * num_kv_heads + g) * block_size + (size_t)(t % block_size)) * head_dim;
        x[t] = scale * dot_rows(q, q_off, k_cache, row[t], head_dim, dtype);
      }
      if (rc) break;
      vrows V = {v_cache, row, dtype};
      softmax_combine(o, x, L, V, head_dim);
    }
  }
  free(x);
  free(row);
  return rc;
}

/*
 * Same attention over K/V stored densely, sequence after sequence:
 * k, v are [total_tokens][num_kv_heads][head_dim]; sequence s owns rows
 * [seq_start[s], seq_start[s+1]). No block table is involved. Used to pin the
 * paged oracle: paging must not change the result.
 */
int orc_dense_attention(double* out, const void* q, const void* k, const void* v,
                        const int64_t* seq_start, int num_seqs, int num_heads, int num_kv_heads,
                        int head_dim, int dtype, double scale) {
  if (!out || !q || !k || !v || !seq_start) return -1;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return -2;
  if (head_dim <= 0 || !elem_bytes(dtype)) return -3;
  const int group = num_heads / num_kv_heads;
  int64_t max_len = 0;
  for (int s = 0; s < num_seqs; ++s) {
    int64_t n = seq_start[s + 1] - seq_start[s];
    if (n < 0) return -5;
    if (n > max_len) max_len = n;
  }
  double* x = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
  size_t* row = (size_t*)malloc(sizeof(size_t) * (size_t)(max_len > 0 ? max_len : 1));
  if (!x || !row) {
    free(x);
    free(row);
    return -6;
  }
  for (int s = 0; s < num_seqs; ++s) {
    const int L = (int)(seq_start[s + 1] - seq_start[s]);
    for (int h = 0; h < num_heads; ++h) {
      const int g = h / group;
      double* o = out + ((size_t)s * num_heads + h) * head_dim;
      if (L == 0) {
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        continue;
      }
      const size_t q_off = ((size_t)s * num_heads + h) * head_dim;
      for (int t = 0; t < L; ++t) {
        row[t] = (((size_t)seq_start[s] + (size_t)t) * num_kv_heads + g) * head_dim;
        x[t] = scale * dot_rows(q, q_off, k, row[t], head_dim, dtype);
      }
      vrows V = {v, row, dtype};
      softmax_combine(o, x, L, V, head_dim);
    }
  }
  free(x);
  free(row);
  return 0;
}

/*
 * Split-context form of the same attention: the context of each (s, h) is cut
 * into consecutive chunks of `chunk` tokens. Chunk c keeps its own maximum
 * m_c, exp-sum l_c = sum_{t in c} exp(x_t - m_c) and normalised output
 * o_c = sum_{t in c} exp(x_t - m_c) V_t / l_c. The chunks are then combined:
 *   M = max_c m_c,  w_c = l_c * exp(m_c - M),  out = sum_c w_c o_c / sum_c w_c.
 * Algebraically equal to the single pass (both are the same softmax); used to
 * pin that combination rule. Paged layout as in orc_paged_attention.
 */
int orc_paged_attention_chunked(double* out, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                int num_heads, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, int dtype, double scale, int chunk) {
  if (chunk <= 0) return -8;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return -1;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return -2;
  if (head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || !elem_bytes(dtype)) return -3;
  const int group = num_heads / num_kv_heads;
  int max_len = 0;
  for (int s = 0; s < num_seqs; ++s) {
    if (context_lens[s] < 0 || context_lens[s] > max_blocks_per_seq * block_size) return -5;
    if (context_lens[s] > max_len) max_len = context_lens[s];
  }
  const int max_chunks = max_len > 0 ? (max_len + chunk - 1) / chunk : 1;
  double* x = (double*)malloc(sizeof(double) * (size_t)chunk);
  size_t* row = (size_t*)malloc(sizeof(size_t) * (size_t)chunk);
  double* cm = (double*)malloc(sizeof(double) * (size_t)max_chunks);               /* m_c */
  double* cl = (double*)malloc(sizeof(double) * (size_t)max_chunks);               /* l_c */
  double* co = (double*)malloc(sizeof(double) * (size_t)max_chunks * head_dim);    /* o_c */
  if (!x || !row || !cm || !cl || !co) {
    free(x);
    free(row);
    free(cm);
    free(cl);
    free(co);
    return -6;
  }
  int rc = 0;
  for (int s = 0; s < num_seqs && rc == 0; ++s) {
    const int L = context_lens[s];
    const int nchunks = (L + chunk - 1) / chunk;
    for (int h = 0; h < num_heads && rc == 0; ++h) {
      const int g = h / group;
      double* o = out + ((size_t)s * num_heads + h) * head_dim;
      const size_t q_off = ((size_t)s * num_heads + h) * head_dim;
      /* each chunk on its own: (m_c, l_c, o_c) */
      for (int c = 0; c < nchunks && rc == 0; ++c) {
        const int t0 = c * chunk;
        const int n = (L - t0) < chunk ? (L - t0) : chunk;
        double mc = -INFINITY, lc = 0.0;
        for (int i = 0; i < n; ++i) {
          const int t = t0 + i;
          const int32_t p = block_tables[(size_t)s * max_blocks_per_seq + t / block_size];
          if (p < 0 || p >= num_blocks) {
            rc = -7;
            break;
          }
          row[i] = (((size_t)p * num_kv_heads + g) * block_size + (size_t)(t % block_size)) * head_dim;
          x[i] = scale * dot_rows(q, q_off, k_cache, row[i], head_dim, dtype);
          if (x[i] > mc) mc = x[i];
        }
        if (rc) break;
        for (int i = 0; i < n; ++i) lc += exp(x[i] - mc);
        vrows V = {v_cache, row, dtype};
        softmax_combine(co + (size_t)c * head_dim, x, n, V, head_dim);
        cm[c] = mc;
        cl[c] = lc;
      }
      if (rc) break;
      if (L == 0) {
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        continue;
      }
      /* merge: M = max_c m_c, w_c = l_c exp(m_c - M), out = sum w_c o_c / sum w_c */
      double M = -INFINITY, wsum = 0.0;
      for (int c = 0; c < nchunks; ++c)
        if (cm[c] > M) M = cm[c];
      for (int c = 0; c < nchunks; ++c) wsum += cl[c] * exp(cm[c] - M);
      for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (int c = 0; c < nchunks; ++c) acc += cl[c] * exp(cm[c] - M) * co[(size_t)c * head_dim + d];
        o[d] = acc / wsum;
      }
    }
  }
  free(x);
  free(row);
  free(cm);
  free(cl);
  free(co);
  return rc;
}

/* ---- cache maintenance (byte copies) ------------------------------------ */

/*
 * [VM] a sequence grows one token per step into its blocks: for token t with
 * slot s = slot_mapping[t] >= 0, every kv head's K row and V row is copied to
 * cache[s / block_size][h][s % block_size][:]. Negative slots are padding and
 * are skipped. Returns the number of slots that were out of range (not
 * written), or a negative code for a bad argument.
 */
int orc_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                          const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                          int head_dim, int block_size, int num_blocks, int dtype) {
  const int es = elem_bytes(dtype);
  if (!es || num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return -1;
  if (num_tokens && (!k || !v || !k_cache || !v_cache || !slot_mapping)) return -1;
  const size_t row_bytes = (size_t)head_dim * es;
  int bad = 0;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= (int64_t)num_blocks * block_size) {
      ++bad;
      continue;
    }
    const int64_t blk = slot / block_size, off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + (size_t)off) * row_bytes;
      const size_t src = ((size_t)t * num_kv_heads + h) * row_bytes;
      memcpy((unsigned char*)k_cache + dst, (const unsigned char*)k + src, row_bytes);
      memcpy((unsigned char*)v_cache + dst, (const unsigned char*)v + src, row_bytes);
    }
  }
  return bad;
}

/*
 * [VM] copy-on-write: for each pair (src, dst) the whole physical block src
 * (every kv head, every row) of both pools is copied onto block dst, in pair
 * order. Returns the number of pairs skipped for out-of-range ids, or a
 * negative code for a bad argument.
 */
int orc_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_pairs, int num_pairs,
                    int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype) {
  const int es = elem_bytes(dtype);
  if (!es || num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return -1;
  if (num_pairs && (!k_cache || !v_cache || !block_pairs)) return -1;
  const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * es;
  int bad = 0;
  for (int i = 0; i < num_pairs; ++i) {
    const int64_t src = block_pairs[2 * i], dst = block_pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      ++bad;
      continue;
    }
    memmove((unsigned char*)k_cache + (size_t)dst * block_bytes,
            (const unsigned char*)k_cache + (size_t)src * block_bytes, block_bytes);
    memmove((unsigned char*)v_cache + (size_t)dst * block_bytes,
            (const unsigned char*)v_cache + (size_t)src * block_bytes, block_bytes);
  }
  return bad;
}

/* ---- fp8 (e4m3) KV cache ------------------------------------------------ */
/*
 * [QKV] "Efficient Memory Management for Large Language Model Serving with
 * PagedAttention" (hackerpapers page), "In the conversation": quantising the
 * KV cache cuts its memory footprint. Format (the reading this oracle takes):
 * OCP E4M3 codes, sign(1) exponent(4, bias 7) mantissa(3), no infinities,
 * S.1111.111 is NaN, largest finite 448; one scale per pool; element x is
 * stored as e4m3(binary32(x / scale)) and read back as scale * code.
 */

/* E4M3 code -> value. */
double orc_decode_e4m3(uint8_t bits) {
  int sign = (bits >> 7) & 1;
  int e = (bits >> 3) & 0xf;
  int m = bits & 0x7;
  double mag;
  if (e == 0)
    mag = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
  else if (e == 15 && m == 7)
    mag = NAN;
  else
    mag = ldexp((double)(m + 8), e - 10); /* (1 + m/8) * 2^(e-7) */
  return sign ? -mag : mag;
}

/* value -> nearest E4M3 code, ties to the even code, finite values beyond
 * the largest (and infinities) saturated to +-448, NaN to 0x7f. The grid is
 * uniform with spacing 2^-9 below 2^-6 (subnormals) and 2^(E-3) in
 * [2^E, 2^(E+1)); codes count up along it, so a rounded grid index that
 * carries into the next binade is still the right code. */
uint8_t orc_encode_e4m3(double x) {
  if (isnan(x)) return 0x7f;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs(x);
  if (a > 448.0) return sign | 0x7e;
  int code;
  if (a < ldexp(1.0, -6)) {
    code = (int)rint(a * 512.0); /* multiples of 2^-9; 8 is the smallest normal */
  } else {
    int k;
    frexp(a, &k); /* a = f * 2^k, f in [0.5, 1) */
    const int E = k - 1;
    const int n = (int)rint(ldexp(a, 3 - E)); /* in [8, 16] */
    code = (E + 7) * 8 + (n - 8);
  }
  if (code > 0x7e) code = 0x7e;
  return (uint8_t)(sign | code);
}

/*
 * Cache write into e4m3 pools ([QKV], [VM]): for token t with slot s >= 0,
 * every element x of its K (V) rows becomes orc_encode_e4m3 of the binary32
 * quotient (float)x / k_scale (v_scale), stored at cache[s / bs][h][s % bs].
 * k, v are binary16 or bfloat16 (src_dtype). Returns the number of
 * out-of-range slots (not written), or a negative code.
 */
int orc_reshape_and_cache_fp8(const void* k, const void* v, uint8_t* k_cache, uint8_t* v_cache,
                              const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                              int block_size, int num_blocks, int src_dtype, float k_scale, float v_scale) {
  if ((src_dtype != ORC_F16 && src_dtype != ORC_BF16) || num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || num_blocks <= 0 || !(k_scale > 0.0f) || !(v_scale > 0.0f))
    return -1;
  if (num_tokens && (!k || !v || !k_cache || !v_cache || !slot_mapping)) return -1;
  int bad = 0;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= (int64_t)num_blocks * block_size) {
      ++bad;
      continue;
    }
    const int64_t blk = slot / block_size, off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h)
      for (int d = 0; d < head_dim; ++d) {
        const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + (size_t)off) * head_dim + d;
        const size_t src = ((size_t)t * num_kv_heads + h) * head_dim + d;
        const float kq = (float)elem(k, src, src_dtype) / k_scale; /* binary32 division */
        const float vq = (float)elem(v, src, src_dtype) / v_scale;
        k_cache[dst] = orc_encode_e4m3((double)kq);
        v_cache[dst] = orc_encode_e4m3((double)vq);
      }
  }
  return bad;
}

/*
 * Paged decode attention over e4m3 pools ([QKV], [VM]): the definition of
 * orc_paged_attention with K element = k_scale * decode(code) and V element =
 * v_scale * decode(code); q in q_dtype. out[s][h][:] for s in
 * [seq_begin, seq_end). Returns 0 or a negative code.
 */
int orc_paged_attention_fp8(double* out, const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                            int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                            int num_blocks, int q_dtype, double scale, double k_scale, double v_scale,
                            int seq_begin, int seq_end) {
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return -1;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return -2;
  if (head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || !elem_bytes(q_dtype)) return -3;
  if (seq_begin < 0 || seq_end > num_seqs || seq_begin > seq_end) return -4;
  const int group = num_heads / num_kv_heads;
  int max_len = 0;
  for (int s = seq_begin; s < seq_end; ++s) {
    if (context_lens[s] < 0 || context_lens[s] > max_blocks_per_seq * block_size) return -5;
    if (context_lens[s] > max_len) max_len = context_lens[s];
  }
  double* x = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
  size_t* row = (size_t*)malloc(sizeof(size_t) * (size_t)(max_len > 0 ? max_len : 1));
  if (!x || !row) {
    free(x);
    free(row);
    return -6;
  }
  int rc = 0;
  for (int s = seq_begin; s < seq_end && rc == 0; ++s) {
    const int L = context_lens[s];
    for (int h = 0; h < num_heads; ++h) {
      const int g = h / group;
      double* o = out + ((size_t)s * num_heads + h) * head_dim;
      if (L == 0) {
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        continue;
      }
      const size_t q_off = ((size_t)s * num_heads + h) * head_dim;
      for (int t = 0; t < L; ++t) {
        const int32_t p = block_tables[(size_t)s * max_blocks_per_seq + t / block_size];
        if (p < 0 || p >= num_blocks) {
          rc = -7;
          break;
        }
        row[t] = (((size_t)p * num_kv_heads + g) * block_size + (size_t)(t % block_size)) * head_dim;
        double acc = 0.0;
        for (int d = 0; d < head_dim; ++d)
          acc += elem(q, q_off + (size_t)d, q_dtype) * (k_scale * orc_decode_e4m3(k_cache[row[t] + (size_t)d]));
        x[t] = scale * acc;
      }
      if (rc) break;
      double m = -INFINITY, z = 0.0;
      for (int t = 0; t < L; ++t)
        if (x[t] > m) m = x[t];
      for (int t = 0; t < L; ++t) {
        x[t] = exp(x[t] - m);
        z += x[t];
      }
      for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (int t = 0; t < L; ++t) acc += x[t] * (v_scale * orc_decode_e4m3(v_cache[row[t] + (size_t)d]));
        o[d] = acc / z;
      }
    }
  }
  free(x);
  free(row);
  return rc;
}

/* ---- paged prefill (multi-token causal queries) -------------------------- */
/*
 * [WL] "PagedAttention: the KV cache was the bottleneck all along", section
 * "What is left": the wish for shared blocks for common system prompts
 * across users, i.e. the prompt side over the same paged cache; [VM] for the
 * paging. Reading taken: sequence s holds context_lens[s] = L tokens in the
 * cache (its new tokens already written); its n = query_start[s+1] -
 * query_start[s] queries are its last n tokens, and query i (at position
 * L - n + i) attends to tokens 0 .. L - n + i (causal). q and out are packed
 * [total_queries][num_heads][head_dim]. Returns 0 or a negative code.
 */
int orc_paged_prefill(double* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                      const int32_t* query_start, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, int dtype, double scale, int seq_begin, int seq_end) {
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start) return -1;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return -2;
  if (head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || !elem_bytes(dtype)) return -3;
  if (seq_begin < 0 || seq_end > num_seqs || seq_begin > seq_end) return -4;
  const int group = num_heads / num_kv_heads;
  int max_len = 0;
  for (int s = seq_begin; s < seq_end; ++s) {
    const int L = context_lens[s], n = query_start[s + 1] - query_start[s];
    if (L < 0 || L > max_blocks_per_seq * block_size || n < 0 || n > L) return -5;
    if (L > max_len) max_len = L;
  }
  double* x = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
  size_t* row = (size_t*)malloc(sizeof(size_t) * (size_t)(max_len > 0 ? max_len : 1));
  if (!x || !row) {
    free(x);
    free(row);
    return -6;
  }
  int rc = 0;
  for (int s = seq_begin; s < seq_end && rc == 0; ++s) {
    const int L = context_lens[s], n = query_start[s + 1] - query_start[s];
    for (int t = 0; t < L; ++t) {
      const int32_t p = block_tables[(size_t)s * max_blocks_per_seq + t / block_size];
      if (p < 0 || p >= num_blocks) {
        rc = -7;
        break;
      }
    }
    if (rc) break;
    for (int i = 0; i < n; ++i) {
      const int pos = L - n + i; /* this query's own position */
      const size_t qi = (size_t)query_start[s] + (size_t)i;
      for (int h = 0; h < num_heads; ++h) {
        const int g = h / group;
        double* o = out + (qi * num_heads + h) * head_dim;
        const size_t q_off = (qi * num_heads + h) * head_dim;
        for (int t = 0; t <= pos; ++t) {
          const int32_t p = block_tables[(size_t)s * max_blocks_per_seq + t / block_size];
          row[t] = (((size_t)p * num_kv_heads + g) * block_size + (size_t)(t % block_size)) * head_dim;
          x[t] = scale * dot_rows(q, q_off, k_cache, row[t], head_dim, dtype);
        }
        vrows V = {v_cache, row, dtype};
        softmax_combine(o, x, pos + 1, V, head_dim);
      }
    }
  }
  free(x);
  free(row);
  return rc;
}

/* ---- 4-bit (q4_0) KV cache ---------------------------------------------- */
/*
 * [QKV] "Efficient Memory Management for Large Language Model Serving with
 * PagedAttention" (hackerpapers page), "In the conversation": a reader notes
 * that 4-bit KV-cache quantisation, the cache type called q4_0, cuts the
 * cache to about a quarter of its size. The pages name the format without
 * defining it. Reading taken: the q4_0 block of the ggml tensor library,
 * where 32 consecutive values share one binary16 scale d and each keeps a
 * 4-bit code q in 0..15 that reads back as d * (q - 8). Quantising a block
 * x[0..31], every step in binary32:
 *   m   = the element of largest magnitude, sign kept (the first on ties;
 *         +0 when every |x| is 0 or NaN)
 *   d   = m / -8                    (m itself gets code 0)
 *   inv = 1 / d, or 0 when d is 0
 *   y   = x_j * inv + 8.5           (a product and a sum, each rounded)
 *   q_j = 15 if y >= 15, else trunc(y) if y >= 0, else 0 (NaN included)
 * Stored: d rounded to binary16 (nearest, ties to even, overflow to
 * infinity); code byte j (0..15) of the block holds q_j in its low and
 * q_(j+16) in its high four bits. A cache row of D values holds D/32
 * blocks: the D/32 scales first (little-endian binary16), then the blocks'
 * 16 code bytes in block order, 9 D / 16 bytes in all (this library's
 * arrangement of the blocks in a row).
 */

/* double -> nearest binary16 bits (ties to even), from the format's
 * definition: subnormals are multiples of 2^-24; in [2^E, 2^(E+1)) the
 * spacing is 2^(E-10); values at or above 65520 overflow to infinity. */
uint16_t orc_encode_f16(double x) {
  if (isnan(x)) return 0x7e00;
  const uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
  const double a = fabs(x);
  int code;
  if (a < ldexp(1.0, -14)) {
    code = (int)rint(ldexp(a, 24)); /* 1024 is the smallest normal: the carry is right */
  } else if (a >= 65520.0) {
    code = 0x7c00;
  } else {
    int k;
    frexp(a, &k); /* a = f * 2^k, f in [0.5, 1) */
    const int E = k - 1;
    const int n = (int)rint(ldexp(a, 10 - E)); /* in [1024, 2048] */
    code = (E + 15) * 1024 + (n - 1024);
  }
  if (code > 0x7c00) code = 0x7c00;
  return (uint16_t)(sign | code);
}

/* One block of 32 binary32 values -> scale bits and 16 code bytes. */
void orc_q4_0_quantize_block(const float* x, uint16_t* d_bits, uint8_t* qs) {
  float amax = 0.0f, m = 0.0f;
  for (int j = 0; j < 32; ++j) {
    const float a = fabsf(x[j]);
    if (a > amax) {
      amax = a;
      m = x[j];
    }
  }
  const float d = m / -8.0f;
  const float inv = d != 0.0f ? 1.0f / d : 0.0f;
  int q[32];
  for (int j = 0; j < 32; ++j) {
    const float prod = x[j] * inv;
    const float y = prod + 8.5f;
    q[j] = y >= 15.0f ? 15 : (y >= 0.0f ? (int)y : 0);
  }
  *d_bits = orc_encode_f16((double)d);
  for (int j = 0; j < 16; ++j) qs[j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

/* Value of element d (0 .. head_dim-1) of a q4_0 row. */
double orc_q4_0_value(const uint8_t* row, int head_dim, int d) {
  const int b = d / 32, j = d % 32;
  const uint16_t sb = (uint16_t)(row[2 * b] | (row[2 * b + 1] << 8));
  const uint8_t byte = row[head_dim / 16 + 16 * b + (j % 16)];
  const int q = j < 16 ? (byte & 0xf) : (byte >> 4);
  return (double)(q - 8) * orc_decode_f16(sb);
}

/* One row of head_dim values of src_dtype (binary16 or bfloat16, converted
 * exactly to binary32) -> 9 head_dim / 16 bytes. */
int orc_q4_0_quantize_row(const void* src, int src_dtype, int head_dim, uint8_t* row) {
  if ((src_dtype != ORC_F16 && src_dtype != ORC_BF16) || head_dim <= 0 || head_dim % 32) return -1;
  for (int b = 0; b < head_dim / 32; ++b) {
    float x[32];
    for (int j = 0; j < 32; ++j) x[j] = (float)elem(src, (size_t)(32 * b + j), src_dtype);
    uint16_t sb;
    orc_q4_0_quantize_block(x, &sb, row + head_dim / 16 + 16 * b);
    row[2 * b] = (uint8_t)(sb & 0xff);
    row[2 * b + 1] = (uint8_t)(sb >> 8);
  }
  return 0;
}

/*
 * Cache write into q4_0 pools ([QKV], [VM]): for token t with slot s >= 0,
 * each kv head's K (V) row is quantised as above into cache row
 * [s / bs][h][s % bs] of the [num_blocks][num_kv_heads][block_size]
 * [9 head_dim / 16] byte pools. Returns the number of out-of-range slots
 * (not written), or a negative code.
 */
int orc_reshape_and_cache_q4_0(const void* k, const void* v, uint8_t* k_cache, uint8_t* v_cache,
                               const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, int src_dtype) {
  if ((src_dtype != ORC_F16 && src_dtype != ORC_BF16) || num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % 32 || block_size <= 0 || num_blocks <= 0)
    return -1;
  if (num_tokens && (!k || !v || !k_cache || !v_cache || !slot_mapping)) return -1;
  const size_t rb = (size_t)head_dim / 16 * 9;
  int bad = 0;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= (int64_t)num_blocks * block_size) {
      ++bad;
      continue;
    }
    const int64_t blk = slot / block_size, off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + (size_t)off) * rb;
      const size_t src = ((size_t)t * num_kv_heads + h) * head_dim * 2;
      orc_q4_0_quantize_row((const unsigned char*)k + src, src_dtype, head_dim, k_cache + dst);
      orc_q4_0_quantize_row((const unsigned char*)v + src, src_dtype, head_dim, v_cache + dst);
    }
  }
  return bad;
}

/*
 * Paged decode attention over q4_0 pools ([QKV], [VM]): the definition of
 * orc_paged_attention with every K and V element read back as d * (q - 8)
 * from its row; q in q_dtype. out[s][h][:] for s in [seq_begin, seq_end).
 * Returns 0 or a negative code.
 */
int orc_paged_attention_q4_0(double* out, const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                             const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                             int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                             int num_blocks, int q_dtype, double scale, int seq_begin, int seq_end) {
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return -1;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return -2;
  if (head_dim <= 0 || head_dim % 32 || block_size <= 0 || num_blocks <= 0 || !elem_bytes(q_dtype)) return -3;
  if (seq_begin < 0 || seq_end > num_seqs || seq_begin > seq_end) return -4;
  const int group = num_heads / num_kv_heads;
  const size_t rb = (size_t)head_dim / 16 * 9;
  int max_len = 0;
  for (int s = seq_begin; s < seq_end; ++s) {
    if (context_lens[s] < 0 || context_lens[s] > max_blocks_per_seq * block_size) return -5;
    if (context_lens[s] > max_len) max_len = context_lens[s];
  }
  double* x = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
  size_t* row = (size_t*)malloc(sizeof(size_t) * (size_t)(max_len > 0 ? max_len : 1));
  if (!x || !row) {
    free(x);
    free(row);
    return -6;
  }
  int rc = 0;
  for (int s = seq_begin; s < seq_end && rc == 0; ++s) {
    const int L = context_lens[s];
    for (int h = 0; h < num_heads; ++h) {
      const int g = h / group;
      double* o = out + ((size_t)s * num_heads + h) * head_dim;
      if (L == 0) {
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        continue;
      }
      const size_t q_off = ((size_t)s * num_heads + h) * head_dim;
      for (int t = 0; t < L; ++t) {
        const int32_t p = block_tables[(size_t)s * max_blocks_per_seq + t / block_size];
        if (p < 0 || p >= num_blocks) {
          rc = -7;
          break;
        }
        row[t] = (((size_t)p * num_kv_heads + g) * block_size + (size_t)(t % block_size)) * rb;
        double acc = 0.0;
        for (int d = 0; d < head_dim; ++d)
          acc += elem(q, q_off + (size_t)d, q_dtype) * orc_q4_0_value(k_cache + row[t], head_dim, d);
        x[t] = scale * acc;
      }
      if (rc) break;
      double m = -INFINITY, z = 0.0;
      for (int t = 0; t < L; ++t)
        if (x[t] > m) m = x[t];
      for (int t = 0; t < L; ++t) {
        x[t] = exp(x[t] - m);
        z += x[t];
      }
      for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (int t = 0; t < L; ++t) acc += x[t] * orc_q4_0_value(v_cache + row[t], head_dim, d);
        o[d] = acc / z;
      }
    }
  }
  free(x);
  free(row);
  return rc;
}
