// Paged decode attention for sequences that share prefix blocks (sm_103a).
//
// Operation ("PagedAttention: the KV cache was the bottleneck all along",
// section "Virtual memory for attention"): sampled completions of one prompt
// (or beams) map the prompt's blocks to the same physical blocks, so their
// attention reads the same K/V rows for the prefix. The result per sequence
// is exactly the plain decode attention; the grouping only lets each shared
// K/V tile be read once for all siblings.
//
// Work: the same persistent, balanced streaming as the plain kernel, over two
// kinds of segments laid end to end:
//   prefix segments (group g, head h, row group c): K/V rows [0, S_g) of the
//     group's shared blocks against the query rows of up to kGroupRows
//     siblings (head h of members 4c .. 4c+3);
//   tail segments (sequence s, head group hg): rows [S_g, L_s) of s's own
//     blocks against its query heads, as in the plain kernel.
// The prefix segments run first, balanced over all warps, then the tails,
// balanced again, as two launches in stream order. A tail row of a sequence
// with a shared prefix merges its prefix result (log-sum-exp) when it writes
// the output. Pieces of a segment cut by warp range boundaries are
// merged as in the plain kernel.
//
// A prologue kernel checks the caller's grouping: group_start must partition
// [0, num_seqs) and the first shared_blocks[g] block-table entries of every
// member must be equal. The usable prefix S_g is the checked shared length
// cut to whole tiles and whole blocks and to the shortest member's context.
// A grouping that fails the check sets PKV_DEV_ERR_GROUP and is ignored (the
// kernel then computes the plain result), so a wrong promise never gives a
// wrong answer silently.
#pragma once

#include "decode.cuh"

namespace pkv {

constexpr int kGroupRows = 4;  // query rows one warp serves against one K/V tile

// The work split charges every segment a fixed cost, in tile units, on top of
// its tiles: entering a segment (metadata, query rows) and finishing it
// (reductions, the prefix merge, the output row) take about as long as
// streaming that many tiles. A warp whose range holds many short tails then
// gets fewer tiles. The charged units hold no tile: a cursor skips them.
constexpr int kSegCostPrefix = 1;
constexpr int kSegCostTail = 2;

struct GroupedParams {
  DecodeParams base;             // ws_counter is unused here
  const int32_t* group_start;    // [num_groups + 1]
  const int32_t* shared_blocks;  // [num_groups]
  int num_groups;
  int32_t* ws_flag;     // [1] 1 = grouping rejected
  int32_t* ws_sync;     // [2] reserved (unused)
  int32_t* ws_group_S;  // [num_groups] usable shared prefix tokens
  int32_t* ws_seq_P;    // [num_seqs] prefix tokens of the sequence's group
  int32_t* ws_seg_ctr;  // [2][num_seqs * num_heads] piece counters (prefix, tail)
  float2* ws_row_ml;    // [num_seqs * num_heads] (m, l) of each row's prefix result
  float* ws_row_o;      // [num_seqs * num_heads][head_dim] o / l of each row's prefix result
};

__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFullMask, v, o));
  return v;
}

// One warp per group: validation of the grouping and the usable prefix.
// (A template only so that every element-type unit owns its own copy.)
template <typename T>
__global__ void __launch_bounds__(256) pa_group_prologue_kernel(const GroupedParams gp) {
  const DecodeParams& p = gp.base;
  const int B = p.num_seqs, G = gp.num_groups, bs = p.block_size, MB = p.max_blocks_per_seq;
  const int cap = min(p.max_context_len, MB * bs);
  if (blockIdx.x == 0) {
    int bad = 0;
    for (int i = threadIdx.x; i <= G; i += blockDim.x) {
      const int a = __ldg(gp.group_start + i);
      if (a < 0 || a > B || (i == 0 && a != 0) || (i == G && a != B)) bad = 1;
      if (i < G && __ldg(gp.group_start + i + 1) < a) bad = 1;
    }
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
      *gp.ws_flag = bad;
      if (bad) set_err(p.dev_err, PKV_DEV_ERR_GROUP);
    }
  }
  const int lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int unit = bs > kTileTokens ? bs : kTileTokens;  // whole tiles and whole blocks
  for (int g = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; g < G; g += nwarps) {
    int lo = __ldg(gp.group_start + g), hi = __ldg(gp.group_start + g + 1);
    lo = max(0, min(lo, B));
    hi = max(lo, min(hi, B));
    int S = 0;
    if (hi - lo >= 2) {
      int sb = max(0, min(__ldg(gp.shared_blocks + g), MB));
      int minL = cap;
      for (int s = lo + lane; s < hi; s += 32) minL = min(minL, load_len(p, s, cap));
      minL = warp_min(minL);
      const int32_t* row0 = p.block_tables + (size_t)lo * MB;
      int first_bad = sb;
      // every (member, entry) pair is an independent comparison: the lanes
      // take them all at once, so the loads are in flight together
      const int pairs = (hi - lo - 1) * sb;
#pragma unroll 4
      for (int i = lane; i < pairs; i += 32) {
        const int m = i / sb, j = i - m * sb;
        if (__ldg(p.block_tables + (size_t)(lo + 1 + m) * MB + j) != __ldg(row0 + j)) first_bad = min(first_bad, j);
      }
      first_bad = warp_min(first_bad);
      if (first_bad < sb) {
        if (lane == 0) set_err(p.dev_err, PKV_DEV_ERR_GROUP);
        sb = first_bad;
      }
      S = min(sb * bs, minL) / unit * unit;
    }
    if (lane == 0) gp.ws_group_S[g] = S;
    for (int s = lo + lane; s < hi; s += 32) gp.ws_seq_P[s] = S;
  }
}

// Position in the global tile sequence of the grouped kernel, with the
// metadata of the current segment.
struct GCursor {
  long long g;  // global tile index
  int part;     // 0 prefix segment, 1 tail segment
  int a;        // group (part 0) or sequence (part 1)
  int b;        // head (part 0) or head group (part 1)
  int c;        // row group (part 0)
  int t, nt;
  int lo, M;            // part 0: members [lo, lo + M)
  int tok0, tok_end;    // token range of the K/V source
  int sbt;              // block-table row of the K/V source
  int sbt_len;          // context length of that row (bounds the entries read from it)
  int kvh, nrows;
};

// Everything the cursors need, by value (no pointer to the kernel parameters).
struct GCtx {
  const int32_t* group_start;
  const int32_t* group_S;
  const int32_t* seq_P;
  const int32_t* context_lens;
  int32_t* dev_err;
  int num_groups, num_seqs, num_heads, head_groups, group, cap, gpw;
  bool use_groups;
};

__device__ __forceinline__ int ctx_len(const GCtx& x, int s) {
  int L = __ldg(x.context_lens + s);
  if (L < 0 || L > x.cap) {
    if (blockIdx.x == 0) set_err(x.dev_err, PKV_DEV_ERR_CONTEXT_LEN);
    L = L < 0 ? 0 : x.cap;
  }
  return L;
}

__device__ __forceinline__ int group_rows(int M) { return (M + kGroupRows - 1) / kGroupRows; }

// Work units of group g's prefix segments: tiles plus the per-segment cost
// (0 when the group has no usable shared prefix).
__device__ __forceinline__ long long prefix_units(const GCtx& x, int g) {
  if (!x.use_groups) return 0;
  const int M = __ldg(x.group_start + g + 1) - __ldg(x.group_start + g);
  const int S = x.group_S[g];
  if (M < 2 || S <= 0) return 0;
  return (long long)x.num_heads * group_rows(M) * (S / kTileTokens + kSegCostPrefix);
}

__device__ __forceinline__ int seq_prefix(const GCtx& x, int s) { return x.use_groups ? x.seq_P[s] : 0; }

__device__ __forceinline__ void gseg_enter(GCursor& c, const GCtx& x) {
  if (c.part == 0) {
    c.lo = __ldg(x.group_start + c.a);
    c.M = __ldg(x.group_start + c.a + 1) - c.lo;
    c.tok0 = 0;
    c.tok_end = x.group_S[c.a];
    c.sbt = c.lo;
    c.sbt_len = ctx_len(x, c.lo);
    c.kvh = c.b / x.group;
    c.nrows = min(kGroupRows, c.M - kGroupRows * c.c);
    c.nt = c.tok_end / kTileTokens;
  } else {
    const int L = ctx_len(x, c.a);
    c.tok0 = seq_prefix(x, c.a);
    c.tok_end = L;
    c.sbt = c.a;
    c.sbt_len = L;
    c.kvh = (c.b * x.gpw) / x.group;
    c.nrows = x.gpw;
    c.nt = tiles_of(L - c.tok0);
  }
}

// Move to the first group at or after c.a with prefix tiles; else to the tails.
__device__ __forceinline__ void gseek_prefix(GCursor& c, const GCtx& x) {
  while (c.a < x.num_groups && prefix_units(x, c.a) == 0) ++c.a;
  if (c.a < x.num_groups) {
    c.part = 0;
  } else {
    c.part = 1;
    c.a = 0;
  }
  c.b = 0;
  c.c = 0;
  c.t = 0;
  if (c.part == 0 || c.a < x.num_seqs) gseg_enter(c, x);
}

// Next segment (c.t is 0).
__device__ __forceinline__ void gseg_next(GCursor& c, const GCtx& x) {
  if (c.part == 0) {
    if (++c.c < group_rows(c.M)) {
      gseg_enter(c, x);
      return;
    }
    c.c = 0;
    if (++c.b < x.num_heads) {
      gseg_enter(c, x);
      return;
    }
    ++c.a;
    gseek_prefix(c, x);
    return;
  }
  if (++c.b < x.head_groups) {
    gseg_enter(c, x);
    return;
  }
  c.b = 0;
  if (++c.a < x.num_seqs) gseg_enter(c, x);
}

// Next tile: c.g is its work unit (the next segment's charged units skipped).
__device__ __forceinline__ void gcursor_next(GCursor& c, const GCtx& x) {
  ++c.g;
  if (++c.t < c.nt) return;
  c.t = 0;
  gseg_next(c, x);
  c.g += c.part == 0 ? kSegCostPrefix : kSegCostTail;
}

// (sequence, head) of row r of the segment under c.
__device__ __forceinline__ int row_seq(const GCursor& c, int r) { return c.part == 0 ? c.lo + kGroupRows * c.c + r : c.a; }
__device__ __forceinline__ int row_head(const GCursor& c, const GCtx& x, int r) {
  return c.part == 0 ? c.b : c.b * x.gpw + r;
}

// ---- tensor-core q.k for prefix tiles ---------------------------------------
// m16n8k16 MMA with fp32 accumulation. Only query rows 0..7 are used, so the
// A registers of rows 8..15 are zero. a_lo / a_hi hold row g's k-positions
// 2t, 2t+1 and 2t+8, 2t+9; b_lo / b_hi the same k-positions of column g.
template <typename T>
struct Mma16816 {
  static constexpr bool kOk = false;
  __device__ __forceinline__ static void run(float (&)[4], uint32_t, uint32_t, uint32_t, uint32_t) {}
  __device__ __forceinline__ static void run2(float&, float&, uint32_t, uint32_t, uint32_t, uint32_t) {}
  __device__ __forceinline__ static uint32_t pack(float, float) { return 0u; }
  __device__ __forceinline__ static float2 unpack(uint32_t) { return make_float2(0.f, 0.f); }
};
template <>
struct Mma16816<__nv_bfloat16> {
  static constexpr bool kOk = true;
  __device__ __forceinline__ static void run(float (&d)[4], uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                             uint32_t b_hi) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a_lo), "r"(0u), "r"(a_hi), "r"(0u), "r"(b_lo), "r"(b_hi));
  }
  // rows 0..7 only: accumulators of rows 8..15 are discarded
  __device__ __forceinline__ static void run2(float& c0, float& c1, uint32_t a_lo, uint32_t a_hi,
                                              uint32_t b_lo, uint32_t b_hi) {
    [[maybe_unused]] float d2, d3;
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(c0), "=f"(c1), "=f"(d2), "=f"(d3)
        : "r"(a_lo), "r"(0u), "r"(a_hi), "r"(0u), "r"(b_lo), "r"(b_hi), "f"(c0), "f"(c1), "f"(0.f), "f"(0.f));
  }
  __device__ __forceinline__ static uint32_t pack(float x, float y) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
  }
  __device__ __forceinline__ static float2 unpack(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  }
};
template <>
struct Mma16816<__half> {
  static constexpr bool kOk = true;
  __device__ __forceinline__ static void run(float (&d)[4], uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                             uint32_t b_hi) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a_lo), "r"(0u), "r"(a_hi), "r"(0u), "r"(b_lo), "r"(b_hi));
  }
  __device__ __forceinline__ static void run2(float& c0, float& c1, uint32_t a_lo, uint32_t a_hi,
                                              uint32_t b_lo, uint32_t b_hi) {
    [[maybe_unused]] float d2, d3;
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(c0), "=f"(c1), "=f"(d2), "=f"(d3)
        : "r"(a_lo), "r"(0u), "r"(a_hi), "r"(0u), "r"(b_lo), "r"(b_hi), "f"(c0), "f"(c1), "f"(0.f), "f"(0.f));
  }
  __device__ __forceinline__ static uint32_t pack(float x, float y) {
    const __half2 h = __floats2half2_rn(x, y);
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
  }
  __device__ __forceinline__ static float2 unpack(uint32_t u) {
    __half2 h;
    memcpy(&h, &u, 4);
    return __half22float2(h);
  }
};

// Transpose an 8x8 matrix of 16-bit elements held one 32-bit register per
// lane (lane 4r + c holds row r, columns 2c and 2c+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// q.k is a sum over head dims, so any permutation of the dims applied to both
// operands leaves it unchanged. Within each 32-dim chunk, lane t of an MMA
// group feeds dims [8t, 8t+4) to k-step 0 and [8t+4, 8t+8) to k-step 1, so
// its K operand for both k-steps of a chunk is one 16-byte shared-memory load
// of one token row. The query operand uses the same mapping.

// One 16-token tile of a prefix segment, entirely on tensor cores. The query
// rows (rows < nr of the MMA's M = 16; only rows 0..7 are ever used) are the
// siblings' queries against one K/V tile.
//   S = Q K^T: K operand from token rows, head dims permuted as above.
//   Online softmax on the S accumulators: lane 4r + t holds row r, tokens
//   2t, 2t+1, 2t+8, 2t+9, so a row's max and sum reduce over its 4 lanes.
//   O += P V: the S accumulators are already P's A-operand layout (k =
//   tokens). P is fed as a hi + lo pair of 16-bit values (two MMAs) so that
//   it keeps ~16 significant bits; V's B operand comes from one 16-byte load
//   per lane per 32-dim chunk and 16-token half, cut into four 8x8 blocks
//   over a permutation of the head dims and transposed with movmatrix.
//   Lane 4r + t ends up with row r, dims [32c + 8t, 32c + 8t + 8) of chunk c
//   in po[c][0..3][0..1].
template <typename T, int D>
__device__ __forceinline__ void mma_prefix_tile(const unsigned char* ks, const unsigned char* vs,
                                                const uint32_t (&qa)[D / 32][2][2], float (&po)[D / 32][4][2],
                                                float& pm, float& pl, int nvalid, float scale_log2) {
  constexpr int ROW = D * (int)sizeof(T);
  const int lane = threadIdx.x & 31;
  const int mg = lane >> 2, mt = lane & 3;
  // two independent accumulator chains per 8-token half (first and second
  // k-step of each chunk), added at the end: half the dependent MMA latency
  float s[2][2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) s[nt][h][0] = s[nt][h][1] = 0.f;
#pragma unroll
  for (int c = 0; c < D / 32; ++c)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint4 kk = *reinterpret_cast<const uint4*>(ks + (mg + 8 * nt) * ROW + c * 64 + mt * 16);
      Mma16816<T>::run2(s[nt][0][0], s[nt][0][1], qa[c][0][0], qa[c][0][1], kk.x, kk.y);
      Mma16816<T>::run2(s[nt][1][0], s[nt][1][1], qa[c][1][0], qa[c][1][1], kk.z, kk.w);
    }
  float xs[4], tmax = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) xs[nt * 2 + e] = (s[nt][0][e] + s[nt][1][e]) * scale_log2;
  if (nvalid < kTileTokens) {  // warp-uniform: only a segment's last tile can be partial
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if ((i >> 1) * 8 + 2 * mt + (i & 1) >= nvalid) xs[i] = -INFINITY;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) tmax = fmaxf(tmax, xs[i]);
  tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, 1));
  tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, 2));
  const float mn = fmaxf(pm, tmax);
  const float alpha = exp2f(pm - mn);  // 0 on the segment's first tile (pm = -inf)
  float pe[4], psum = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    pe[i] = exp2f(xs[i] - mn);
    psum += pe[i];
  }
  psum += __shfl_xor_sync(kFullMask, psum, 1);
  psum += __shfl_xor_sync(kFullMask, psum, 2);
  pl = pl * alpha + psum;
  pm = mn;
#pragma unroll
  for (int c = 0; c < D / 32; ++c)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      po[c][q][0] *= alpha;
      po[c][q][1] *= alpha;
    }
  // P (k = tokens 2t, 2t+1 | 2t+8, 2t+9) as hi + lo 16-bit pairs
  const uint32_t hi0 = Mma16816<T>::pack(pe[0], pe[1]);
  const uint32_t hi1 = Mma16816<T>::pack(pe[2], pe[3]);
  const float2 h0 = Mma16816<T>::unpack(hi0), h1 = Mma16816<T>::unpack(hi1);
  const uint32_t lo0 = Mma16816<T>::pack(pe[0] - h0.x, pe[1] - h0.y);
  const uint32_t lo1 = Mma16816<T>::pack(pe[2] - h1.x, pe[3] - h1.y);
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint4 v0 = *reinterpret_cast<const uint4*>(vs + mg * ROW + c * 64 + mt * 16);        // token mg
    uint4 v1 = *reinterpret_cast<const uint4*>(vs + (mg + 8) * ROW + c * 64 + mt * 16);  // token mg + 8
    if (nvalid < kTileTokens) {  // rows past the context may hold poison
      if (mg >= nvalid) v0 = make_uint4(0u, 0u, 0u, 0u);
      if (mg + 8 >= nvalid) v1 = make_uint4(0u, 0u, 0u, 0u);
    }
    const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
    const uint32_t w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t b_lo = movmatrix_trans(w0[q]);
      const uint32_t b_hi = movmatrix_trans(w1[q]);
      Mma16816<T>::run2(po[c][q][0], po[c][q][1], hi0, hi1, b_lo, b_hi);
      Mma16816<T>::run2(po[c][q][0], po[c][q][1], lo0, lo1, b_lo, b_hi);
    }
  }
}

// One 16-token tile on CUDA cores for NR query rows against one K/V tile
// (rows >= nr skipped when PRED): the same math as the plain kernel.
template <typename T, int D, int QR, int NR, bool PRED, int ORows>
__device__ __forceinline__ void core_tile(const unsigned char* ks, const unsigned char* vs,
                                          const float (&qf)[QR][D / 8], float (&o)[ORows][D / 8],
                                          float (&m)[ORows], float (&l)[ORows], int nvalid, int nr) {
  constexpr int ROW = D * (int)sizeof(T);
  constexpr int VEC = Chunk<T>::kElems;
  constexpr int CPL = ROW / 16 / 8;
  const int lane = threadIdx.x & 31;
  const int grp = lane >> 3, sub = lane & 7;
  float x4[NR][4];
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 4 + grp;
    const uint4* krow = reinterpret_cast<const uint4*>(ks + r * ROW);
    float acc[NR];
#pragma unroll
    for (int g = 0; g < NR; ++g) acc[g] = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      float f[VEC];
      Chunk<T>::widen(krow[sub + 8 * k], f);
#pragma unroll
      for (int g = 0; g < NR; ++g)
        if (!PRED || g < nr) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[g] = fmaf(qf[g][k * VEC + e], f[e], acc[g]);
        }
    }
#pragma unroll
    for (int g = 0; g < NR; ++g)
      if (!PRED || g < nr) {
        float a = acc[g];
        a += __shfl_xor_sync(kFullMask, a, 1);
        a += __shfl_xor_sync(kFullMask, a, 2);
        a += __shfl_xor_sync(kFullMask, a, 4);
        x4[g][it] = r < nvalid ? a : -INFINITY;
      }
  }
  float pw[NR][4];
#pragma unroll
  for (int g = 0; g < NR; ++g)
    if (!PRED || g < nr) {
      float mt = fmaxf(fmaxf(x4[g][0], x4[g][1]), fmaxf(x4[g][2], x4[g][3]));
      mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 8));
      mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 16));
      const float mn = fmaxf(m[g], mt);
      const float alpha = exp2f(m[g] - mn);
      float ps = 0.f;
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        pw[g][it] = exp2f(x4[g][it] - mn);
        ps += pw[g][it];
      }
      l[g] = l[g] * alpha + ps;
#pragma unroll
      for (int e = 0; e < D / 8; ++e) o[g][e] *= alpha;
      m[g] = mn;
    }
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 4 + grp;
    if (r < nvalid) {
      const uint4* vrow = reinterpret_cast<const uint4*>(vs + r * ROW);
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        float f[VEC];
        Chunk<T>::widen(vrow[sub + 8 * k], f);
#pragma unroll
        for (int g = 0; g < NR; ++g)
          if (!PRED || g < nr) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[g][k * VEC + e] = fmaf(pw[g][it], f[e], o[g][k * VEC + e]);
          }
      }
    }
  }
}

// Ring budget of a phase kernel of NW warps: two stages per warp for 16-bit
// data while that fits (the default budget for 8 warps), at most 200 KB.
template <typename T, int D, int NW>
__host__ __device__ constexpr int grouped_ring_budget() {
  return NW == kDecodeWarps ? 0
                            : (NW * 4 * kTileTokens * D * (int)sizeof(T) < 200 * 1024
                                   ? NW * 4 * kTileTokens * D * (int)sizeof(T)
                                   : 200 * 1024);
}

// One phase of the grouped decode over persistent warps: PH = 0 runs every
// prefix segment, PH = 1 every tail segment, each balanced over all warps.
// The two phases are two launches in stream order, so the tail phase sees
// every prefix result (and the partial slots the prefix phase used are free);
// the tail launch may start early (programmatic dependent launch) and waits
// for the prefix grid right after issuing its first K/V copies.
template <typename T, int D, int TG, int PH, int NW>
__global__ void __launch_bounds__(NW * 32)
    pa_decode_grouped_kernel(const GroupedParams gp) {
  using S = DecodeShape<T, D, kGroupRows, T, NW, grouped_ring_budget<T, D, NW>()>;
  constexpr int R = kGroupRows;
  constexpr bool kMma = Mma16816<T>::kOk;
  constexpr int QR = kMma ? TG : R;  // query rows kept in fp32 registers
  constexpr int OR = kMma ? TG : R;  // rows of the CUDA-core accumulators
  constexpr int ST = S::kStages;
  constexpr int DPL = S::kDimsPerLane;
  constexpr int CPL = S::kChunksPerLane;
  constexpr int VEC = S::kVec;
  constexpr int ROW = S::kRowBytes;
  constexpr int DL = D / 32;  // dims per lane in merges
  const DecodeParams& p = gp.base;

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  long long* scan = reinterpret_cast<long long*>(smem + S::kScanOff);
  __shared__ longlong2 starts[NW];  // (group or sequence, offset) of each warp's first unit

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = lane >> 3;
  const int sub = lane & 7;
  const int mg = lane >> 2, mt = lane & 3;
  const int bs = p.block_size;
  GCtx x;
  x.group_start = gp.group_start;
  x.group_S = gp.ws_group_S;
  x.seq_P = gp.ws_seq_P;
  x.context_lens = p.context_lens;
  x.dev_err = p.dev_err;
  x.num_groups = gp.num_groups;
  x.num_seqs = p.num_seqs;
  x.num_heads = p.num_heads;
  x.head_groups = p.head_groups;
  x.group = p.group;
  x.cap = min(p.max_context_len, p.max_blocks_per_seq * bs);
  x.gpw = p.num_heads / p.head_groups;
  x.use_groups = __ldcg(gp.ws_flag) == 0;
  const int B = p.num_seqs, G = gp.num_groups, HG = p.head_groups, H = p.num_heads;

  // ---- start-up: work units of this phase, then each warp's first segment ----
  const long long W = (long long)gridDim.x * NW;
  const long long wid = (long long)blockIdx.x * NW + warp;
  long long mine = 0, Ttot = 0;
  if constexpr (PH == 0) {
    for (int g = threadIdx.x; g < G; g += NW * 32) mine += prefix_units(x, g);
  } else {
    for (int s = threadIdx.x; s < B; s += NW * 32)
      mine += (long long)HG * (tiles_of(ctx_len(x, s) - seq_prefix(x, s)) + kSegCostTail);
  }
  block_exclusive_scan<NW>(mine, scan, Ttot);
  const long long Weff = W < Ttot ? W : Ttot;  // 0 when the phase has no work
  if (threadIdx.x < NW) starts[threadIdx.x] = make_longlong2(-1, 0);
  __syncthreads();
  long long carry = 0;
  const int nitems = PH == 0 ? G : B;
  for (int base = 0; base < nitems; base += NW * 32) {
    const int i0 = base + threadIdx.x;
    long long cnt = 0;
    if (i0 < nitems) {
      if constexpr (PH == 0)
        cnt = prefix_units(x, i0);
      else
        cnt = (long long)HG * (tiles_of(ctx_len(x, i0) - seq_prefix(x, i0)) + kSegCostTail);
    }
    long long tot;
    const long long excl = carry + block_exclusive_scan<NW>(cnt, scan, tot);
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const long long w = (long long)blockIdx.x * NW + i;
      if (w < Weff) {
        const long long a = w * Ttot / Weff;
        if (cnt > 0 && a >= excl && a < excl + cnt) starts[i] = make_longlong2(i0, a - excl);
      }
    }
    carry += tot;
  }
  __syncthreads();  // the last block-wide barrier

  unsigned char* my_ring = smem + warp * ST * S::kStageBytes;
  uint64_t* my_bars = bars + warp * ST;
  int32_t* my_bt = reinterpret_cast<int32_t*>(smem + S::kBtOff) + warp * kBtChunk;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < ST; ++i) mbar_init(&my_bars[i], 1);
    mbar_init_fence();
  }
  __syncwarp();

  const char* kbase = static_cast<const char*>(p.k_cache);
  const char* vbase = static_cast<const char*>(p.v_cache);
  const char* qbase = static_cast<const char*>(p.q);
  const int seg = bs < kTileTokens ? bs : kTileTokens;
  const int nseg = kTileTokens / seg;
  int bt_s = -1, bt_j0 = 0;
  int ring = 0;  // tiles this warp has consumed so far (ring position)

  float qf[QR][DPL];
  uint32_t qa[D / 32][2][2];        // prefix query rows as MMA A-operands (16-bit types)
  float m[OR], l[OR], o[OR][DPL];   // CUDA-core state (tails; prefixes of fp32 data)
  float pm = -INFINITY, pl = 0.f;   // tensor-core state of a prefix: row mg
  float po[D / 32][4][2];

  {
    constexpr int phase = PH;
    const long long Tp = Ttot, Wp = Weff;
    const int E = phase == 0 ? kSegCostPrefix : kSegCostTail;
    const long long a_begin = wid < Wp ? wid * Tp / Wp : Tp;
    const long long a_end = wid < Wp ? (wid + 1) * Tp / Wp : Tp;
    if (a_begin < a_end) {
      GCursor ci;
      {
        const longlong2 st0 = starts[warp];
        ci.part = phase;
        ci.a = static_cast<int>(st0.x);
        ci.b = 0;
        ci.c = 0;
        gseg_enter(ci, x);  // nt does not depend on b or c
        const long long per = ci.nt + E;  // units of one segment
        const long long seg_idx = st0.y / per;
        const int r = static_cast<int>(st0.y % per) - E;
        ci.t = r < 0 ? 0 : r;  // a range that starts on charged units starts at tile 0
        ci.g = a_begin + (ci.t - r);
        if (phase == 0) {
          ci.b = static_cast<int>(seg_idx / group_rows(ci.M));
          ci.c = static_cast<int>(seg_idx % group_rows(ci.M));
        } else {
          ci.b = static_cast<int>(seg_idx);
        }
        gseg_enter(ci, x);
      }
      GCursor cc = ci;
      const long long g_first = ci.g;  // unit of this warp's first tile in the phase

      auto issue = [&](const GCursor& c, int n) {
        const int t0 = c.tok0 + c.t * kTileTokens;
        const int nvalid = min(max(c.tok_end - t0, 0), kTileTokens);
        const bool with_q = (c.t == 0 || c.g == g_first) && nvalid > 0;
        if (nvalid > 0) {
          const int j_first = t0 / bs;
          const int j_last = (t0 + nvalid - 1) / bs;
          if (c.sbt != bt_s || j_first < bt_j0 || j_last >= bt_j0 + kBtChunk) {
            // entries of the row's whole context: the chunk then serves any
            // segment that reads this row (prefix or tail)
            const int nblk = (c.sbt_len + bs - 1) / bs;
            const int32_t* row = p.block_tables + (size_t)c.sbt * p.max_blocks_per_seq;
            __syncwarp();
            for (int i = lane; i < kBtChunk; i += 32) {
              const int j = j_first + i;
              int id = 0;
              if (j < nblk) {
                id = __ldg(row + j);
                if (id < 0 || id >= p.num_blocks) {
                  set_err(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
                  id = 0;
                }
              }
              my_bt[i] = id;
            }
            __syncwarp();
            bt_s = c.sbt;
            bt_j0 = j_first;
          }
        }
        if (lane == 0) {
          unsigned char* kdst = my_ring + (n % ST) * S::kStageBytes;
          unsigned char* vdst = kdst + S::kTileBytes;
          unsigned char* qdst = kdst + 2 * S::kTileBytes;
          uint64_t* bar = my_bars + (n % ST);
          uint32_t bytes = with_q ? c.nrows * ROW : 0;
          for (int c2 = 0; c2 < nseg; ++c2)
            if (t0 + c2 * seg < c.tok_end) bytes += 2u * seg * ROW;
          mbar_arrive_expect_tx(bar, bytes);
          for (int c2 = 0; c2 < nseg; ++c2) {
            const int t = t0 + c2 * seg;
            if (t >= c.tok_end) break;
            const size_t off =
                (((size_t)my_bt[t / bs - bt_j0] * p.num_kv_heads + c.kvh) * bs + (t % bs)) * ROW;
            bulk_copy_g2s(kdst + c2 * seg * ROW, kbase + off, seg * ROW, bar);
            bulk_copy_g2s(vdst + c2 * seg * ROW, vbase + off, seg * ROW, bar);
          }
          if (with_q) {
            if (c.part == 1) {
              bulk_copy_g2s(qdst, qbase + ((size_t)c.a * H + (size_t)c.b * c.nrows) * ROW, c.nrows * ROW, bar);
            } else {
              for (int r = 0; r < c.nrows; ++r)
                bulk_copy_g2s(qdst + r * ROW, qbase + ((size_t)row_seq(c, r) * H + c.b) * ROW, ROW, bar);
            }
          }
        }
      };

      int issued = ring;
      for (; issued < ring + ST && ci.g < a_end; ++issued) {
        issue(ci, issued);
        gcursor_next(ci, x);
      }
      // the tail phase reads prefix results and reuses the partial slots:
      // wait for the prefix grid (its first K/V copies are already in flight)
      if constexpr (PH == 1) asm volatile("griddepcontrol.wait;" ::: "memory");
      bool visit_from_start = true;

      for (; cc.g < a_end; ++ring) {
        if (!__all_sync(kFullMask, mbar_wait_bounded(my_bars + (ring % ST), (ring / ST) & 1, p.wait_limit_ns))) {
          if (lane == 0) set_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
          for (int k2 = ring; k2 < issued; ++k2)
            mbar_wait_bounded(my_bars + (k2 % ST), (k2 / ST) & 1, kDrainLimitNs);
          return;  // outputs of this call are not valid
        }
        const unsigned char* ks = my_ring + (ring % ST) * S::kStageBytes;
        const unsigned char* vs = ks + S::kTileBytes;
        const int t0 = cc.tok0 + cc.t * kTileTokens;
        const int nvalid = min(max(cc.tok_end - t0, 0), kTileTokens);
        const bool first = cc.t == 0 || cc.g == g_first;
        const bool last = cc.t == cc.nt - 1 || cc.g == a_end - 1;
        const int nr = cc.nrows;
        const bool tc_prefix = kMma && phase == 0;  // state in the tensor-core layout

        if (first) {
          visit_from_start = cc.t == 0;
          pm = -INFINITY;
          pl = 0.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c)
#pragma unroll
            for (int q = 0; q < 4; ++q) po[c][q][0] = po[c][q][1] = 0.f;
#pragma unroll
          for (int g = 0; g < OR; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[g][e] = 0.f;
          }
          if (nvalid > 0) {
            const unsigned char* qs = ks + 2 * S::kTileBytes;
            if (tc_prefix) {
#pragma unroll
              for (int c = 0; c < D / 32; ++c)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                  const int d0 = c * 32 + 8 * mt + 4 * j;  // dims d0, d0+1 | d0+2, d0+3 (see Mma16816)
                  const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qs + mg * ROW);
                  qa[c][j][0] = mg < nr ? qrow[d0 / 2] : 0u;
                  qa[c][j][1] = mg < nr ? qrow[d0 / 2 + 1] : 0u;
                }
            } else {
#pragma unroll
              for (int g = 0; g < QR; ++g) {
                if (g < nr) {
                  const uint4* qrow = reinterpret_cast<const uint4*>(qs + g * ROW);
#pragma unroll
                  for (int k = 0; k < CPL; ++k) {
                    float f[VEC];
                    Chunk<T>::widen(qrow[sub + 8 * k], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) qf[g][k * VEC + e] = f[e] * p.scale_log2;
                  }
                }
              }
            }
          }
        }

        if (nvalid > 0) {
          if (phase == 1) {
            core_tile<T, D, QR, TG, false, OR>(ks, vs, qf, o, m, l, nvalid, TG);
          } else if constexpr (kMma) {
            mma_prefix_tile<T, D>(ks, vs, qa, po, pm, pl, nvalid, p.scale_log2);
          } else {
            core_tile<T, D, QR, R, true, OR>(ks, vs, qf, o, m, l, nvalid, nr);
          }
        }
        __syncwarp();
        if (ci.g < a_end) {
          issue(ci, issued++);
          gcursor_next(ci, x);
        }

        if (last) {
          // ---- end of this warp's visit of the segment under cc --------------
#pragma unroll
          for (int g = 0; g < OR; ++g)
            if (!tc_prefix && g < nr) {
              l[g] += __shfl_xor_sync(kFullMask, l[g], 8);
              l[g] += __shfl_xor_sync(kFullMask, l[g], 16);
#pragma unroll
              for (int e = 0; e < DPL; ++e) {
                o[g][e] += __shfl_xor_sync(kFullMask, o[g][e], 8);
                o[g][e] += __shfl_xor_sync(kFullMask, o[g][e], 16);
              }
            }
          // phase 1 rows of a sequence with a shared prefix merge with its result
          const bool with_prefix = phase == 1 && cc.tok0 > 0;
          const bool whole = visit_from_start && cc.t == cc.nt - 1;
          if (whole && tc_prefix) {
            // prefix result of each sibling row (rows are quads of lanes)
            if (mg < nr) {
              const size_t row = (size_t)row_seq(cc, mg) * H + row_head(cc, x, mg);
              const float inv = 1.f / pl;
              float4* dst = reinterpret_cast<float4*>(gp.ws_row_o + row * D);
#pragma unroll
              for (int c = 0; c < D / 32; ++c) {
                dst[(c * 32 + 8 * mt) / 4] = make_float4(po[c][0][0] * inv, po[c][0][1] * inv,
                                                         po[c][1][0] * inv, po[c][1][1] * inv);
                dst[(c * 32 + 8 * mt) / 4 + 1] = make_float4(po[c][2][0] * inv, po[c][2][1] * inv,
                                                             po[c][3][0] * inv, po[c][3][1] * inv);
              }
              if (mt == 0) gp.ws_row_ml[row] = make_float2(pm, pl);
            }
          } else if (whole) {
#pragma unroll
            for (int g = 0; g < OR; ++g) {
              if (g >= nr) continue;
              const size_t row = (size_t)row_seq(cc, g) * H + row_head(cc, x, g);
              if (phase == 0) {  // prefix result (fp32 data)
                const float inv = 1.f / l[g];
                if (grp == 0) {
                  float4* dst = reinterpret_cast<float4*>(gp.ws_row_o + row * D);
#pragma unroll
                  for (int k = 0; k < CPL; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; e += 4)
                      dst[((sub + 8 * k) * VEC + e) / 4] =
                          make_float4(o[g][k * VEC + e] * inv, o[g][k * VEC + e + 1] * inv,
                                      o[g][k * VEC + e + 2] * inv, o[g][k * VEC + e + 3] * inv);
                }
                if (lane == 0) gp.ws_row_ml[row] = make_float2(m[g], l[g]);
                continue;
              }
              float w_own = 1.f, w_pre = 0.f, denom = l[g];
              if (with_prefix) {
                const float2 pr = __ldcg(gp.ws_row_ml + row);
                const float M = fmaxf(m[g], pr.x);
                w_own = m[g] == -INFINITY ? 0.f : exp2f(m[g] - M);
                w_pre = pr.y * exp2f(pr.x - M);
                denom = l[g] * w_own + w_pre;
              }
              const float inv = denom > 0.f ? 1.f / denom : 0.f;
              if (grp == 0) {
                uint4* orow = reinterpret_cast<uint4*>(static_cast<char*>(p.out) + row * ROW);
                const float* pre = gp.ws_row_o + row * D;
#pragma unroll
                for (int k = 0; k < CPL; ++k) {
                  float f[VEC];
#pragma unroll
                  for (int e = 0; e < VEC; ++e) {
                    const float pv = with_prefix ? __ldcg(pre + (sub + 8 * k) * VEC + e) : 0.f;
                    f[e] = (o[g][k * VEC + e] * w_own + pv * w_pre) * inv;
                  }
                  orow[sub + 8 * k] = Chunk<T>::narrow(f);
                }
              }
            }
          } else {
            // one piece of a segment shared with neighbouring warps
            const long long Wq = Wp, Tq = Tp;
            // slot 0: the piece holding the warp's first tile (its range starts
            // in this segment, charged units included); slot 1: its last piece
            const int slot = cc.g - cc.t - E <= a_begin ? 0 : 1;
            const size_t base = ((size_t)wid * 2 + slot) * R;
            if (tc_prefix) {
              if (mg < nr) {
                const float inv = 1.f / pl;
                float4* dst = reinterpret_cast<float4*>(p.ws_o + (base + mg) * D);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                  dst[(c * 32 + 8 * mt) / 4] = make_float4(po[c][0][0] * inv, po[c][0][1] * inv,
                                                           po[c][1][0] * inv, po[c][1][1] * inv);
                  dst[(c * 32 + 8 * mt) / 4 + 1] = make_float4(po[c][2][0] * inv, po[c][2][1] * inv,
                                                               po[c][3][0] * inv, po[c][3][1] * inv);
                }
                if (mt == 0) p.ws_ml[base + mg] = make_float2(pm, pl);
              }
            } else {
#pragma unroll
              for (int g = 0; g < OR; ++g) {
                if (g >= nr) continue;
                const float inv = l[g] > 0.f ? 1.f / l[g] : 0.f;
                if (grp == 0) {
                  float4* dst = reinterpret_cast<float4*>(p.ws_o + (base + g) * D);
#pragma unroll
                  for (int k = 0; k < CPL; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; e += 4)
                      dst[((sub + 8 * k) * VEC + e) / 4] =
                          make_float4(o[g][k * VEC + e] * inv, o[g][k * VEC + e + 1] * inv,
                                      o[g][k * VEC + e + 2] * inv, o[g][k * VEC + e + 3] * inv);
                }
                if (lane == 0) p.ws_ml[base + g] = make_float2(m[g], l[g]);
              }
            }
            __syncwarp();  // the partial's writes precede lane 0's release below
            const long long seg_start = cc.g - cc.t;  // unit of the segment's first tile
            const long long seg_end = seg_start + cc.nt;
            const long long seg_units0 = seg_start - E;  // its first charged unit
            const long long w_first = ((seg_start + 1) * Wq + Tq - 1) / Tq - 1;
            const long long w_last = (seg_end * Wq + Tq - 1) / Tq - 1;
            int is_last = 0;
            if (lane == 0) {
              const size_t ci_idx = phase == 0 ? (size_t)(cc.lo + kGroupRows * cc.c) * H + cc.b
                                               : (size_t)B * H + (size_t)cc.a * HG + cc.b;
              int32_t* ctr = gp.ws_seg_ctr + ci_idx;
              const int prev = atomic_add_acq_rel_gpu(ctr, 1);
              is_last = prev == (int)(w_last - w_first);
              if (is_last) *ctr = 0;
            }
            is_last = __shfl_sync(kFullMask, is_last, 0);
            if (is_last) {
              __syncwarp();  // the other pieces' partials, acquired by lane 0, are visible to all lanes
              for (int g = 0; g < nr; ++g) {
                const size_t row = (size_t)row_seq(cc, g) * H + row_head(cc, x, g);
                float M = -INFINITY;
                for (long long w = w_first; w <= w_last; ++w) {
                  const int sl = (w == w_first && w * Tq / Wq < seg_units0) ? 1 : 0;
                  M = fmaxf(M, __ldcg(p.ws_ml + ((size_t)w * 2 + sl) * R + g).x);
                }
                float2 pr = make_float2(-INFINITY, 0.f);
                if (with_prefix) {
                  pr = __ldcg(gp.ws_row_ml + row);
                  M = fmaxf(M, pr.x);
                }
                float Ls = 0.f, O[DL];
#pragma unroll
                for (int e = 0; e < DL; ++e) O[e] = 0.f;
                for (long long w = w_first; w <= w_last; ++w) {
                  const int sl = (w == w_first && w * Tq / Wq < seg_units0) ? 1 : 0;
                  const size_t idx = ((size_t)w * 2 + sl) * R + g;
                  const float2 v = __ldcg(p.ws_ml + idx);
                  const float wt = v.x == -INFINITY ? 0.f : v.y * exp2f(v.x - M);
                  Ls += wt;
                  const float* src = p.ws_o + idx * D + lane * DL;
#pragma unroll
                  for (int e = 0; e < DL; ++e) O[e] += __ldcg(src + e) * wt;
                }
                if (with_prefix) {
                  const float wt = pr.y * exp2f(pr.x - M);
                  Ls += wt;
                  const float* src = gp.ws_row_o + row * D + lane * DL;
#pragma unroll
                  for (int e = 0; e < DL; ++e) O[e] += __ldcg(src + e) * wt;
                }
                if (phase == 0) {  // merged prefix result of this row
                  float* dst = gp.ws_row_o + row * D + lane * DL;
#pragma unroll
                  for (int e = 0; e < DL; ++e) dst[e] = O[e] / Ls;
                  if (lane == 0) gp.ws_row_ml[row] = make_float2(M, Ls);
                } else {
                  T* orow = static_cast<T*>(p.out) + row * D + lane * DL;
#pragma unroll
                  for (int e = 0; e < DL; ++e) store_elem(orow + e, Ls > 0.f ? O[e] / Ls : 0.f);
                }
              }
            }
          }
        }
        gcursor_next(cc, x);
      }
    }
  }
}

// Persistent grid of one phase kernel on the current device (cached).
template <typename T, int D, int TG, int PH, int NW>
cudaError_t grouped_grid(int& grid) {
  using S = DecodeShape<T, D, kGroupRows, T, NW, grouped_ring_budget<T, D, NW>()>;
  static int grid_of_device[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  grid = (dev >= 0 && dev < 64) ? __atomic_load_n(&grid_of_device[dev], __ATOMIC_ACQUIRE) : 0;
  if (grid != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(pa_decode_grouped_kernel<T, D, TG, PH, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           S::kSmemBytes);
  if (e != cudaSuccess) return e;
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pa_decode_grouped_kernel<T, D, TG, PH, NW>, NW * 32,
                                                    S::kSmemBytes);
  if (e != cudaSuccess) return e;
  grid = sms * (per_sm > 0 ? per_sm : 1);
  if (grid > kMaxDecodeWarps / NW) grid = kMaxDecodeWarps / NW;
  if (dev >= 0 && dev < 64) __atomic_store_n(&grid_of_device[dev], grid, __ATOMIC_RELEASE);
  return cudaSuccess;
}

// Warps per block of each phase kernel: the tail phase of 16-bit data runs
// 12 warps (measured on the copy-on-write workload: prefix/tail warps 8/8
// 160.1 us, 8/12 157.4 us, 12/8 167.9 us, 12/12 165.9 us, 12/16 168.3 us).
template <typename T, int PH>
__host__ __device__ constexpr int grouped_warps() { return sizeof(T) == 2 && PH == 1 ? 12 : kDecodeWarps; }

// Validation prologue, the prefix phase, then the tail phase (launched as a
// programmatic dependent of the prefix phase, so its start-up overlaps the
// prefix phase's last blocks).
template <typename T, int D, int TG>
cudaError_t launch_pa_decode_grouped(const GroupedParams& gp, cudaStream_t stream) {
  constexpr int NW0 = grouped_warps<T, 0>(), NW1 = grouped_warps<T, 1>();
  using S0 = DecodeShape<T, D, kGroupRows, T, NW0, grouped_ring_budget<T, D, NW0>()>;
  using S1 = DecodeShape<T, D, kGroupRows, T, NW1, grouped_ring_budget<T, D, NW1>()>;
  int grid0 = 0, grid1 = 0;
  cudaError_t e = grouped_grid<T, D, TG, 0, NW0>(grid0);
  if (e != cudaSuccess) return e;
  e = grouped_grid<T, D, TG, 1, NW1>(grid1);
  if (e != cudaSuccess) return e;
  int pro = (gp.num_groups + 7) / 8;
  pro = pro < 1 ? 1 : (pro > 4096 ? 4096 : pro);
  pa_group_prologue_kernel<T><<<pro, 256, 0, stream>>>(gp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pa_decode_grouped_kernel<T, D, TG, 0, NW0><<<grid0, NW0 * 32, S0::kSmemBytes, stream>>>(gp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid1);
  cfg.blockDim = dim3(NW1 * 32);
  cfg.dynamicSmemBytes = S1::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, pa_decode_grouped_kernel<T, D, TG, 1, NW1>, gp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

using GroupedLauncher = cudaError_t (*)(const GroupedParams&, cudaStream_t);

// gpw_index: query heads per warp in the tails, 0 -> 1, 1 -> 2, 2 -> 4.
GroupedLauncher grouped_launcher_f32(int head_dim, int gpw_index);
GroupedLauncher grouped_launcher_f16(int head_dim, int gpw_index);
GroupedLauncher grouped_launcher_bf16(int head_dim, int gpw_index);

}  // namespace pkv
