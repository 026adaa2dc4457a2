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
//     group's shared blocks against the query rows of up to prefix_rows<T>()
//     siblings (head h of members R c .. R c + R - 1, R = prefix_rows<T>());
//   tail segments (sequence s, head group hg): rows [S_g, L_s) of s's own
//     blocks against its query heads, as in the plain kernel.
// 16-bit data: one persistent launch (pa_decode_shared_kernel) walks, per
// (group, head group), the prefix segment and then the members' tails, all
// balanced over the warps by cost units; a row's prefix and tail results meet
// by the log-sum-exp rule in the warp's shared memory or through the
// workspace. fp32 data: the prefix segments run first, balanced over all
// warps, then the tails, balanced again, as two launches in stream order; a
// tail row merges its prefix result when it writes the output. Pieces of a
// segment cut by warp range boundaries are merged as in the plain kernel.
//
// A prologue kernel checks the caller's grouping: group_start must partition
// [0, num_seqs) and the first shared_blocks[g] block-table entries of every
// member must be equal. The usable prefix S_g is the checked shared length
// cut to whole tiles and whole blocks and to the shortest member's context.
// A grouping that fails the check sets PKV_DEV_ERR_GROUP and is ignored (the
// kernel then computes the plain result), so a wrong promise never gives a
// wrong answer silently.
#pragma once

#include <cstring>
#include <type_traits>

#include "decode.cuh"
#include "tc.cuh"

namespace pkv {

// Query rows one warp serves against each shared K/V tile of a prefix
// segment: 16-bit data, the N = 8 columns of an m16n8k16 MMA whose M is the
// tile's 16 tokens; fp32 data, 4 rows on CUDA cores.
template <typename T>
__host__ __device__ constexpr int prefix_rows() { return sizeof(T) == 2 ? 8 : 4; }
constexpr int kMaxPrefixRows = 8;

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
  int32_t* ws_group_S;  // [num_groups] usable shared prefix tokens
  long long* ws_group_units;  // [num_groups] work units of the group (single-launch kernel)
  int32_t* ws_seq_P;    // [num_seqs] prefix tokens of the sequence's group
  int32_t* ws_seg_ctr;  // [2][num_seqs * num_heads] piece counters (prefix, tail)
  float2* ws_row_ml;    // [num_seqs * num_heads] (m, l) of each row's prefix result
  float* ws_row_o;      // [num_seqs * num_heads][head_dim] o / l of each row's prefix result
  // single-launch kernel (16-bit data): the tail part of rows whose parts meet
  // through the workspace, and each row's count of arrived parts
  float2* ws_tail_ml;   // [num_seqs * num_heads]
  float* ws_tail_o;     // [num_seqs * num_heads][head_dim]
  int32_t* ws_row_ctr;  // [num_seqs * num_heads]
};

// Work units of the single-launch kernel, in eighths of a prefix tile's
// time (measured per warp on the copy-on-write step): a prefix tile 8, a
// tail tile 10 (one query row on CUDA cores, its last tile often partly
// filled), the end of a prefix segment 28 and of a tail segment 25
// (reductions, and the two parts of each row meeting in shared memory or
// through the workspace). A tile belongs to the warp whose unit range holds
// its first unit; ranges are at least kUnitMax long, so every warp between
// the first and the last of a segment's warps gets some of its tiles.
constexpr int kUnitP = 8, kUnitT = 10, kChargeP = 28, kChargeT = 25, kUnitMax = 10;

__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFullMask, v, o));
  return v;
}

// One warp per group: validation of the grouping and the usable prefix.
// (A template only so that every element-type unit owns its own copy.)
template <typename T>
__global__ void __launch_bounds__(256) pa_group_prologue_kernel(const GroupedParams gp) {
  grid_launch_dependents();  // the prefix launch may start; it waits for these results
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
    // the group's work units (head groups x (prefix segments + member tails)),
    // read by the single-launch kernel's start-up instead of recomputing them
    const int HG = p.head_groups, gpw = p.num_heads / p.head_groups;
    long long u = 0;
    for (int s = lo + lane; s < hi; s += 32) {
      u += (long long)tiles_of(load_len(p, s, cap) - S) * kUnitT + kChargeT;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(kFullMask, u, o);
    if (S > 0) u += (long long)gpw * ((hi - lo + kMaxPrefixRows - 1) / kMaxPrefixRows) *
                    ((long long)(S / kTileTokens) * kUnitP + kChargeP);
    if (lane == 0) {
      gp.ws_group_S[g] = S;
      gp.ws_group_units[g] = (long long)HG * u;
    }
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
  int rows;  // query rows of a prefix segment
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

__device__ __forceinline__ int group_rows(int M, int rows) { return (M + rows - 1) / rows; }

// Work units of group g's prefix segments: tiles plus the per-segment cost
// (0 when the group has no usable shared prefix).
__device__ __forceinline__ long long prefix_units(const GCtx& x, int g) {
  if (!x.use_groups) return 0;
  const int M = __ldg(x.group_start + g + 1) - __ldg(x.group_start + g);
  const int S = __ldcg(x.group_S + g);
  if (M < 2 || S <= 0) return 0;
  return (long long)x.num_heads * group_rows(M, x.rows) * (S / kTileTokens + kSegCostPrefix);
}

__device__ __forceinline__ int seq_prefix(const GCtx& x, int s) { return x.use_groups ? __ldcg(x.seq_P + s) : 0; }

__device__ __forceinline__ void gseg_enter(GCursor& c, const GCtx& x) {
  if (c.part == 0) {
    c.lo = __ldg(x.group_start + c.a);
    c.M = __ldg(x.group_start + c.a + 1) - c.lo;
    c.tok0 = 0;
    c.tok_end = __ldcg(x.group_S + c.a);
    c.sbt = c.lo;
    c.sbt_len = ctx_len(x, c.lo);
    c.kvh = c.b / x.group;
    c.nrows = min(x.rows, c.M - x.rows * c.c);
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
    if (++c.c < group_rows(c.M, x.rows)) {
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
__device__ __forceinline__ int row_seq(const GCursor& c, const GCtx& x, int r) {
  return c.part == 0 ? c.lo + x.rows * c.c + r : c.a;
}
__device__ __forceinline__ int row_head(const GCursor& c, const GCtx& x, int r) {
  return c.part == 0 ? c.b : c.b * x.gpw + r;
}

// ---- tensor-core prefix tiles ------------------------------------------------
// m16n8k16 MMA with fp32 accumulation, D += A B: A 16x16 (four registers of
// 16-bit pairs), B 16x8 (two), D 16x8 (four fp32). Lane 4g + t holds
// A rows g and g+8, k-pairs 2t and 2t+8; B column g, k-pairs 2t and 2t+8;
// D rows g and g+8, columns 2t and 2t+1.
template <typename T>
struct Mma16816 {
  static constexpr bool kOk = false;
  __device__ __forceinline__ static void run(float (&)[4], const uint32_t (&)[4], uint32_t, uint32_t) {}
  __device__ __forceinline__ static uint32_t pack(float, float) { return 0u; }
  __device__ __forceinline__ static float2 unpack(uint32_t) { return make_float2(0.f, 0.f); }
};
template <>
struct Mma16816<__nv_bfloat16> {
  static constexpr bool kOk = true;
  __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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
  __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

// Shared-memory stage of the tensor-core prefix phase: the K and then the V
// rows of one 16-token tile, each as D/64 column blocks of 16 rows x 128 bytes
// with the 128-byte swizzle (16-byte chunk c of row r at position c ^ (r & 7)),
// exactly as TMA boxes of {64 elements, up to 16 rows} land in 1024-byte
// aligned memory; then the segment's query rows (plain, D elements each).
template <int D>
struct PrefixStage {
  static constexpr int kColBytes = kTileTokens * 128;
  static constexpr int kTensorBytes = (D / 64) * kColBytes;
  static constexpr int kQOff = 2 * kTensorBytes;
  static constexpr int kBytes = kQOff + kMaxPrefixRows * D * 2;
  static_assert(kBytes % 1024 == 0, "stages stay 1024-byte aligned");
};

// Byte offset of 16-byte chunk `ch` (0 .. D/8 - 1) of token row `tok` in a
// swizzled K or V tile.
__device__ __forceinline__ uint32_t sw_tile_off(int tok, int ch) {
  return (uint32_t)((ch >> 3) * (kTileTokens * 128) + tok * 128 + (((ch & 7) ^ (tok & 7)) << 4));
}

// One 16-token tile of a prefix segment on tensor cores, with the tile's
// tokens as the MMA's M and the segment's query rows (up to 8) as its N:
//   S^T = K Q^T   (A = K rows from shared memory by ldmatrix; B = Q^T, the
//                  query rows' fragments qb, fixed for the segment);
//   online softmax of each query row (a column of S^T): lane 4g + t holds
//     rows 2t and 2t+1 for tokens g and g+8, so a row's maximum reduces over
//     the 8 lanes of equal t; the row sums stay per lane until the segment
//     ends;
//   O^T += V^T P^T (A = V^T by transposed ldmatrix of the V rows; B = P^T,
//     the S^T accumulators as 16-bit pairs transposed by movmatrix). P goes
//     in as a high and a low 16-bit part (two MMAs), so the probabilities
//     keep about 16 significant bits.
// acc[mb] holds O^T rows (head dims) 16 mb + g and 16 mb + g + 8 for query
// rows 2t, 2t+1. Prefix tiles are always full (16 valid tokens).
template <typename T, int D>
__device__ __forceinline__ void mma_prefix_tile(uint32_t stage, const uint32_t (&qb)[D / 16][2],
                                                float (&acc)[D / 16][4], float (&pm)[2], float (&pl)[2],
                                                float scale_log2) {
  using M = Mma16816<T>;
  const int lane = threadIdx.x & 31;
  // K: lane i addresses token (i & 7) + 8 ((i >> 3) & 1), chunk 2 ks + (i >> 4)
  const int ktok = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int khi = lane >> 4;
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};  // even / odd k-steps
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t a[4];
    ldsm_x4(stage + sw_tile_off(ktok, 2 * ks + khi), a);
    M::run((ks & 1) ? s1 : s0, a, qb[ks][0], qb[ks][1]);
  }
  float x[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = (s0[i] + s1[i]) * scale_log2;
  float mt[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mt[0] = fmaxf(mt[0], __shfl_xor_sync(kFullMask, mt[0], o));
    mt[1] = fmaxf(mt[1], __shfl_xor_sync(kFullMask, mt[1], o));
  }
  float alpha[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float mn = fmaxf(pm[e], mt[e]);
    alpha[e] = exp2f(pm[e] - mn);  // 0 on the segment's first tile (pm = -inf)
    pm[e] = mn;
  }
  float pe[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) pe[i] = exp2f(x[i] - pm[i & 1]);
  pl[0] = pl[0] * alpha[0] + (pe[0] + pe[2]);
  pl[1] = pl[1] * alpha[1] + (pe[1] + pe[3]);
  if (!__all_sync(kFullMask, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
    for (int mb = 0; mb < D / 16; ++mb) {
      acc[mb][0] *= alpha[0];
      acc[mb][1] *= alpha[1];
      acc[mb][2] *= alpha[0];
      acc[mb][3] *= alpha[1];
    }
  }
  // P^T fragments: (token g | g+8) x (rows 2t, 2t+1) pairs, transposed.
  // bfloat16 P (8 significant bits) goes as a high part and a remainder;
  // binary16 P (11 bits) alone keeps the outputs within the tolerance.
  constexpr bool kSplit = !std::is_same<T, __half>::value;
  const uint32_t h0 = M::pack(pe[0], pe[1]), h1 = M::pack(pe[2], pe[3]);
  const uint32_t bh0 = movmatrix_trans(h0), bh1 = movmatrix_trans(h1);
  uint32_t bl0 = 0u, bl1 = 0u;
  if constexpr (kSplit) {
    const float2 u0 = M::unpack(h0), u1 = M::unpack(h1);
    bl0 = movmatrix_trans(M::pack(pe[0] - u0.x, pe[1] - u0.y));
    bl1 = movmatrix_trans(M::pack(pe[2] - u1.x, pe[3] - u1.y));
  }
  // V: lane i addresses token (i & 7) + 8 (i >> 4), chunk 2 mb + ((i >> 3) & 1)
  const int vtok = (lane & 7) + ((lane >> 4) << 3);
  const int vhi = (lane >> 3) & 1;
  const uint32_t vstage = stage + PrefixStage<D>::kTensorBytes;
#pragma unroll
  for (int mb = 0; mb < D / 16; ++mb) {
    uint32_t a[4];
    ldsm_x4_trans(vstage + sw_tile_off(vtok, 2 * mb + vhi), a);
    M::run(acc[mb], a, bh0, bh1);
    if constexpr (kSplit) M::run(acc[mb], a, bl0, bl1);
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

// Shared memory of the tensor-core prefix phase (16-bit data): two
// PrefixStage stages per warp from a 1024-byte aligned base, then the
// warps' mbarriers, block-table chunks and the start-up scan's scratch.
template <int D, int NW>
struct PrefixShape {
  static constexpr int kStages = 2;
  static constexpr int kStageBytes = PrefixStage<D>::kBytes;
  static constexpr int kBarOff = NW * kStages * kStageBytes;
  static constexpr int kBtOff = kBarOff + NW * kStages * 8;
  static constexpr int kScanOff = kBtOff + NW * kBtChunk * 4;
  static constexpr int kSmemBytes = kScanOff + NW * 8 + 1024;  // + alignment of the base
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = PrefixStage<D>::kTensorBytes;
  static constexpr int kDimsPerLane = D / 8;
  static constexpr int kChunksPerLane = kRowBytes / 16 / 8;
  static constexpr int kVec = 8;
};

template <typename T, int D, int NW, int PH>
using GroupedShape = typename std::conditional<Mma16816<T>::kOk && PH == 0, PrefixShape<D, NW>,
                                               DecodeShape<T, D, kMaxGroupPerWarp, T, NW,
                                                           grouped_ring_budget<T, D, NW>()>>::type;

// One phase of the grouped decode over persistent warps: PH = 0 runs every
// prefix segment, PH = 1 every tail segment, each balanced over all warps.
// The two phases are two launches in stream order, so the tail phase sees
// every prefix result (and the partial slots the prefix phase used are free);
// the tail launch may start early (programmatic dependent launch) and waits
// for the prefix grid right after issuing its first K/V copies.
// The prefix phase of 16-bit data loads K/V tiles by TMA (kmap, vmap: the
// pools as rows of head_dim elements, boxes of {64, min(block_size, 16)}
// rows, 128-byte swizzle) and runs them on tensor cores; the tail phase and
// fp32 data use 1-D bulk copies (the maps are then unused).
template <typename T, int D, int TG, int PH, int NW>
__global__ void __launch_bounds__(NW * 32)
    pa_decode_grouped_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                             const GroupedParams gp) {
  using S = GroupedShape<T, D, NW, PH>;
  constexpr int R = prefix_rows<T>();
  constexpr bool kMma = Mma16816<T>::kOk;
  constexpr bool kTma = kMma && PH == 0;  // tensor-core prefix tiles, TMA-fed
  constexpr int QR = kMma ? TG : R;  // query rows kept in fp32 registers
  constexpr int OR = kMma ? TG : R;  // rows of the CUDA-core accumulators
  constexpr int ST = S::kStages;
  constexpr int DPL = S::kDimsPerLane;
  constexpr int CPL = S::kChunksPerLane;
  constexpr int VEC = S::kVec;
  constexpr int ROW = S::kRowBytes;
  constexpr int DL = D / 32;  // dims per lane in merges
  const DecodeParams& p = gp.base;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = kTma ? smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u) : smem_raw;
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
  x.rows = R;
  // the prefix launch is a programmatic dependent of the grouping check:
  // wait for its results (the tail launch may read them at once: its primary,
  // the prefix grid, started its work only after the check completed)
  if constexpr (PH == 0) grid_dependency_wait();
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
  float m[OR], l[OR], o[OR][DPL];   // CUDA-core state (tails; prefixes of fp32 data)
  // tensor-core state of a prefix segment (see mma_prefix_tile): query rows
  // as B fragments, O^T accumulators, running max and per-lane row sums of
  // rows 2t and 2t+1
  uint32_t qb[D / 16][2];
  float acc[D / 16][4];
  float tm[2] = {-INFINITY, -INFINITY}, tl[2] = {0.f, 0.f};

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
          ci.b = static_cast<int>(seg_idx / group_rows(ci.M, R));
          ci.c = static_cast<int>(seg_idx % group_rows(ci.M, R));
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
        if constexpr (kTma) {
          // prefix tiles are whole (the usable prefix is cut to whole tiles):
          // the K and V rows as TMA boxes of {64 dims, rb rows} into the
          // swizzled stage, from parallel lanes; the query rows by lane 0
          unsigned char* st = my_ring + (n % ST) * S::kStageBytes;
          uint64_t* bar = my_bars + (n % ST);
          if (lane == 0) mbar_arrive_expect_tx(bar, 2u * kTileTokens * ROW + (with_q ? c.nrows * ROW : 0u));
          __syncwarp();
          const int rb = bs < kTileTokens ? bs : kTileTokens;
          constexpr int CB = D / 64;
          const int per = (kTileTokens / rb) * CB;  // boxes per tensor
          if (lane < 2 * per) {
            const int tsr = lane / per, rem = lane - tsr * per;
            const int b = rem / CB, cb = rem - b * CB;
            const int t = t0 + b * rb;
            const int y = (my_bt[t / bs - bt_j0] * p.num_kv_heads + c.kvh) * bs + (t % bs);
            tma_load_2d(st + tsr * PrefixStage<D>::kTensorBytes + cb * PrefixStage<D>::kColBytes + b * rb * 128,
                        tsr ? &vmap : &kmap, cb * 64, y, bar);
          }
          if (with_q && lane == 0) {
            for (int r = 0; r < c.nrows; ++r)
              bulk_copy_g2s(st + PrefixStage<D>::kQOff + r * ROW,
                            qbase + ((size_t)row_seq(c, x, r) * H + c.b) * ROW, ROW, bar);
          }
        } else if (lane == 0) {
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
                bulk_copy_g2s(qdst + r * ROW, qbase + ((size_t)row_seq(c, x, r) * H + c.b) * ROW, ROW, bar);
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
      if constexpr (PH == 1) grid_dependency_wait();
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

        if (first) {
          visit_from_start = cc.t == 0;
          if constexpr (kTma) {
            tm[0] = tm[1] = -INFINITY;
            tl[0] = tl[1] = 0.f;
#pragma unroll
            for (int mb = 0; mb < D / 16; ++mb) acc[mb][0] = acc[mb][1] = acc[mb][2] = acc[mb][3] = 0.f;
          }
#pragma unroll
          for (int g = 0; g < OR; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[g][e] = 0.f;
          }
          if (nvalid > 0) {
            const unsigned char* qs = ks + (kTma ? PrefixStage<D>::kQOff : 2 * S::kTileBytes);
            if constexpr (kTma) {
              // B fragments of Q^T: lane 4g + t holds query row g, dims
              // 16 ks + 2t, +1 and 16 ks + 2t + 8, +9 (rows past nr: zero)
              const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qs + mg * ROW);
#pragma unroll
              for (int ks2 = 0; ks2 < D / 16; ++ks2) {
                qb[ks2][0] = mg < nr ? qrow[8 * ks2 + mt] : 0u;
                qb[ks2][1] = mg < nr ? qrow[8 * ks2 + mt + 4] : 0u;
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
          } else if constexpr (kTma) {
            mma_prefix_tile<T, D>(smem_u32(ks), qb, acc, tm, tl, p.scale_log2);
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
            if (!kTma && g < nr) {
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
          if constexpr (kTma) {
            // row sums: per-lane shares of rows 2t, 2t+1 over the 8 lanes of equal t
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              tl[e] += __shfl_xor_sync(kFullMask, tl[e], 4);
              tl[e] += __shfl_xor_sync(kFullMask, tl[e], 8);
              tl[e] += __shfl_xor_sync(kFullMask, tl[e], 16);
            }
          }
          // (m, l, o / l) of query rows 2t and 2t+1 of a tensor-core prefix
          // segment: into the rows' prefix results, or into partial slot `base`
          auto store_tc_rows = [&](bool prefix_result, size_t base) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int r = 2 * mt + e;
              if (r < nr) {
                const size_t dst = prefix_result ? (size_t)row_seq(cc, x, r) * H + row_head(cc, x, r) : base + r;
                float2* ml = prefix_result ? gp.ws_row_ml : p.ws_ml;
                float* orow = (prefix_result ? gp.ws_row_o : p.ws_o) + dst * D + mg;
                const float inv = 1.f / tl[e];
#pragma unroll
                for (int mb = 0; mb < D / 16; ++mb) {
                  orow[16 * mb] = acc[mb][e] * inv;
                  orow[16 * mb + 8] = acc[mb][e + 2] * inv;
                }
                if (mg == 0) ml[dst] = make_float2(tm[e], tl[e]);
              }
            }
          };
          if (whole && kTma) {
            store_tc_rows(true, 0);  // the prefix result of each sibling row
          } else if (whole) {
#pragma unroll
            for (int g = 0; g < OR; ++g) {
              if (g >= nr) continue;
              const size_t row = (size_t)row_seq(cc, x, g) * H + row_head(cc, x, g);
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
            if constexpr (kTma) {
              store_tc_rows(false, base);
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
              const size_t ci_idx = phase == 0 ? (size_t)(cc.lo + R * cc.c) * H + cc.b
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
                const size_t row = (size_t)row_seq(cc, x, g) * H + row_head(cc, x, g);
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

// ---- single-launch grouped decode (16-bit data) ------------------------------
//
// One persistent launch after the grouping check. Work units, laid end to
// end: for every group, for every head group hg, the group's prefix
// segments for the heads of hg (rows [0, S_g) of the shared blocks against up
// to 8 siblings' query rows, on tensor cores), then the tail segment of every
// member (rows [S_g, L_s) of its own blocks, CUDA cores). A row (member s,
// head h) of a group with a shared prefix has two parts, each merged over
// its pieces when warp ranges cut its segment (as in the plain kernel). The
// two parts of a row meet
//   - in the warp's shared memory, when one warp's range holds the row's
//     whole prefix segment and whole tail segment (the prefix results wait in
//     the warp's buffer until its tails end; nothing goes through global
//     memory);
//   - through the workspace otherwise: each part stores its (m, l, o / l)
//     and counts itself on the row's counter; the part that arrives second
//     merges both by the log-sum-exp rule, writes the output and clears the
//     counter.
// Sequences of rejected or single-member groups have tails only.


// Warps per block and ring stages per warp of the single-launch kernel
// (measured on the copy-on-write step, attention: 8 x 2 139.6 us, 6 x 3 164.9
// us, 4 x 3 213.4 us, 4 x 4 214.1 us; registers (244 per thread) and shared
// memory leave no room for more warps).
constexpr int kSharedWarps = 8, kSharedStages = 2;

// Rows whose pieces one warp loads together when it merges a segment cut by
// warp ranges (fewer where more query heads per warp leave fewer registers
// free).
template <int TG>
__host__ __device__ constexpr int merge_rows() { return TG == 1 ? 4 : TG == 2 ? 2 : 1; }

__device__ __forceinline__ int sunit(int part) { return part == 0 ? kUnitP : kUnitT; }
__device__ __forceinline__ int scharge(int part) { return part == 0 ? kChargeP : kChargeT; }

struct SCursor {
  long long g;        // first unit of the current tile
  int grp, hg, part, j, t, nt;
  int lo, M, S, nch;  // group: members [lo, lo + M), usable prefix S (0: none), row chunks of 8
  int h, c;           // prefix segment: query head and row chunk
  int tok0, tok_end, sbt, sbt_len, kvh, nrows;
};

// Groups the work runs over: the caller's groups, or one per sequence when the
// grouping was rejected.
__device__ __forceinline__ int sgroup_count(const GCtx& x) { return x.use_groups ? x.num_groups : x.num_seqs; }

__device__ __forceinline__ void sgroup_load(SCursor& c, const GCtx& x) {
  if (x.use_groups) {
    c.lo = __ldg(x.group_start + c.grp);
    c.M = __ldg(x.group_start + c.grp + 1) - c.lo;
    c.S = c.M >= 2 ? __ldcg(x.group_S + c.grp) : 0;
  } else {
    c.lo = c.grp;
    c.M = 1;
    c.S = 0;
  }
  c.nch = (c.M + kMaxPrefixRows - 1) / kMaxPrefixRows;
}

// Units of one prefix segment and of one head group of the loaded group.
__device__ __forceinline__ long long sprefix_seg_units(const SCursor& c) {
  return (long long)(c.S / kTileTokens) * kUnitP + kChargeP;
}
__device__ __forceinline__ long long shg_units(const SCursor& c, const GCtx& x) {
  long long u = c.S > 0 ? (long long)x.gpw * c.nch * sprefix_seg_units(c) : 0;
  for (int k = 0; k < c.M; ++k) u += (long long)tiles_of(ctx_len(x, c.lo + k) - c.S) * kUnitT + kChargeT;
  return u;
}

__device__ __forceinline__ void sseg_enter(SCursor& c, const GCtx& x) {
  if (c.part == 0) {
    const int hi = c.j / c.nch;
    c.c = c.j - hi * c.nch;
    c.h = c.hg * x.gpw + hi;
    c.nrows = min(kMaxPrefixRows, c.M - kMaxPrefixRows * c.c);
    c.tok0 = 0;
    c.tok_end = c.S;
    c.sbt = c.lo;
    c.sbt_len = ctx_len(x, c.lo);
    c.kvh = c.h / x.group;
    c.nt = c.S / kTileTokens;
  } else {
    const int s = c.lo + c.j;
    const int L = ctx_len(x, s);
    c.tok0 = c.S;
    c.tok_end = L;
    c.sbt = s;
    c.sbt_len = L;
    c.kvh = (c.hg * x.gpw) / x.group;
    c.nrows = x.gpw;
    c.nt = tiles_of(L - c.S);
  }
}

// Next segment (c.t is 0); past the last group the cursor stops changing.
__device__ __forceinline__ void sseg_next(SCursor& c, const GCtx& x, int NG) {
  if (c.part == 0) {
    if (++c.j < x.gpw * c.nch) {
      sseg_enter(c, x);
      return;
    }
    c.part = 1;
    c.j = 0;
    sseg_enter(c, x);
    return;
  }
  if (++c.j < c.M) {
    sseg_enter(c, x);
    return;
  }
  c.j = 0;
  if (++c.hg >= x.head_groups) {
    c.hg = 0;
    do {
      if (++c.grp >= NG) return;
      sgroup_load(c, x);
    } while (c.M == 0);
  }
  c.part = c.S > 0 ? 0 : 1;
  sseg_enter(c, x);
}

// Next tile: c.g is its first unit (the next segment's charge skipped).
__device__ __forceinline__ void scursor_next(SCursor& c, const GCtx& x, int NG) {
  c.g += sunit(c.part);
  if (++c.t < c.nt) return;
  c.t = 0;
  sseg_next(c, x, NG);
  c.g += scharge(c.part);
}

// Shared memory of the single-launch kernel: two stages per warp (a prefix
// tile as swizzled TMA boxes, or a tail tile as plain rows at the same
// offsets), then per warp the prefix results of its latest prefix segment
// (8 rows of o / l, m, l) and the results of its current tail segment (4
// rows), then mbarriers, block-table chunks and the start-up scan.
template <int D, int NW>
struct SharedShape {
  static constexpr int kStages = kSharedStages;
  static constexpr int kStageBytes = PrefixStage<D>::kBytes;
  static constexpr int kRowFloats = D + 4;  // o / l, then m and l
  static constexpr int kPbufOff = NW * kStages * kStageBytes;
  static constexpr int kTbufOff = kPbufOff + NW * kMaxPrefixRows * kRowFloats * 4;
  static constexpr int kBarOff = kTbufOff + NW * kMaxGroupPerWarp * kRowFloats * 4;
  static constexpr int kBtOff = kBarOff + NW * kStages * 8;
  static constexpr int kScanOff = kBtOff + NW * kBtChunk * 4;
  static constexpr int kSmemBytes = kScanOff + NW * 8 + 1024;  // + alignment of the base
};

// out = (a.o a.l 2^(a.m - M) + b.o b.l 2^(b.m - M)) / (a.l 2^(a.m - M) + b.l 2^(b.m - M)),
// M = max(a.m, b.m), for this lane's DL dims; a, b hold normalised o (o / l).
template <int DL>
__device__ __forceinline__ void lse_combine(float am, float al, const float (&ao)[DL], float bm, float bl,
                                            const float (&bo)[DL], float (&out)[DL]) {
  const float M = fmaxf(am, bm);
  const float wa = am == -INFINITY ? 0.f : al * exp2f(am - M);
  const float wb = bm == -INFINITY ? 0.f : bl * exp2f(bm - M);
  const float den = wa + wb;
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int e = 0; e < DL; ++e) out[e] = (ao[e] * wa + bo[e] * wb) * inv;
}

template <typename T, int D, int TG>
__global__ void __launch_bounds__(kSharedWarps * 32)
    pa_decode_shared_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                            const GroupedParams gp) {
  constexpr int NW = kSharedWarps;
  using S = SharedShape<D, NW>;
  using St = PrefixStage<D>;
  constexpr int R = kMaxPrefixRows;
  constexpr int ST = S::kStages;
  constexpr int ROW = D * 2;
  constexpr int VEC = 8;
  constexpr int CPL = ROW / 16 / 8;
  constexpr int DPL = D / 8;
  constexpr int DL = D / 32;  // dims per lane in merges and combines
  constexpr int RF = S::kRowFloats;
  constexpr int kMergeRows = merge_rows<TG>();
  const DecodeParams& p = gp.base;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  long long* scan = reinterpret_cast<long long*>(smem + S::kScanOff);
  __shared__ longlong2 starts[NW];  // (group, offset) of each warp's first unit

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
  x.rows = R;
  grid_dependency_wait();  // the grouping check's results
  x.use_groups = __ldcg(gp.ws_flag) == 0;
  const int NG = sgroup_count(x);
  const int H = p.num_heads, HG = p.head_groups;

  // ---- start-up: units of every group, then each warp's first segment -------
  const long long W = (long long)gridDim.x * NW;
  const long long wid = (long long)blockIdx.x * NW + warp;
  auto group_units = [&](int gi) -> long long {
    if (x.use_groups) return __ldcg(gp.ws_group_units + gi);  // from the grouping check
    SCursor c;
    c.grp = gi;
    sgroup_load(c, x);
    return (long long)HG * shg_units(c, x);
  };
  long long mine = 0, Ttot = 0;
  for (int gi = threadIdx.x; gi < NG; gi += NW * 32) mine += group_units(gi);
  block_exclusive_scan<NW>(mine, scan, Ttot);
  const long long Weff = W < Ttot / kUnitMax ? W : Ttot / kUnitMax;
  if (threadIdx.x < NW) starts[threadIdx.x] = make_longlong2(-1, 0);
  __syncthreads();
  long long carry = 0;
  for (int base = 0; base < NG; base += NW * 32) {
    const int i0 = base + threadIdx.x;
    const long long cnt = i0 < NG ? group_units(i0) : 0;
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

  const long long a_begin = wid < Weff ? wid * Ttot / Weff : Ttot;
  const long long a_end = wid < Weff ? (wid + 1) * Ttot / Weff : Ttot;
  if (a_begin >= a_end) return;

  unsigned char* my_ring = smem + warp * ST * S::kStageBytes;
  float* pbuf = reinterpret_cast<float*>(smem + S::kPbufOff) + warp * R * RF;
  float* tbuf = reinterpret_cast<float*>(smem + S::kTbufOff) + warp * kMaxGroupPerWarp * RF;
  uint64_t* my_bars = bars + warp * ST;
  int32_t* my_bt = reinterpret_cast<int32_t*>(smem + S::kBtOff) + warp * kBtChunk;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < ST; ++i) mbar_init(&my_bars[i], 1);
    mbar_init_fence();
  }
  __syncwarp();

  // ---- this warp's first segment ----------------------------------------------
  SCursor ci;
  {
    const longlong2 st0 = starts[warp];
    ci.grp = static_cast<int>(st0.x);
    sgroup_load(ci, x);
    const long long uhg = x.use_groups ? __ldcg(gp.ws_group_units + ci.grp) / HG : shg_units(ci, x);
    ci.hg = static_cast<int>(st0.y / uhg);
    long long r = st0.y - ci.hg * uhg;
    const long long pseg = sprefix_seg_units(ci);
    const long long pu = ci.S > 0 ? (long long)x.gpw * ci.nch * pseg : 0;
    long long r2;  // the range's start relative to the segment's first tile
    if (r < pu) {
      ci.part = 0;
      ci.j = static_cast<int>(r / pseg);
      r2 = r - ci.j * pseg - kChargeP;
    } else {
      r -= pu;
      ci.part = 1;
      int k = 0;
      for (;;) {
        const long long uk = (long long)tiles_of(ctx_len(x, ci.lo + k) - ci.S) * kUnitT + kChargeT;
        if (r < uk || k == ci.M - 1) break;
        r -= uk;
        ++k;
      }
      ci.j = k;
      r2 = r - kChargeT;
    }
    ci.t = 0;
    sseg_enter(ci, x);
    // the first tile whose first unit is inside the range
    const int w = sunit(ci.part);
    const long long t = r2 <= 0 ? 0 : (r2 + w - 1) / w;
    if (t < ci.nt) {
      ci.t = static_cast<int>(t);
      ci.g = a_begin - r2 + t * w;
    } else {  // the segment's last tile began before the range: start at the next one
      ci.g = a_begin - r2 + (long long)ci.nt * w;
      sseg_next(ci, x, NG);
      ci.g += scharge(ci.part);
    }
  }
  SCursor cc = ci;
  const long long g_first = ci.g;

  const char* kbase = static_cast<const char*>(p.k_cache);
  const char* vbase = static_cast<const char*>(p.v_cache);
  const char* qbase = static_cast<const char*>(p.q);
  const int seg = bs < kTileTokens ? bs : kTileTokens;
  const int nseg = kTileTokens / seg;
  int bt_s = -1, bt_j0 = 0;

  auto issue = [&](const SCursor& c, int n) {
    const int t0 = c.tok0 + c.t * kTileTokens;
    const int nvalid = min(max(c.tok_end - t0, 0), kTileTokens);
    const bool with_q = (c.t == 0 || c.g == g_first) && nvalid > 0;
    if (nvalid > 0) {
      const int j_first = t0 / bs;
      const int j_last = (t0 + nvalid - 1) / bs;
      if (c.sbt != bt_s || j_first < bt_j0 || j_last >= bt_j0 + kBtChunk) {
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
    unsigned char* st = my_ring + (n % ST) * S::kStageBytes;
    uint64_t* bar = my_bars + (n % ST);
    if (c.part == 0) {
      // a whole prefix tile: K and V as TMA boxes of {64 dims, rb rows} into
      // the swizzled stage, from parallel lanes; the siblings' query rows
      if (lane == 0) mbar_arrive_expect_tx(bar, 2u * kTileTokens * ROW + (with_q ? c.nrows * ROW : 0u));
      __syncwarp();
      const int rb = bs < kTileTokens ? bs : kTileTokens;
      constexpr int CB = D / 64;
      const int per = (kTileTokens / rb) * CB;
      if (lane < 2 * per) {
        const int tsr = lane / per, rem = lane - tsr * per;
        const int b = rem / CB, cb = rem - b * CB;
        const int t = t0 + b * rb;
        const int y = (my_bt[t / bs - bt_j0] * p.num_kv_heads + c.kvh) * bs + (t % bs);
        tma_load_2d(st + tsr * St::kTensorBytes + cb * St::kColBytes + b * rb * 128, tsr ? &vmap : &kmap, cb * 64, y,
                    bar);
      }
      // the siblings' query rows, one lane each after the boxes' lanes
      const int qr = lane - 2 * per;
      if (with_q && qr >= 0 && qr < c.nrows)
        bulk_copy_g2s(st + St::kQOff + qr * ROW, qbase + ((size_t)(c.lo + R * c.c + qr) * H + c.h) * ROW, ROW, bar);
    } else {
      // a tail tile: plain K and V rows by 1-D bulk copies (lane 2 c2 the K
      // rows of segment c2, lane 2 c2 + 1 its V rows: copies issued from one
      // lane queue behind one another), the query rows from lane 2 nsv
      const int nsv = min(nseg, (nvalid + seg - 1) / seg);
      if (lane == 0) mbar_arrive_expect_tx(bar, (with_q ? c.nrows * ROW : 0u) + 2u * nsv * seg * ROW);
      __syncwarp();
      if (lane < 2 * nsv) {
        const int c2 = lane >> 1, isv = lane & 1;
        const int t = t0 + c2 * seg;
        const size_t off = (((size_t)my_bt[t / bs - bt_j0] * p.num_kv_heads + c.kvh) * bs + (t % bs)) * ROW;
        bulk_copy_g2s(st + isv * St::kTensorBytes + c2 * seg * ROW, (isv ? vbase : kbase) + off, seg * ROW, bar);
      } else if (lane == 2 * nsv && with_q) {
        bulk_copy_g2s(st + St::kQOff, qbase + ((size_t)(c.lo + c.j) * H + (size_t)c.hg * c.nrows) * ROW,
                      c.nrows * ROW, bar);
      }
    }
  };

  int issued = 0;
  for (; issued < ST && ci.g < a_end; ++issued) {
    issue(ci, issued);
    scursor_next(ci, x, NG);
  }

  // prefix state (tensor-core layout, see mma_prefix_tile) and tail state
  uint32_t qb[D / 16][2];
  float acc[D / 16][4];
  float tm[2] = {-INFINITY, -INFINITY}, tl[2] = {0.f, 0.f};
  float qf[TG][DPL];
  float m[TG], l[TG], o[TG][DPL];
  bool visit_from_start = true;
  // the prefix results in pbuf: group, head group and the members (bits)
  // whose rows meet their tails there
  int pb_grp = -1, pb_hg = -1;
  unsigned pb_local = 0u;

  // Second part of a row to arrive: merge with the other part's stored
  // result and write the output. `mine` is this part's row in shared memory.
  auto write_out = [&](size_t row, const float* mine, float om, float ol, const float* other_o, float other_m,
                       float other_l, bool other_global) {
    float a[DL], b[DL], r[DL];
#pragma unroll
    for (int e = 0; e < DL; ++e) {
      a[e] = mine[lane * DL + e];
      b[e] = other_global ? __ldcg(other_o + lane * DL + e) : other_o[lane * DL + e];
    }
    lse_combine<DL>(om, ol, a, other_m, other_l, b, r);
    T* orow = static_cast<T*>(p.out) + row * D + lane * DL;
#pragma unroll
    for (int e = 0; e < DL; ++e) store_elem(orow + e, r[e]);
  };

  // The prefix part of rows [0, nr) of segment c is complete in pbuf.
  auto complete_prefix = [&](const SCursor& c, bool whole) {
    unsigned local = 0u;
    if (whole && x.gpw == 1 && c.nch == 1) {
      // member k's tail ends at unit c.g + sum_{i <= k} (charge + tiles_i):
      // its row stays local when that is still inside this warp's range
      // member k's tail: its last tile starts at c.g + kUnitP - kUnitT +
      // sum_{i <= k} (kChargeT + kUnitT tiles_i); the row stays local when
      // that tile is still inside this warp's range
      long long u = lane < c.M ? (long long)tiles_of(ctx_len(x, c.lo + lane) - c.S) * kUnitT + kChargeT : 0;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const long long y = __shfl_up_sync(kFullMask, u, o2);
        if (lane >= o2) u += y;
      }
      local = __ballot_sync(kFullMask, lane < c.M && c.g + kUnitP - kUnitT + u <= a_end - 1);
      pb_grp = c.grp;
      pb_hg = c.hg;
    } else {
      pb_grp = -1;
    }
    pb_local = local;
    const int nr = c.nrows;
    // rows that do not stay local: publish, count, merge when second
    unsigned pub = __ballot_sync(kFullMask, lane < nr && !((local >> lane) & 1u)) & ((1u << nr) - 1u);
    if (pub == 0u) return;
    for (unsigned q = pub; q; q &= q - 1) {
      const int r = __ffs(q) - 1;
      const size_t row = (size_t)(c.lo + R * c.c + r) * H + c.h;
      const float* src = pbuf + r * RF;
#pragma unroll
      for (int e = 0; e < DL; ++e) gp.ws_row_o[row * D + lane * DL + e] = src[lane * DL + e];
      if (lane == 0) gp.ws_row_ml[row] = make_float2(src[D], src[D + 1]);
    }
    __syncwarp();  // the rows' stores precede the releases below
    int prev = 0;
    if ((pub >> lane) & 1u) {
      const size_t row = (size_t)(c.lo + R * c.c + lane) * H + c.h;
      prev = atomic_add_acq_rel_gpu(gp.ws_row_ctr + row, 1);
      if (prev == 1) gp.ws_row_ctr[row] = 0;
    }
    const unsigned second = __ballot_sync(kFullMask, prev == 1);
    __syncwarp();
    for (unsigned q = second; q; q &= q - 1) {
      const int r = __ffs(q) - 1;
      const size_t row = (size_t)(c.lo + R * c.c + r) * H + c.h;
      const float* src = pbuf + r * RF;
      const float2 tml = __ldcg(gp.ws_tail_ml + row);
      write_out(row, src, src[D], src[D + 1], gp.ws_tail_o + row * D, tml.x, tml.y, true);
    }
  };

  // The tail part of rows [0, gpw) of segment c is complete in tbuf.
  auto complete_tail = [&](const SCursor& c, bool whole) {
    const int s = c.lo + c.j;
    const int nr = c.nrows;
    if (c.S == 0) {  // no shared prefix: the tail is the whole row
      for (int r = 0; r < nr; ++r) {
        const size_t row = (size_t)s * H + (size_t)c.hg * nr + r;
        const float* src = tbuf + r * RF;
        T* orow = static_cast<T*>(p.out) + row * D + lane * DL;
#pragma unroll
        for (int e = 0; e < DL; ++e) store_elem(orow + e, src[lane * DL + e]);
      }
      return;
    }
    if (whole && pb_grp == c.grp && pb_hg == c.hg && ((pb_local >> c.j) & 1u)) {
      // the prefix result waits in this warp's buffer (gpw 1, one row chunk)
      const size_t row = (size_t)s * H + c.hg;
      const float* src = tbuf;
      const float* pre = pbuf + c.j * RF;
      write_out(row, src, src[D], src[D + 1], pre, pre[D], pre[D + 1], false);
      return;
    }
    for (int r = 0; r < nr; ++r) {
      const size_t row = (size_t)s * H + (size_t)c.hg * nr + r;
      const float* src = tbuf + r * RF;
#pragma unroll
      for (int e = 0; e < DL; ++e) gp.ws_tail_o[row * D + lane * DL + e] = src[lane * DL + e];
      if (lane == 0) gp.ws_tail_ml[row] = make_float2(src[D], src[D + 1]);
    }
    __syncwarp();
    int prev = 0;
    if (lane < nr) {
      const size_t row = (size_t)s * H + (size_t)c.hg * nr + lane;
      prev = atomic_add_acq_rel_gpu(gp.ws_row_ctr + row, 1);
      if (prev == 1) gp.ws_row_ctr[row] = 0;
    }
    const unsigned second = __ballot_sync(kFullMask, prev == 1);
    __syncwarp();
    for (unsigned q = second; q; q &= q - 1) {
      const int r = __ffs(q) - 1;
      const size_t row = (size_t)s * H + (size_t)c.hg * nr + r;
      const float* src = tbuf + r * RF;
      const float2 pml = __ldcg(gp.ws_row_ml + row);
      write_out(row, src, src[D], src[D + 1], gp.ws_row_o + row * D, pml.x, pml.y, true);
    }
  };

  for (int ring = 0; cc.g < a_end; ++ring) {
    if (!__all_sync(kFullMask, mbar_wait_bounded(my_bars + (ring % ST), (ring / ST) & 1, p.wait_limit_ns))) {
      if (lane == 0) set_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
      for (int k2 = ring; k2 < issued; ++k2) mbar_wait_bounded(my_bars + (k2 % ST), (k2 / ST) & 1, kDrainLimitNs);
      return;  // outputs of this call are not valid
    }
    const unsigned char* ks = my_ring + (ring % ST) * S::kStageBytes;
    const int t0 = cc.tok0 + cc.t * kTileTokens;
    const int nvalid = min(max(cc.tok_end - t0, 0), kTileTokens);
    const bool first = cc.t == 0 || cc.g == g_first;
    const bool last = cc.t == cc.nt - 1 || cc.g + sunit(cc.part) >= a_end;
    const int nr = cc.nrows;

    if (cc.part == 0) {
      if (first) {
        visit_from_start = cc.t == 0;
        tm[0] = tm[1] = -INFINITY;
        tl[0] = tl[1] = 0.f;
#pragma unroll
        for (int mb = 0; mb < D / 16; ++mb) acc[mb][0] = acc[mb][1] = acc[mb][2] = acc[mb][3] = 0.f;
        // B fragments of Q^T: lane 4g + t holds query row g, dims 16 k + 2t,
        // +1 and 16 k + 2t + 8, +9 (rows past nr: zero)
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(ks + St::kQOff + mg * ROW);
#pragma unroll
        for (int k2 = 0; k2 < D / 16; ++k2) {
          qb[k2][0] = mg < nr ? qrow[8 * k2 + mt] : 0u;
          qb[k2][1] = mg < nr ? qrow[8 * k2 + mt + 4] : 0u;
        }
      }
      mma_prefix_tile<T, D>(smem_u32(ks), qb, acc, tm, tl, p.scale_log2);
    } else {
      if (first) {
        visit_from_start = cc.t == 0;
#pragma unroll
        for (int g = 0; g < TG; ++g) {
          m[g] = -INFINITY;
          l[g] = 0.f;
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[g][e] = 0.f;
        }
        if (nvalid > 0) {
#pragma unroll
          for (int g = 0; g < TG; ++g) {
            const uint4* qrow = reinterpret_cast<const uint4*>(ks + St::kQOff + g * ROW);
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
      if (nvalid > 0) core_tile<T, D, TG, TG, false, TG>(ks, ks + St::kTensorBytes, qf, o, m, l, nvalid, TG);
    }
    __syncwarp();
    if (ci.g < a_end) {
      issue(ci, issued++);
      scursor_next(ci, x, NG);
    }

    if (last) {
      // ---- end of this warp's visit of the segment under cc ------------------
      const bool whole = visit_from_start && cc.t == cc.nt - 1;
      float* rows_buf = cc.part == 0 ? pbuf : tbuf;
      if (cc.part == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          tl[e] += __shfl_xor_sync(kFullMask, tl[e], 4);
          tl[e] += __shfl_xor_sync(kFullMask, tl[e], 8);
          tl[e] += __shfl_xor_sync(kFullMask, tl[e], 16);
        }
      } else {
#pragma unroll
        for (int g = 0; g < TG; ++g) {
          l[g] += __shfl_xor_sync(kFullMask, l[g], 8);
          l[g] += __shfl_xor_sync(kFullMask, l[g], 16);
#pragma unroll
          for (int e = 0; e < DPL; ++e) {
            o[g][e] += __shfl_xor_sync(kFullMask, o[g][e], 8);
            o[g][e] += __shfl_xor_sync(kFullMask, o[g][e], 16);
          }
        }
      }
      // this warp's (m, l, o / l) of the segment's rows: into the row buffer
      // (whole segment) or into a partial slot (one piece)
      const int slot = cc.g - (long long)cc.t * sunit(cc.part) - scharge(cc.part) <= a_begin ? 0 : 1;
      const size_t base = ((size_t)wid * 2 + slot) * R;
      float* o_dst = whole ? rows_buf : p.ws_o + base * D;
      const int o_stride = whole ? RF : D;
      if (cc.part == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = 2 * mt + e;
          if (r < nr) {
            const float inv = 1.f / tl[e];
            float* orow = o_dst + r * o_stride + mg;
#pragma unroll
            for (int mb = 0; mb < D / 16; ++mb) {
              orow[16 * mb] = acc[mb][e] * inv;
              orow[16 * mb + 8] = acc[mb][e + 2] * inv;
            }
            if (mg == 0) {
              if (whole) {
                rows_buf[r * RF + D] = tm[e];
                rows_buf[r * RF + D + 1] = tl[e];
              } else {
                p.ws_ml[base + r] = make_float2(tm[e], tl[e]);
              }
            }
          }
        }
      } else {
#pragma unroll
        for (int g = 0; g < TG; ++g) {
          const float inv = l[g] > 0.f ? 1.f / l[g] : 0.f;
          if (grp == 0) {
            float* orow = o_dst + g * o_stride;
#pragma unroll
            for (int k = 0; k < CPL; ++k)
#pragma unroll
              for (int e = 0; e < VEC; ++e) orow[(sub + 8 * k) * VEC + e] = o[g][k * VEC + e] * inv;
          }
          if (lane == 0) {
            if (whole) {
              rows_buf[g * RF + D] = m[g];
              rows_buf[g * RF + D + 1] = l[g];
            } else {
              p.ws_ml[base + g] = make_float2(m[g], l[g]);
            }
          }
        }
      }
      __syncwarp();  // the rows (shared) or the partial (global, before the release below)
      bool done = whole;
      if (!whole) {
        // one piece of a segment shared with neighbouring warps: the last
        // piece to arrive merges all pieces into the row buffer
        // the warps holding the first units of the segment's first and last tiles
        const long long seg_start = cc.g - (long long)cc.t * sunit(cc.part);
        const long long seg_last = seg_start + (long long)(cc.nt - 1) * sunit(cc.part);
        const long long seg_units0 = seg_start - scharge(cc.part);
        const long long w_first = ((seg_start + 1) * Weff + Ttot - 1) / Ttot - 1;
        const long long w_last = ((seg_last + 1) * Weff + Ttot - 1) / Ttot - 1;
        int is_last = 0;
        if (lane == 0) {
          const size_t ci_idx = cc.part == 0 ? (size_t)(cc.lo + R * cc.c) * H + cc.h
                                             : (size_t)x.num_seqs * H + (size_t)(cc.lo + cc.j) * HG + cc.hg;
          int32_t* ctr = gp.ws_seg_ctr + ci_idx;
          const int prev = atomic_add_acq_rel_gpu(ctr, 1);
          is_last = prev == (int)(w_last - w_first);
          if (is_last) *ctr = 0;
        }
        is_last = __shfl_sync(kFullMask, is_last, 0);
        if (is_last) {
          __syncwarp();
          // kMergeRows rows at a time, their pieces' loads in flight together;
          // each piece folds in by the running-maximum rule
          for (int r0 = 0; r0 < nr; r0 += kMergeRows) {
            float Mx[kMergeRows], Ls[kMergeRows], O[kMergeRows][DL];
#pragma unroll
            for (int i = 0; i < kMergeRows; ++i) {
              Mx[i] = -INFINITY;
              Ls[i] = 0.f;
#pragma unroll
              for (int e = 0; e < DL; ++e) O[i][e] = 0.f;
            }
            for (long long w = w_first; w <= w_last; ++w) {
              const int sl = (w == w_first && w * Ttot / Weff < seg_units0) ? 1 : 0;
              const size_t idx0 = ((size_t)w * 2 + sl) * R + r0;
              float2 v[kMergeRows];
              float ov[kMergeRows][DL];
#pragma unroll
              for (int i = 0; i < kMergeRows; ++i) {
                v[i] = make_float2(-INFINITY, 0.f);
                if (r0 + i < nr) {
                  v[i] = __ldcg(p.ws_ml + idx0 + i);
#pragma unroll
                  for (int e = 0; e < DL; ++e) ov[i][e] = __ldcg(p.ws_o + (idx0 + i) * D + lane * DL + e);
                }
              }
#pragma unroll
              for (int i = 0; i < kMergeRows; ++i) {
                if (v[i].x != -INFINITY) {  // an empty piece adds nothing
                  const float Mn = fmaxf(Mx[i], v[i].x);
                  const float a = exp2f(Mx[i] - Mn);  // 0 while nothing was folded in
                  const float b = v[i].y * exp2f(v[i].x - Mn);
                  Ls[i] = Ls[i] * a + b;
#pragma unroll
                  for (int e = 0; e < DL; ++e) O[i][e] = O[i][e] * a + ov[i][e] * b;
                  Mx[i] = Mn;
                }
              }
            }
#pragma unroll
            for (int i = 0; i < kMergeRows; ++i) {
              if (r0 + i < nr) {
                float* dst = rows_buf + (r0 + i) * RF;
                const float inv = Ls[i] > 0.f ? 1.f / Ls[i] : 0.f;
#pragma unroll
                for (int e = 0; e < DL; ++e) dst[lane * DL + e] = O[i][e] * inv;
                if (lane == 0) {
                  dst[D] = Mx[i];
                  dst[D + 1] = Ls[i];
                }
              }
            }
          }
          __syncwarp();
          done = true;
        }
      }
      if (done) {
        if (cc.part == 0)
          complete_prefix(cc, whole);
        else
          complete_tail(cc, whole);
      }
    }
    scursor_next(cc, x, NG);
  }
}

// Persistent grid of one phase kernel on the current device (cached).
template <typename T, int D, int TG, int PH, int NW>
cudaError_t grouped_grid(int& grid) {
  using S = GroupedShape<T, D, NW, PH>;
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

// Launch of a phase kernel as a programmatic dependent of the kernel before
// it in the stream: its launch overlaps that kernel, and it waits for that
// kernel's results at griddepcontrol.wait.
template <typename T, int D, int TG, int PH, int NW>
cudaError_t launch_phase(int grid, const CUtensorMap& kmap, const CUtensorMap& vmap, const GroupedParams& gp,
                         cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = GroupedShape<T, D, NW, PH>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, pa_decode_grouped_kernel<T, D, TG, PH, NW>, kmap, vmap, gp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Persistent grid of the single-launch kernel on the current device (cached).
template <typename T, int D, int TG>
cudaError_t shared_grid(int& grid) {
  using S = SharedShape<D, kSharedWarps>;
  static int grid_of_device[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  grid = (dev >= 0 && dev < 64) ? __atomic_load_n(&grid_of_device[dev], __ATOMIC_ACQUIRE) : 0;
  if (grid != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(pa_decode_shared_kernel<T, D, TG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           S::kSmemBytes);
  if (e != cudaSuccess) return e;
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pa_decode_shared_kernel<T, D, TG>,
                                                    kSharedWarps * 32, S::kSmemBytes);
  if (e != cudaSuccess) return e;
  grid = sms * (per_sm > 0 ? per_sm : 1);
  if (grid > kMaxDecodeWarps / kSharedWarps) grid = kMaxDecodeWarps / kSharedWarps;
  if (dev >= 0 && dev < 64) __atomic_store_n(&grid_of_device[dev], grid, __ATOMIC_RELEASE);
  return cudaSuccess;
}

// Validation prologue, then the work as a programmatic dependent of it: for
// 16-bit data one single-launch kernel (the pools' tensor maps, boxes of
// {64, min(block_size, 16)} rows, feed its prefix tiles); for fp32 data the
// prefix phase and then the tail phase.
template <typename T, int D, int TG>
cudaError_t launch_pa_decode_grouped(const GroupedParams& gp, cudaStream_t stream) {
  CUtensorMap kmap, vmap;
  memset(&kmap, 0, sizeof(kmap));
  memset(&vmap, 0, sizeof(vmap));
  int pro = (gp.num_groups + 7) / 8;
  pro = pro < 1 ? 1 : (pro > 4096 ? 4096 : pro);
  if constexpr (Mma16816<T>::kOk) {
    int grid = 0;
    cudaError_t e = shared_grid<T, D, TG>(grid);
    if (e != cudaSuccess) return e;
    const DecodeParams& p = gp.base;
    const uint64_t rows = (uint64_t)p.num_blocks * p.num_kv_heads * p.block_size;
    const int box_rows = p.block_size < kTileTokens ? p.block_size : kTileTokens;
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    e = encode_pool_rows_map(&kmap, p.k_cache, rows, D, box_rows, bf16);
    if (e != cudaSuccess) return e;
    e = encode_pool_rows_map(&vmap, p.v_cache, rows, D, box_rows, bf16);
    if (e != cudaSuccess) return e;
    pa_group_prologue_kernel<T><<<pro, 256, 0, stream>>>(gp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSharedWarps * 32);
    cfg.dynamicSmemBytes = SharedShape<D, kSharedWarps>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, pa_decode_shared_kernel<T, D, TG>, kmap, vmap, gp);
    return e != cudaSuccess ? e : cudaGetLastError();
  } else {
    constexpr int NW0 = grouped_warps<T, 0>(), NW1 = grouped_warps<T, 1>();
    int grid0 = 0, grid1 = 0;
    cudaError_t e = grouped_grid<T, D, TG, 0, NW0>(grid0);
    if (e != cudaSuccess) return e;
    e = grouped_grid<T, D, TG, 1, NW1>(grid1);
    if (e != cudaSuccess) return e;
    pa_group_prologue_kernel<T><<<pro, 256, 0, stream>>>(gp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_phase<T, D, TG, 0, NW0>(grid0, kmap, vmap, gp, stream);
    if (e != cudaSuccess) return e;
    return launch_phase<T, D, TG, 1, NW1>(grid1, kmap, vmap, gp, stream);
  }
}

using GroupedLauncher = cudaError_t (*)(const GroupedParams&, cudaStream_t);

// gpw_index: query heads per warp in the tails, 0 -> 1, 1 -> 2, 2 -> 4.
GroupedLauncher grouped_launcher_f32(int head_dim, int gpw_index);
GroupedLauncher grouped_launcher_f16(int head_dim, int gpw_index);
GroupedLauncher grouped_launcher_bf16(int head_dim, int gpw_index);

}  // namespace pkv
