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
// A row (s, h) whose sequence has a shared prefix gets two results — the
// prefix segment's and the tail segment's — which the second to arrive
// merges (log-sum-exp) into the output. Pieces of a segment cut by warp
// range boundaries are first merged as in the plain kernel.
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

struct GroupedParams {
  DecodeParams base;             // ws_counter is unused here
  const int32_t* group_start;    // [num_groups + 1]
  const int32_t* shared_blocks;  // [num_groups]
  int num_groups;
  int32_t* ws_flag;     // [1] 1 = grouping rejected
  int32_t* ws_group_S;  // [num_groups] usable shared prefix tokens
  int32_t* ws_seq_P;    // [num_seqs] prefix tokens of the sequence's group
  int32_t* ws_seg_ctr;  // [2][num_seqs * num_heads] piece counters (prefix, tail)
  int32_t* ws_row_ctr;  // [num_seqs * num_heads] prefix + tail arrivals
  float2* ws_row_ml;    // [num_seqs * num_heads][2] (m, l) of the prefix / tail result
  float* ws_row_o;      // [num_seqs * num_heads][2][head_dim] o / l
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
      for (int j = lane; j < sb; j += 32) {
        const int32_t id0 = __ldg(row0 + j);
        for (int s = lo + 1; s < hi; ++s)
          if (__ldg(p.block_tables + (size_t)s * MB + j) != id0) {
            first_bad = min(first_bad, j);
            break;
          }
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

// Prefix tiles of group g (0 when it has no usable shared prefix).
__device__ __forceinline__ long long prefix_tiles(const GCtx& x, int g) {
  if (!x.use_groups) return 0;
  const int M = __ldg(x.group_start + g + 1) - __ldg(x.group_start + g);
  const int S = x.group_S[g];
  if (M < 2 || S <= 0) return 0;
  return (long long)x.num_heads * group_rows(M) * (S / kTileTokens);
}

__device__ __forceinline__ int seq_prefix(const GCtx& x, int s) { return x.use_groups ? x.seq_P[s] : 0; }

__device__ __forceinline__ void gseg_enter(GCursor& c, const GCtx& x) {
  if (c.part == 0) {
    c.lo = __ldg(x.group_start + c.a);
    c.M = __ldg(x.group_start + c.a + 1) - c.lo;
    c.tok0 = 0;
    c.tok_end = x.group_S[c.a];
    c.sbt = c.lo;
    c.kvh = c.b / x.group;
    c.nrows = min(kGroupRows, c.M - kGroupRows * c.c);
    c.nt = c.tok_end / kTileTokens;
  } else {
    const int L = ctx_len(x, c.a);
    c.tok0 = seq_prefix(x, c.a);
    c.tok_end = L;
    c.sbt = c.a;
    c.kvh = (c.b * x.gpw) / x.group;
    c.nrows = x.gpw;
    c.nt = tiles_of(L - c.tok0);
  }
}

// Move to the first group at or after c.a with prefix tiles; else to the tails.
__device__ __forceinline__ void gseek_prefix(GCursor& c, const GCtx& x) {
  while (c.a < x.num_groups && prefix_tiles(x, c.a) == 0) ++c.a;
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

__device__ __forceinline__ void gcursor_next(GCursor& c, const GCtx& x) {
  ++c.g;
  if (++c.t < c.nt) return;
  c.t = 0;
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

// (sequence, head) of row r of the segment under c.
__device__ __forceinline__ int row_seq(const GCursor& c, int r) { return c.part == 0 ? c.lo + kGroupRows * c.c + r : c.a; }
__device__ __forceinline__ int row_head(const GCursor& c, const GCtx& x, int r) {
  return c.part == 0 ? c.b : c.b * x.gpw + r;
}

// Second-level merge of row (seq, head): the caller has deposited its
// result (m, l, o/l) in the row's slot for its part; the second of the two
// results to arrive merges both and writes the output.
template <typename T, int D>
__device__ __forceinline__ void row_merge_tail(const GroupedParams& gp, int seq, int head) {
  const DecodeParams& p = gp.base;
  const int lane = threadIdx.x & 31;
  const size_t row = (size_t)seq * p.num_heads + head;
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    const int prev = atomicAdd(gp.ws_row_ctr + row, 1);
    last = prev == 1;
    if (last) gp.ws_row_ctr[row] = 0;
  }
  last = __shfl_sync(kFullMask, last, 0);
  if (!last) return;
  __threadfence();
  constexpr int DL = D / 32;
  const float2 a = __ldcg(gp.ws_row_ml + row * 2), b = __ldcg(gp.ws_row_ml + row * 2 + 1);
  const float M = fmaxf(a.x, b.x);
  const float wa = a.x == -INFINITY ? 0.f : a.y * exp2f(a.x - M);
  const float wb = b.x == -INFINITY ? 0.f : b.y * exp2f(b.x - M);
  const float inv = 1.f / (wa + wb);
  const float* oa = gp.ws_row_o + (row * 2) * D + lane * DL;
  const float* ob = gp.ws_row_o + (row * 2 + 1) * D + lane * DL;
  T* orow = static_cast<T*>(p.out) + row * D + lane * DL;
#pragma unroll
  for (int e = 0; e < DL; ++e) store_elem(orow + e, (__ldcg(oa + e) * wa + __ldcg(ob + e) * wb) * inv);
}

template <typename T, int D>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    pa_decode_grouped_kernel(const GroupedParams gp) {
  using S = DecodeShape<T, D, kGroupRows>;
  constexpr int NW = kDecodeWarps;
  constexpr int R = kGroupRows;
  constexpr int ST = S::kStages;
  constexpr int DPL = S::kDimsPerLane;
  constexpr int CPL = S::kChunksPerLane;
  constexpr int VEC = S::kVec;
  constexpr int ROW = S::kRowBytes;
  const DecodeParams& p = gp.base;

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  long long* scan = reinterpret_cast<long long*>(smem + S::kScanOff);
  longlong2* starts = reinterpret_cast<longlong2*>(smem + S::kStartOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = lane >> 3;
  const int sub = lane & 7;
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
  const int B = p.num_seqs, G = gp.num_groups, HG = p.head_groups;

  // ---- start-up: tiles of both parts, then each warp's first segment --------
  long long mine = 0;
  for (int g = threadIdx.x; g < G; g += NW * 32) mine += prefix_tiles(x, g);
  long long TA;
  block_exclusive_scan(mine, scan, TA);
  mine = 0;
  for (int s = threadIdx.x; s < B; s += NW * 32)
    mine += (long long)HG * tiles_of(ctx_len(x, s) - seq_prefix(x, s));
  long long TB;
  block_exclusive_scan(mine, scan, TB);
  const long long Ttot = TA + TB;
  const long long W = (long long)gridDim.x * NW;
  const long long Weff = W < Ttot ? W : Ttot;
  const long long wid = (long long)blockIdx.x * NW + warp;
  const long long a_begin = wid < Weff ? wid * Ttot / Weff : Ttot;
  const long long a_end = wid < Weff ? (wid + 1) * Ttot / Weff : Ttot;
  if (threadIdx.x < NW) starts[threadIdx.x] = make_longlong2(-1, 0);
  __syncthreads();
  // starts[i].x: group (prefix part) or B + sequence (tail part); .y: offset in it
  long long carry = 0;
  for (int base = 0; base < G; base += NW * 32) {
    const int g = base + threadIdx.x;
    const long long cnt = g < G ? prefix_tiles(x, g) : 0;
    long long tot;
    const long long excl = carry + block_exclusive_scan(cnt, scan, tot);
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const long long w = (long long)blockIdx.x * NW + i;
      if (w < Weff) {
        const long long a = w * Ttot / Weff;
        if (cnt > 0 && a >= excl && a < excl + cnt) starts[i] = make_longlong2(g, a - excl);
      }
    }
    carry += tot;
  }
  carry = TA;
  for (int base = 0; base < B; base += NW * 32) {
    const int s = base + threadIdx.x;
    const long long cnt =
        s < B ? (long long)HG * tiles_of(ctx_len(x, s) - seq_prefix(x, s)) : 0;
    long long tot;
    const long long excl = carry + block_exclusive_scan(cnt, scan, tot);
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const long long w = (long long)blockIdx.x * NW + i;
      if (w < Weff) {
        const long long a = w * Ttot / Weff;
        if (cnt > 0 && a >= excl && a < excl + cnt) starts[i] = make_longlong2((long long)G + s, a - excl);
      }
    }
    carry += tot;
  }
  __syncthreads();
  if (a_begin >= a_end) return;  // idle warp; no block barrier follows

  unsigned char* my_ring = smem + warp * ST * S::kStageBytes;
  uint64_t* my_bars = bars + warp * ST;
  int32_t* my_bt = reinterpret_cast<int32_t*>(smem + S::kBtOff) + warp * kBtChunk;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < ST; ++i) mbar_init(&my_bars[i], 1);
    mbar_init_fence();
  }
  __syncwarp();

  GCursor ci;
  {
    const longlong2 st0 = starts[warp];
    ci.g = a_begin;
    ci.c = 0;
    if (st0.x < G) {
      ci.part = 0;
      ci.a = static_cast<int>(st0.x);
      ci.b = 0;
      gseg_enter(ci, x);  // sets M and nt (nt does not depend on b or c)
      const long long per_seg = ci.nt;
      const long long seg = st0.y / per_seg;
      ci.t = static_cast<int>(st0.y % per_seg);
      ci.b = static_cast<int>(seg / group_rows(ci.M));
      ci.c = static_cast<int>(seg % group_rows(ci.M));
      gseg_enter(ci, x);
    } else {
      ci.part = 1;
      ci.a = static_cast<int>(st0.x - G);
      ci.b = 0;
      gseg_enter(ci, x);
      ci.b = static_cast<int>(st0.y / ci.nt);
      ci.t = static_cast<int>(st0.y % ci.nt);
      gseg_enter(ci, x);
    }
  }
  GCursor cc = ci;
  int bt_s = -1, bt_j0 = 0;

  const char* kbase = static_cast<const char*>(p.k_cache);
  const char* vbase = static_cast<const char*>(p.v_cache);
  const char* qbase = static_cast<const char*>(p.q);
  const int seg = bs < kTileTokens ? bs : kTileTokens;
  const int nseg = kTileTokens / seg;
  const int H = p.num_heads;

  auto issue = [&](const GCursor& c, int n) {
    const int t0 = c.tok0 + c.t * kTileTokens;
    const int nvalid = min(max(c.tok_end - t0, 0), kTileTokens);
    const bool with_q = (c.t == 0 || c.g == a_begin) && nvalid > 0;
    if (nvalid > 0) {
      const int j_first = t0 / bs;
      const int j_last = (t0 + nvalid - 1) / bs;
      if (c.sbt != bt_s || j_first < bt_j0 || j_last >= bt_j0 + kBtChunk) {
        const int nblk = (c.tok_end + bs - 1) / bs;
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

  int issued = 0;
  for (; issued < ST && ci.g < a_end; ++issued) {
    issue(ci, issued);
    gcursor_next(ci, x);
  }

  float qf[R][DPL];
  float m[R], l[R], o[R][DPL];
  bool visit_from_start = true;

  for (int n = 0; cc.g < a_end; ++n) {
    if (!__all_sync(kFullMask, mbar_wait_bounded(my_bars + (n % ST), (n / ST) & 1, p.wait_limit_ns))) {
      if (lane == 0) set_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
      for (int k2 = n; k2 < issued; ++k2) mbar_wait_bounded(my_bars + (k2 % ST), (k2 / ST) & 1, kDrainLimitNs);
      return;
    }
    const unsigned char* ks = my_ring + (n % ST) * S::kStageBytes;
    const unsigned char* vs = ks + S::kTileBytes;
    const int t0 = cc.tok0 + cc.t * kTileTokens;
    const int nvalid = min(max(cc.tok_end - t0, 0), kTileTokens);
    const bool first = cc.t == 0 || cc.g == a_begin;
    const bool last = cc.t == cc.nt - 1 || cc.g == a_end - 1;
    const int nr = cc.nrows;

    if (first) {
      visit_from_start = cc.t == 0;
#pragma unroll
      for (int g = 0; g < R; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[g][e] = 0.f;
      }
      if (nvalid > 0) {
        const unsigned char* qs = ks + 2 * S::kTileBytes;
#pragma unroll
        for (int g = 0; g < R; ++g) {
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

    if (nvalid > 0) {
      float x4[R][4];
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int r = it * 4 + grp;
        const uint4* krow = reinterpret_cast<const uint4*>(ks + r * ROW);
        float acc[R];
#pragma unroll
        for (int g = 0; g < R; ++g) acc[g] = 0.f;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          float f[VEC];
          Chunk<T>::widen(krow[sub + 8 * k], f);
#pragma unroll
          for (int g = 0; g < R; ++g)
            if (g < nr) {
#pragma unroll
              for (int e = 0; e < VEC; ++e) acc[g] = fmaf(qf[g][k * VEC + e], f[e], acc[g]);
            }
        }
#pragma unroll
        for (int g = 0; g < R; ++g)
          if (g < nr) {
            float a = acc[g];
            a += __shfl_xor_sync(kFullMask, a, 1);
            a += __shfl_xor_sync(kFullMask, a, 2);
            a += __shfl_xor_sync(kFullMask, a, 4);
            x4[g][it] = r < nvalid ? a : -INFINITY;
          }
      }
      float pw[R][4];
#pragma unroll
      for (int g = 0; g < R; ++g)
        if (g < nr) {
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
          for (int e = 0; e < DPL; ++e) o[g][e] *= alpha;
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
            for (int g = 0; g < R; ++g)
              if (g < nr) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[g][k * VEC + e] = fmaf(pw[g][it], f[e], o[g][k * VEC + e]);
              }
          }
        }
      }
    }
    __syncwarp();
    if (ci.g < a_end) {
      issue(ci, issued++);
      gcursor_next(ci, x);
    }

    if (last) {
#pragma unroll
      for (int g = 0; g < R; ++g)
        if (g < nr) {
          l[g] += __shfl_xor_sync(kFullMask, l[g], 8);
          l[g] += __shfl_xor_sync(kFullMask, l[g], 16);
#pragma unroll
          for (int e = 0; e < DPL; ++e) {
            o[g][e] += __shfl_xor_sync(kFullMask, o[g][e], 8);
            o[g][e] += __shfl_xor_sync(kFullMask, o[g][e], 16);
          }
        }
      // a row has two results when its sequence has a shared prefix
      const bool two_source = cc.part == 0 || cc.tok0 > 0;
      if (visit_from_start && cc.t == cc.nt - 1) {
#pragma unroll
        for (int g = 0; g < R; ++g) {
          if (g >= nr) continue;
          const int seq = row_seq(cc, g), head = row_head(cc, x, g);
          const size_t row = (size_t)seq * H + head;
          const float inv = l[g] > 0.f ? 1.f / l[g] : 0.f;
          if (!two_source) {
            if (grp == 0) {
              uint4* orow = reinterpret_cast<uint4*>(static_cast<char*>(p.out) + row * ROW);
#pragma unroll
              for (int k = 0; k < CPL; ++k) {
                float f[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) f[e] = o[g][k * VEC + e] * inv;
                orow[sub + 8 * k] = Chunk<T>::narrow(f);
              }
            }
          } else {
            const size_t slot = row * 2 + cc.part;
            if (grp == 0) {
              float4* po = reinterpret_cast<float4*>(gp.ws_row_o + slot * D);
#pragma unroll
              for (int k = 0; k < CPL; ++k)
#pragma unroll
                for (int e = 0; e < VEC; e += 4)
                  po[((sub + 8 * k) * VEC + e) / 4] =
                      make_float4(o[g][k * VEC + e] * inv, o[g][k * VEC + e + 1] * inv,
                                  o[g][k * VEC + e + 2] * inv, o[g][k * VEC + e + 3] * inv);
            }
            if (lane == 0) gp.ws_row_ml[slot] = make_float2(m[g], l[g]);
            row_merge_tail<T, D>(gp, seq, head);
          }
        }
      } else {
        const int slot = cc.g - cc.t <= a_begin ? 0 : 1;
        const size_t base = ((size_t)wid * 2 + slot) * R;
#pragma unroll
        for (int g = 0; g < R; ++g) {
          if (g >= nr) continue;
          const float inv = 1.f / l[g];
          if (grp == 0) {
            float4* po = reinterpret_cast<float4*>(p.ws_o + (base + g) * D);
#pragma unroll
            for (int k = 0; k < CPL; ++k)
#pragma unroll
              for (int e = 0; e < VEC; e += 4)
                po[((sub + 8 * k) * VEC + e) / 4] =
                    make_float4(o[g][k * VEC + e] * inv, o[g][k * VEC + e + 1] * inv,
                                o[g][k * VEC + e + 2] * inv, o[g][k * VEC + e + 3] * inv);
          }
          if (lane == 0) p.ws_ml[base + g] = make_float2(m[g], l[g]);
        }
        __threadfence();
        __syncwarp();
        const long long seg_start = cc.g - cc.t;
        const long long seg_end = seg_start + cc.nt;
        const long long w_first = ((seg_start + 1) * Weff + Ttot - 1) / Ttot - 1;
        const long long w_last = (seg_end * Weff + Ttot - 1) / Ttot - 1;
        int is_last = 0;
        if (lane == 0) {
          const size_t ci_idx = cc.part == 0 ? (size_t)(cc.lo + kGroupRows * cc.c) * H + cc.b
                                             : (size_t)B * H + (size_t)cc.a * HG + cc.b;
          int32_t* ctr = gp.ws_seg_ctr + ci_idx;
          const int prev = atomicAdd(ctr, 1);
          is_last = prev == (int)(w_last - w_first);
          if (is_last) *ctr = 0;
        }
        is_last = __shfl_sync(kFullMask, is_last, 0);
        if (is_last) {
          __threadfence();
          constexpr int DL = D / 32;
          for (int g = 0; g < nr; ++g) {
            float M = -INFINITY;
            for (long long w = w_first; w <= w_last; ++w) {
              const int sl = (w == w_first && w * Ttot / Weff < seg_start) ? 1 : 0;
              M = fmaxf(M, __ldcg(p.ws_ml + ((size_t)w * 2 + sl) * R + g).x);
            }
            float Ls = 0.f, O[DL];
#pragma unroll
            for (int e = 0; e < DL; ++e) O[e] = 0.f;
            for (long long w = w_first; w <= w_last; ++w) {
              const int sl = (w == w_first && w * Ttot / Weff < seg_start) ? 1 : 0;
              const size_t idx = ((size_t)w * 2 + sl) * R + g;
              const float2 v = __ldcg(p.ws_ml + idx);
              const float wt = v.y * exp2f(v.x - M);
              Ls += wt;
              const float* po = p.ws_o + idx * D + lane * DL;
#pragma unroll
              for (int e = 0; e < DL; ++e) O[e] += __ldcg(po + e) * wt;
            }
            const int seq = row_seq(cc, g), head = row_head(cc, x, g);
            const size_t row = (size_t)seq * H + head;
            if (!two_source) {
              T* orow = static_cast<T*>(p.out) + row * D + lane * DL;
#pragma unroll
              for (int e = 0; e < DL; ++e) store_elem(orow + e, O[e] / Ls);
            } else {
              const size_t slot2 = row * 2 + cc.part;
              float* po = gp.ws_row_o + slot2 * D + lane * DL;
#pragma unroll
              for (int e = 0; e < DL; ++e) po[e] = O[e] / Ls;
              if (lane == 0) gp.ws_row_ml[slot2] = make_float2(M, Ls);
              row_merge_tail<T, D>(gp, seq, head);
            }
          }
        }
      }
    }
    gcursor_next(cc, x);
  }
}

// Validation prologue, then the persistent grid sized to the device.
template <typename T, int D>
cudaError_t launch_pa_decode_grouped(const GroupedParams& gp, cudaStream_t stream) {
  using S = DecodeShape<T, D, kGroupRows>;
  static int grid_of_device[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int grid = (dev >= 0 && dev < 64) ? __atomic_load_n(&grid_of_device[dev], __ATOMIC_ACQUIRE) : 0;
  if (grid == 0) {
    e = cudaFuncSetAttribute(pa_decode_grouped_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::kSmemBytes);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pa_decode_grouped_kernel<T, D>,
                                                      kDecodeWarps * 32, S::kSmemBytes);
    if (e != cudaSuccess) return e;
    grid = sms * (per_sm > 0 ? per_sm : 1);
    if (grid > kMaxDecodeWarps / kDecodeWarps) grid = kMaxDecodeWarps / kDecodeWarps;
    if (dev >= 0 && dev < 64) __atomic_store_n(&grid_of_device[dev], grid, __ATOMIC_RELEASE);
  }
  int pro = (gp.num_groups + 7) / 8;
  pro = pro < 1 ? 1 : (pro > 4096 ? 4096 : pro);
  pa_group_prologue_kernel<T><<<pro, 256, 0, stream>>>(gp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pa_decode_grouped_kernel<T, D><<<grid, kDecodeWarps * 32, S::kSmemBytes, stream>>>(gp);
  return cudaGetLastError();
}

using GroupedLauncher = cudaError_t (*)(const GroupedParams&, cudaStream_t);

GroupedLauncher grouped_launcher_f32(int head_dim);
GroupedLauncher grouped_launcher_f16(int head_dim);
GroupedLauncher grouped_launcher_bf16(int head_dim);

}  // namespace pkv
