// Paged decode attention kernel (sm_103a).
//
// Operation ("PagedAttention: the KV cache was the bottleneck all along",
// section "Virtual memory for attention"): one query token per sequence
// attends over its context, whose K/V rows sit in fixed-size blocks scattered
// through a pool and are found through the sequence's block table.
//
// Work decomposition
//   grid.x  kv head x query-head subgroup (GPW query heads share one kv head)
//   grid.y  sequence
//   grid.z  context partition of P tokens (split-context decode); CUDA hands
//           out all partition-0 blocks first, so the last wave holds short
//           partitions only.
//   block   4 warps. A partition is cut into 16-token tiles; warp w takes
//           tiles w, w+4, ... and runs its own pipeline of STAGES shared-memory
//           slots. Lane 0 of the warp issues 1-D bulk copies (cp.async.bulk,
//           completion counted in bytes on an mbarrier) of the tile's K rows
//           and V rows; all lanes wait on the slot's mbarrier (bounded), then
//           compute. No block-wide barrier inside the loop.
//
// Per tile and warp: lanes form 4 groups of 8; group g holds tokens g, g+4,
// g+8, g+12 of the tile and lane i of a group owns 16-byte chunks i, i+8, ...
// of every row (a quarter-warp reads 128 contiguous bytes of one row: no
// shared-memory bank conflicts). q.k partial sums are reduced over the 8
// lanes of a group with shuffles; the running max m, exp-sum l and output o
// are updated with the online softmax in base 2 (q is pre-scaled by
// scale * log2(e)); tokens past the context are masked by select, never by
// multiplication, so poisoned rows never reach the result.
//
// Partitions of one (sequence, head group) write (m, l, o/l) to the workspace;
// the last thread block to finish (atomic counter) merges them with the
// log-sum-exp rule and writes the output, then re-zeroes its counter.
#pragma once

#include "common.cuh"

namespace pkv {

struct DecodeParams {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float scale_log2;  // scale * log2(e)
  int num_heads;
  int num_kv_heads;
  int group;           // num_heads / num_kv_heads
  int head_subgroups;  // group / GPW
  int block_size;
  int max_blocks_per_seq;
  int num_blocks;
  int max_context_len;
  int partition_tokens;  // P
  int max_splits;        // S = ceil(max_context_len / P)
  int32_t* ws_counter;   // [num_seqs * num_heads / GPW]
  float2* ws_ml;         // [num_seqs][num_heads][S]  (m, l)
  float* ws_o;           // [num_seqs][num_heads][S][head_dim]
  int32_t* dev_err;
  uint64_t wait_limit_ns;
};

constexpr int kTileTokens = 16;
constexpr int kDecodeWarps = 4;
constexpr int kMaxSplitBlocks = 64;  // block-table entries of one partition (P / min block_size)

template <typename T, int D>
struct DecodeShape {
  static constexpr int kElemBytes = sizeof(T);
  static constexpr int kRowBytes = D * kElemBytes;
  static constexpr int kTileBytes = kTileTokens * kRowBytes;  // K (or V) rows of one tile
  static constexpr int kStageBytes = 2 * kTileBytes;          // K and V
  static constexpr int kRingBudget = 64 * 1024;
  static constexpr int kStagesRaw = kRingBudget / (kDecodeWarps * kStageBytes);
  static constexpr int kStages = kStagesRaw < 1 ? 1 : (kStagesRaw > 4 ? 4 : kStagesRaw);
  static constexpr int kChunksPerRow = kRowBytes / 16;
  static constexpr int kChunksPerLane = kChunksPerRow / 8;
  static constexpr int kVec = Chunk<T>::kElems;
  static constexpr int kDimsPerLane = kChunksPerLane * kVec;  // = D / 8
  static constexpr int kRingBytes = kDecodeWarps * kStages * kStageBytes;
  static constexpr int kSmemBytes =
      kRingBytes + kDecodeWarps * kStages * 8 + kMaxSplitBlocks * 4 + 16;
  static_assert(kChunksPerRow % 8 == 0, "row must split into 8 lanes of 16-byte chunks");
  static_assert(kDimsPerLane * 8 == D, "lane mapping");
};

template <typename T, int D, int GPW>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    pa_decode_kernel(const DecodeParams p) {
  using S = DecodeShape<T, D>;
  constexpr int NW = kDecodeWarps;
  constexpr int ST = S::kStages;
  constexpr int DPL = S::kDimsPerLane;
  constexpr int CPL = S::kChunksPerLane;
  constexpr int VEC = S::kVec;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kRingBytes);
  int32_t* s_bt = reinterpret_cast<int32_t*>(bars + NW * ST);
  int32_t* s_last = s_bt + kMaxSplitBlocks;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = lane >> 3;  // token sub-index within a 4-row step
  const int sub = lane & 7;   // chunk index within a row
  const int seq = blockIdx.y;
  const int split = blockIdx.z;
  const int kvh = blockIdx.x / p.head_subgroups;
  const int h0 = kvh * p.group + (blockIdx.x % p.head_subgroups) * GPW;
  const int bs = p.block_size;

  // ---- context range of this partition ---------------------------------
  int L = __ldg(p.context_lens + seq);
  const int L_cap = min(p.max_context_len, p.max_blocks_per_seq * bs);
  if (L < 0 || L > L_cap) {
    if (threadIdx.x == 0 && split == 0) set_err(p.dev_err, PKV_DEV_ERR_CONTEXT_LEN);
    L = L < 0 ? 0 : L_cap;
  }
  const int P = p.partition_tokens;
  const int nsplit = L > 0 ? (L + P - 1) / P : 1;
  if (split >= nsplit) return;  // uniform over the block, before any barrier
  const int t_begin = split * P;
  const int t_end = min(L, t_begin + P);
  const int ntiles = (t_end - t_begin + kTileTokens - 1) / kTileTokens;  // 0 iff L == 0
  const int blk0 = t_begin / bs;
  const int nblk = L > 0 ? (t_end + bs - 1) / bs - blk0 : 0;

  // ---- stage the partition's block-table entries in shared memory ------
  const int32_t* bt_row = p.block_tables + (size_t)seq * p.max_blocks_per_seq;
  for (int i = threadIdx.x; i < nblk; i += NW * 32) {
    int id = __ldg(bt_row + blk0 + i);
    if (id < 0 || id >= p.num_blocks) {
      set_err(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
      id = 0;
    }
    s_bt[i] = id;
  }
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < ST; ++s) mbar_init(&bars[warp * ST + s], 1);
    mbar_init_fence();
  }
  __syncthreads();

  const int my_tiles = ntiles > warp ? (ntiles - warp + NW - 1) / NW : 0;
  unsigned char* my_ring = ring + warp * ST * S::kStageBytes;
  uint64_t* my_bars = bars + warp * ST;
  const char* kbase = static_cast<const char*>(p.k_cache);
  const char* vbase = static_cast<const char*>(p.v_cache);
  const int seg = bs < kTileTokens ? bs : kTileTokens;  // rows per bulk copy
  const int nseg = kTileTokens / seg;

  // Lane 0: copy the K rows and V rows of the warp's kt-th tile into slot kt % ST.
  auto issue = [&](int kt) {
    if (kt >= my_tiles) return;
    const int t0 = t_begin + (warp + kt * NW) * kTileTokens;
    unsigned char* kdst = my_ring + (kt % ST) * S::kStageBytes;
    unsigned char* vdst = kdst + S::kTileBytes;
    uint64_t* bar = my_bars + (kt % ST);
    uint32_t bytes = 0;
    for (int c = 0; c < nseg; ++c)
      if (t0 + c * seg < t_end) bytes += 2u * seg * S::kRowBytes;
    mbar_arrive_expect_tx(bar, bytes);
    for (int c = 0; c < nseg; ++c) {
      const int t = t0 + c * seg;
      if (t >= t_end) break;
      const size_t off =
          (((size_t)s_bt[t / bs - blk0] * p.num_kv_heads + kvh) * bs + (t % bs)) * S::kRowBytes;
      bulk_copy_g2s(kdst + c * seg * S::kRowBytes, kbase + off, seg * S::kRowBytes, bar);
      bulk_copy_g2s(vdst + c * seg * S::kRowBytes, vbase + off, seg * S::kRowBytes, bar);
    }
  };
  if (lane == 0)
    for (int kt = 0; kt < ST; ++kt) issue(kt);

  // ---- query rows (fp32, pre-scaled into the base-2 exponent domain) ------
  float qf[GPW][DPL];
#pragma unroll
  for (int g = 0; g < GPW; ++g) {
    const uint4* qrow = reinterpret_cast<const uint4*>(
        static_cast<const char*>(p.q) + ((size_t)seq * p.num_heads + h0 + g) * S::kRowBytes);
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      float f[VEC];
      Chunk<T>::widen(__ldg(qrow + sub + 8 * k), f);
#pragma unroll
      for (int e = 0; e < VEC; ++e) qf[g][k * VEC + e] = f[e] * p.scale_log2;
    }
  }

  float m[GPW], l[GPW], o[GPW][DPL];
#pragma unroll
  for (int g = 0; g < GPW; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[g][e] = 0.f;
  }

  // ---- main loop over this warp's tiles -------------------------------
  bool ok = true;
  int kt = 0;
  for (; kt < my_tiles; ++kt) {
    const bool arrived = mbar_wait_bounded(my_bars + (kt % ST), (kt / ST) & 1, p.wait_limit_ns);
    if (!__all_sync(kFullMask, arrived)) {
      ok = false;
      break;
    }
    const unsigned char* ks = my_ring + (kt % ST) * S::kStageBytes;
    const unsigned char* vs = ks + S::kTileBytes;
    const int t0 = t_begin + (warp + kt * NW) * kTileTokens;
    const int nvalid = min(kTileTokens, t_end - t0);

    // logits of rows grp, grp+4, grp+8, grp+12
    float x[GPW][4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int r = it * 4 + grp;
      const uint4* krow = reinterpret_cast<const uint4*>(ks + r * S::kRowBytes);
      float acc[GPW];
#pragma unroll
      for (int g = 0; g < GPW; ++g) acc[g] = 0.f;
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        float f[VEC];
        Chunk<T>::widen(krow[sub + 8 * k], f);
#pragma unroll
        for (int g = 0; g < GPW; ++g)
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[g] = fmaf(qf[g][k * VEC + e], f[e], acc[g]);
      }
#pragma unroll
      for (int g = 0; g < GPW; ++g) {
        float a = acc[g];
        a += __shfl_xor_sync(kFullMask, a, 1);
        a += __shfl_xor_sync(kFullMask, a, 2);
        a += __shfl_xor_sync(kFullMask, a, 4);
        x[g][it] = r < nvalid ? a : -INFINITY;
      }
    }

    // online softmax update (base 2)
    float pw[GPW][4];
#pragma unroll
    for (int g = 0; g < GPW; ++g) {
      float mt = fmaxf(fmaxf(x[g][0], x[g][1]), fmaxf(x[g][2], x[g][3]));
      mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 8));
      mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 16));
      const float mn = fmaxf(m[g], mt);
      const float alpha = exp2f(m[g] - mn);  // 0 on the first tile (m = -inf)
      float ps = 0.f;
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        pw[g][it] = exp2f(x[g][it] - mn);
        ps += pw[g][it];
      }
      l[g] = l[g] * alpha + ps;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[g][e] *= alpha;
      m[g] = mn;
    }

    // o += p . V over the valid rows (masked rows may hold poison: skip them)
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int r = it * 4 + grp;
      if (r < nvalid) {
        const uint4* vrow = reinterpret_cast<const uint4*>(vs + r * S::kRowBytes);
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          float f[VEC];
          Chunk<T>::widen(vrow[sub + 8 * k], f);
#pragma unroll
          for (int g = 0; g < GPW; ++g)
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[g][k * VEC + e] = fmaf(pw[g][it], f[e], o[g][k * VEC + e]);
        }
      }
    }
    __syncwarp();  // every lane is done with this slot before it is refilled
    if (lane == 0) issue(kt + ST);
  }

  if (!ok) {
    // A wait ran out: report it, then let this warp's copies in flight land
    // (bounded) before the shared memory they target is reused or released.
    if (lane == 0) set_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
    const int issued_end = min(my_tiles, kt + ST);
    for (int k2 = kt; k2 < issued_end; ++k2)
      mbar_wait_bounded(my_bars + (k2 % ST), (k2 / ST) & 1, kDrainLimitNs);
  }

  // ---- combine the 4 row groups of the warp -----------------------------
#pragma unroll
  for (int g = 0; g < GPW; ++g) {
    l[g] += __shfl_xor_sync(kFullMask, l[g], 8);
    l[g] += __shfl_xor_sync(kFullMask, l[g], 16);
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      o[g][e] += __shfl_xor_sync(kFullMask, o[g][e], 8);
      o[g][e] += __shfl_xor_sync(kFullMask, o[g][e], 16);
    }
  }

  // ---- combine the warps through shared memory (each warp its own ring) --
  float* wsm = reinterpret_cast<float*>(my_ring);  // [GPW][D] o, [GPW] m, [GPW] l
  __syncwarp();
  if (grp == 0) {
#pragma unroll
    for (int g = 0; g < GPW; ++g)
#pragma unroll
      for (int k = 0; k < CPL; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) wsm[g * D + (sub + 8 * k) * VEC + e] = o[g][k * VEC + e];
  }
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < GPW; ++g) {
      wsm[GPW * D + g] = m[g];
      wsm[GPW * D + GPW + g] = l[g];
    }
  }
  __syncthreads();

  const size_t H = p.num_heads;
  const bool direct = nsplit == 1;  // the whole context was this block's partition
  for (int idx = threadIdx.x; idx < GPW * D; idx += NW * 32) {
    const int g = idx / D, d = idx - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* ww = reinterpret_cast<const float*>(ring + w * ST * S::kStageBytes);
      M = fmaxf(M, ww[GPW * D + g]);
    }
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* ww = reinterpret_cast<const float*>(ring + w * ST * S::kStageBytes);
      const float mw = ww[GPW * D + g];
      const float sc = mw == -INFINITY ? 0.f : exp2f(mw - M);
      Ls += ww[GPW * D + GPW + g] * sc;
      O += ww[g * D + d] * sc;
    }
    const size_t row = (size_t)seq * H + h0 + g;
    if (direct) {
      store_elem(static_cast<T*>(p.out) + row * D + d, L > 0 ? O / Ls : 0.f);
    } else {
      p.ws_o[(row * p.max_splits + split) * D + d] = O / Ls;
      if (d == 0) p.ws_ml[row * p.max_splits + split] = make_float2(M, Ls);
    }
  }
  if (direct) return;

  // ---- last partition to finish merges all of them (log-sum-exp) --------
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t* ctr = p.ws_counter + (size_t)seq * gridDim.x + blockIdx.x;
    const int prev = atomicAdd(ctr, 1);
    const int last = prev == nsplit - 1;
    if (last) *ctr = 0;  // every partition has counted: leave the counter zero
    *s_last = last;
  }
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  for (int idx = threadIdx.x; idx < GPW * D; idx += NW * 32) {
    const int g = idx / D, d = idx - g * D;
    const size_t row = (size_t)seq * H + h0 + g;
    const float2* ml = p.ws_ml + row * p.max_splits;
    const float* po = p.ws_o + row * p.max_splits * D + d;
    float M = -INFINITY;
    for (int j = 0; j < nsplit; ++j) M = fmaxf(M, __ldcg(ml + j).x);
    float Ls = 0.f, O = 0.f;
    for (int j = 0; j < nsplit; ++j) {
      const float2 v = __ldcg(ml + j);
      const float w = v.y * exp2f(v.x - M);  // l_j 2^(m_j - M)
      Ls += w;
      O += __ldcg(po + (size_t)j * D) * w;   // partials hold o_j / l_j
    }
    store_elem(static_cast<T*>(p.out) + row * D + d, O / Ls);
  }
}

// Launch one instantiation (sets the dynamic shared-memory limit once per device).
template <typename T, int D, int GPW>
cudaError_t launch_pa_decode(const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  using S = DecodeShape<T, D>;
  static unsigned long long configured = 0;  // one bit per device ordinal < 64
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(pa_decode_kernel<T, D, GPW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::kSmemBytes);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&configured, bit, __ATOMIC_ACQ_REL);
  }
  pa_decode_kernel<T, D, GPW><<<grid, kDecodeWarps * 32, S::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

using DecodeLauncher = cudaError_t (*)(const DecodeParams&, dim3, cudaStream_t);

// Per-dtype tables, defined in decode_<dtype>.cu. gpw_index: 0 -> 1, 1 -> 2, 2 -> 4.
DecodeLauncher decode_launcher_f32(int head_dim, int gpw_index);
DecodeLauncher decode_launcher_f16(int head_dim, int gpw_index);
DecodeLauncher decode_launcher_bf16(int head_dim, int gpw_index);

}  // namespace pkv
