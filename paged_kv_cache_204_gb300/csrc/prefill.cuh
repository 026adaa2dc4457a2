// Paged prefill attention (sm_103a): causal attention of each sequence's
// newest tokens over its paged context.
//
// Operation ("PagedAttention: the KV cache was the bottleneck all along",
// section "What is left": shared blocks for common system prompts, i.e. the
// prompt side over the same paged cache; section "Virtual memory for
// attention": K/V in fixed-size blocks reached through a block table).
// Sequence s holds L = context_lens[s] tokens in the cache (its new tokens
// already written); its n = query_start[s+1] - query_start[s] queries are its
// last n tokens, and query i (position L - n + i) attends to tokens
// 0 .. L - n + i. Sequences sharing a system prompt share its blocks, so the
// prompt's K/V is written once.
//
// Work: one CTA per (128-query tile, sequence, query head) on the
// fifth-generation tensor cores. K/V tiles of 64 tokens arrive by TMA, one box
// per cache block found in the block table, in the 128-byte-swizzled layout
// the MMAs read; S = Q K^T and O += P V accumulate in fp32 in tensor memory;
// each query row's online softmax (base 2, causal mask by select) runs in
// the thread that owns that row's tensor-memory lane. For bfloat16 data P
// is fed as a high and a low 16-bit part (two MMAs) so that the
// probabilities keep ~16 significant bits; binary16 P (11 bits) goes as one.
#pragma once

#include <type_traits>

#include "tc.cuh"

namespace pkv {

constexpr int kPfRows = 128;            // query rows per CTA = tensor-memory lanes
constexpr int kPfTokens = 64;           // K/V tokens per tile
constexpr int kPfSoftThreads = 256;     // 8 softmax warps: 4 row quarters x 2 token halves
constexpr int kPfThreads = 320;         // + 1 MMA warp + 1 TMA warp
constexpr int kPfStages = 2;            // K and V tiles in flight
constexpr uint32_t kPfTmemCols = 256;   // two S/P buffers (64 columns each) + O (up to 128)
constexpr float kPfRescaleLog2 = 8.f;   // base of the running max moves only when it grows by more

struct PrefillParams {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  float scale_log2;  // scale * log2(e)
  int num_seqs, num_heads, num_kv_heads, group, block_size, max_blocks_per_seq, num_blocks;
  int32_t* dev_err;
  uint64_t wait_limit_ns;  // limit of every wait on another role's progress
};

// 16-bit packing of two fp32 values (round to nearest) and its exact inverse.
template <typename T>
struct Pack16;
template <>
struct Pack16<__half> {
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
template <>
struct Pack16<__nv_bfloat16> {
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

// 16-byte asynchronous copy; src_bytes 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16_zfill(void* smem, const void* gmem, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// 2^x by the hardware's approximate base-2 exponential (PTX ex2.approx.ftz:
// relative error about 2^-22, -inf -> +0); the probabilities it produces are
// rounded to ~16 bits afterwards.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte chunk c (0..7) of 128-byte row r in a tile with the
// 128-byte swizzle.
__device__ __forceinline__ int sw128_off(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// Shared memory of one CTA (offsets from a 1024-byte aligned base):
//   Q      [2 or 1 column blocks][128 rows][128 B]          (K-major A operand)
//   K, V   [2 stages][D/64 column blocks][64 tokens][128 B]  (K: K-major B of S;
//                                                            V: MN-major B of O)
//   mbarriers, softmax exchange (row maxima and sums), ring of TMA row
//   coordinates, tensor-memory address slot.
// Tensor memory (256 columns, lanes = query rows): S/P buffers at columns 0
// and 64 (S as fp32; P overwrites it as 16-bit hi (/ lo, bfloat16) pairs in columns
// +0..31 / +32..63), O (fp32, D columns) at column 128.
template <int D>
struct PrefillShape {
  static constexpr int kBlocksD = D / 64;                 // 64-element column blocks of a row
  static constexpr int kColBlock = kPfTokens * 128;       // bytes of one column block of a K/V tile
  static constexpr int kTileBytes = kPfTokens * D * 2;
  static constexpr int kQColBlock = kPfRows * 128;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kPfRows * D * 2;
  static constexpr int kVOff = kKOff + kPfStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kPfStages * kTileBytes;
  static constexpr int kXchOff = kBarOff + 16 * 8;         // softmax exchange: 6 x 128 floats
  static constexpr int kRingOff = kXchOff + 6 * kPfRows * 4;  // TMA rows of 8 tiles' blocks
  static constexpr int kSlotOff = kRingOff + 8 * 8 * 4;
  static constexpr int kUsed = kSlotOff + 16 + 1024;      // + alignment slack
  // at least 80 KB, so that at most two CTAs share an SM and their tensor
  // memory (2 x 256 columns) always fits
  static constexpr int kSmemBytes = kUsed > 80 * 1024 ? kUsed : 80 * 1024;
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
};

// One CTA per (128-query tile, sequence, query head); 10 warps:
//   warps 0-7  softmax: warp w reads tensor-memory lanes (query rows)
//              32 (w % 4) .. +31, token half w / 4 of each tile;
//   warp 8     one thread issues the MMAs;
//   warp 9     the TMA loads of K and V tiles (block-table entries fetched
//              ahead by the whole warp, a tile's boxes issued by parallel lanes).
// Per 64-token tile j (stage and S/P buffer j & 1):
//   load:    K_j, V_j box by box (one box = one cache block of one kv head,
//            64 head dims), through the block table;
//   MMA:     S_j = Q K_j^T into buffer j & 1 (issued one tile ahead), then,
//            once P_j is written, O += P_hi V_j and O += P_lo V_j;
//   softmax: scale, causal mask, running max, P = 2^(s - m) (bfloat16: as a
//            high and a low part, the two MMAs together keep ~16 bits); the
//            running max is re-based (and O rescaled in tensor memory) only
//            when it grows by more than kPfRescaleLog2, which leaves every
//            P <= 2^kPfRescaleLog2 and the result exact (O and the row sum
//            use the same base).
template <typename T, int D>
__global__ void __launch_bounds__(kPfThreads, 2)
    pa_prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const PrefillParams p) {
  using S = PrefillShape<D>;
  using P16 = Pack16<T>;
  constexpr int kBf16 = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
  // bfloat16 P (8 significant bits) is fed as a high and a low part; binary16
  // P (11 bits) keeps the outputs well within the tolerance on its own
  constexpr int kPParts = kBf16 ? 2 : 1;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::kBarOff);
  uint64_t* full_k = bars;       // [2] K tile landed
  uint64_t* full_v = bars + 2;   // [2] V tile landed
  uint64_t* empty_k = bars + 4;  // [2] S MMA done with the K stage
  uint64_t* empty_v = bars + 6;  // [2] O MMAs done with the V stage
  uint64_t* s_full = bars + 8;   // [2] S of the buffer computed
  uint64_t* p_full = bars + 10;  // [2] P of the buffer written (one arrival per softmax thread)
  uint64_t* o_done = bars + 12;  // one phase per tile's O MMAs, all tiles but the last
  uint64_t* o_last = bars + 13;  // the last tile's O MMAs: every MMA of the CTA done (one phase)
  uint64_t* q_full = bars + 14;  // Q rows landed (one arrival per loading thread)
  uint64_t* drained = bars + 15; // every MMA the issuing thread started has completed (tear-down)
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + S::kSlotOff);

  // blocks launch in x order: every (sequence, head)'s last query tile (the
  // longest causal range) before any earlier tile
  const int tile = gridDim.y - 1 - blockIdx.y;
  const int s = blockIdx.x / p.num_heads, h = blockIdx.x % p.num_heads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = __ldg(p.context_lens + s);
  const int q0 = __ldg(p.query_start + s), n = __ldg(p.query_start + s + 1) - q0;
  if (L < 0 || L > p.max_blocks_per_seq * p.block_size || n < 0 || n > L) {
    if (tid == 0 && tile == 0 && h == 0) set_err(p.dev_err, PKV_DEV_ERR_CONTEXT_LEN);
    return;
  }
  const int row0 = tile * kPfRows;
  if (row0 >= n) return;  // this tile has no queries (before any allocation)
  const int rows = min(kPfRows, n - row0);
  const int first_pos = L - n + row0;   // position of the tile's first query
  const int kv_end = first_pos + rows;  // tokens the tile's queries can see
  const int ntiles = (kv_end + kPfTokens - 1) / kPfTokens;
  const int kvh = h / p.group;
  const int bs = p.block_size;

  // ---- set-up: Q rows, barriers, tensor memory --------------------------------
  if (tid < kPfRows) {
    const bool ok = tid < rows;
    const T* src = static_cast<const T*>(p.q) + ((size_t)(q0 + row0 + (ok ? tid : 0)) * p.num_heads + h) * D;
#pragma unroll
    for (int c16 = 0; c16 < D / 8; ++c16)
      cp_async16_zfill(sm + S::kQOff + (c16 >> 3) * S::kQColBlock + sw128_off(tid, c16 & 7), src + c16 * 8,
                       ok ? 16 : 0);
    cp_async_commit();
  }
  if (tid == 0) {
    for (int i = 0; i < 16; ++i) mbar_init(&bars[i], (i == 10 || i == 11) ? kPfSoftThreads : (i == 14 ? kPfRows : 1));
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(slot, kPfTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *slot;

  if (warp == 9) {
    // ---- TMA producer ----------------------------------------------------------
    // The warp fetches block-table entries four tiles ahead (lane 8 t + b holds
    // block b of tile t of a group of four) into a shared ring of TMA row
    // coordinates, so that no global load sits between a free stage and its
    // copies.
    const int32_t* bt = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    const int per_tile = kPfTokens / bs;                     // cache blocks per tile (<= 8)
    const int oob_row = p.num_blocks * p.num_kv_heads * bs;  // first row past the pool: reads zeros
    const uint32_t box_bytes = (uint32_t)bs * 128u;
    int* ring = reinterpret_cast<int*>(sm + S::kRingOff);    // [8 tiles][8 blocks]
    auto nblk_of = [&](int j) { return min(per_tile, (kv_end - j * kPfTokens + bs - 1) / bs); };
    const int gt = lane >> 3, gb = lane & 7;  // this lane's tile in a group of four, block in the tile
    auto fetch_group = [&](int g) -> int {    // issues the load only
      const int t = 4 * g + gt;
      return (t < ntiles && gb < nblk_of(t)) ? __ldg(bt + t * per_tile + gb) : 0;
    };
    auto store_group = [&](int g, int id) {
      const int t = 4 * g + gt;
      if (t < ntiles && gb < nblk_of(t)) {
        int y = oob_row;
        if (id >= 0 && id < p.num_blocks)
          y = (id * p.num_kv_heads + kvh) * bs;
        else
          set_err(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
        ring[(t & 7) * 8 + gb] = y;
      }
    };
    // all lanes: lane 0 posts the tile's bytes, then lane 2 b + cb issues the
    // box of block b, column block cb (boxes from one lane issue ~100 cycles apart)
    auto issue = [&](int j, const CUtensorMap* map, unsigned char* stage_base, uint64_t* full) {
      const int nblk = nblk_of(j);
      if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)nblk * S::kBlocksD * box_bytes);
      __syncwarp();
      if (lane < nblk * S::kBlocksD) {
        const int b = lane / S::kBlocksD, cb = lane % S::kBlocksD;
        tma_load_2d(stage_base + cb * S::kColBlock + b * bs * 128, map, cb * 64, ring[(j & 7) * 8 + b], full);
      }
    };
    store_group(0, fetch_group(0));  // the first group waits for its loads
    int pending = fetch_group(1);
    // K and V tiles go as soon as their own stage is free (a K tile is
    // needed by S two tiles before the V tile of the same stage frees); V_j
    // after K_j, whose step wrote tile j's rows into the ring
    int kj = 0, vj = 0;
    bool ok = true;
    uint64_t t_last = 0;
    while (kj < ntiles || vj < ntiles) {
      bool k_go = false, v_go = false;
      if (lane == 0) {
        k_go = kj < ntiles && (kj < 2 || mbar_test_wait(&empty_k[kj & 1], ((kj >> 1) + 1) & 1));
        v_go = vj < kj && (vj < 2 || mbar_test_wait(&empty_v[vj & 1], ((vj >> 1) + 1) & 1));
      }
      k_go = __shfl_sync(kFullMask, k_go ? 1 : 0, 0) != 0;
      v_go = __shfl_sync(kFullMask, v_go ? 1 : 0, 0) != 0;
      if (k_go) {
        if (kj > 0 && (kj & 3) == 0) {  // tiles kj .. kj+3 into the ring, the next group requested
          store_group(kj >> 2, pending);
          pending = fetch_group((kj >> 2) + 1);
        }
        __syncwarp();
        issue(kj, &kmap, sm + S::kKOff + (kj & 1) * S::kTileBytes, &full_k[kj & 1]);
        ++kj;
      }
      if (v_go) {
        issue(vj, &vmap, sm + S::kVOff + (vj & 1) * S::kTileBytes, &full_v[vj & 1]);
        ++vj;
      }
      if (k_go || v_go) {
        t_last = 0;
        continue;
      }
      // nothing free: sleep in the barrier of the tile needed first (K while
      // it is not ahead of V by two, else V), with the overall limit
      if (lane == 0) {
        const uint64_t now = globaltimer_ns();
        if (t_last == 0) t_last = now;
        if (now - t_last >= p.wait_limit_ns) {
          ok = false;
        } else if (kj < ntiles && kj <= vj + 1) {
          mbar_try_wait(&empty_k[kj & 1], ((kj >> 1) + 1) & 1);
        } else if (vj < kj) {
          mbar_try_wait(&empty_v[vj & 1], ((vj >> 1) + 1) & 1);
        }
      }
      ok = __shfl_sync(kFullMask, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
    }
    if (!ok && lane == 0) set_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
    // Every box this warp issued must land before the CTA can leave (its
    // shared memory would otherwise be written after exit). Per stage only
    // the latest tile's phase can still be open: a stage is reissued only
    // after its previous tile was consumed, which needed that tile's bytes.
    if (lane == 0) {
      for (int st = 0; st < kPfStages; ++st) {
        if (kj > st) {
          const int j = st + kPfStages * ((kj - 1 - st) / kPfStages);
          mbar_wait_bounded(&full_k[st], (j >> 1) & 1, kDrainLimitNs);
        }
        if (vj > st) {
          const int j = st + kPfStages * ((vj - 1 - st) / kPfStages);
          mbar_wait_bounded(&full_v[st], (j >> 1) & 1, kDrainLimitNs);
        }
      }
    }
    __syncwarp();
  } else if (warp == 8) {
    // ---- MMA issue ------------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t id_s = mma_idesc_f16(kPfRows, kPfTokens, kBf16, 0);
      constexpr uint32_t id_o = mma_idesc_f16(kPfRows, D, kBf16, 1);
      // descriptors built once; a k-step only moves the start address, whose
      // field (address / 16, low bits of the descriptor) never carries here
      // (shared addresses stay below 256 KB)
      const uint64_t q_desc = smem_desc_sw128(smem_u32(sm + S::kQOff), 16, 1024);
      const uint64_t k_desc0 = smem_desc_sw128(smem_u32(sm + S::kKOff), 16, 1024);
      const uint64_t k_desc1 = smem_desc_sw128(smem_u32(sm + S::kKOff + S::kTileBytes), 16, 1024);
      const uint64_t v_desc0 = smem_desc_sw128(smem_u32(sm + S::kVOff), S::kColBlock, 1024);
      const uint64_t v_desc1 = smem_desc_sw128(smem_u32(sm + S::kVOff + S::kTileBytes), S::kColBlock, 1024);
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait_bounded(&full_k[st], (j >> 1) & 1, p.wait_limit_ns)) return false;
        tc_fence_after();
        const uint64_t kd = st ? k_desc1 : k_desc0;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int cb = ks >> 2, kk = ks & 3;
          mma_ss(tbase + 64 * st, q_desc + (uint64_t)((cb * S::kQColBlock + kk * 32) >> 4),
                 kd + (uint64_t)((cb * S::kColBlock + kk * 32) >> 4), id_s, ks > 0);
        }
        mma_commit(&s_full[st]);
        if (j + 2 < ntiles) mma_commit(&empty_k[st]);  // only commits that someone waits for
        return true;
      };
      // Q (loaded by the first four warps) before the first S
      bool ok = mbar_wait_bounded(q_full, 0, p.wait_limit_ns);
      if (ok) {
        tc_fence_after();
        ok = issue_s(0);
      }
      for (int j = 0; j < ntiles && ok; ++j) {
        const int b = j & 1;
        if (j + 1 < ntiles && !issue_s(j + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait_bounded(&p_full[b], (j >> 1) & 1, p.wait_limit_ns) ||
            !mbar_wait_bounded(&full_v[b], (j >> 1) & 1, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pa = tbase + 64 * b;
        const uint64_t vd = b ? v_desc1 : v_desc0;
#pragma unroll
        for (int part = 0; part < kPParts; ++part)  // high (then low) halves of P
#pragma unroll
          for (int ks = 0; ks < kPfTokens / 16; ++ks)
            mma_ts(tbase + 128, pa + 32 * part + 8 * ks, vd + (uint64_t)((ks * 2048) >> 4), id_o,
                   (j > 0 || part > 0 || ks > 0) ? 1u : 0u);
        // a separate barrier for the last tile: a parity wait tells apart only
        // adjacent phases, and the final wait may come two phases late
        mma_commit(j + 1 < ntiles ? o_done : o_last);
        if (j + 2 < ntiles) mma_commit(&empty_v[b]);
      }
      if (!ok) set_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
      // A commit tracks every MMA this thread issued before it: once it
      // arrives, nothing of the CTA reads shared memory or writes tensor
      // memory any more (after a timeout, MMAs may still be running here).
      mma_commit(drained);
      mbar_wait_bounded(drained, 0, kDrainLimitNs);
    }
    __syncwarp();
  } else {
    // ---- softmax and output --------------------------------------------------
    // Warp w owns query rows 32 (w % 4) .. +31 (its tensor-memory lane
    // quarter) and token half w / 4 of every tile (and that half of the O
    // columns). The two warps of a row quarter exchange partial maxima through
    // shared memory at one named barrier per tile; the barrier also ORs the
    // threads' timeout flags, so that all softmax threads leave together.
    if (tid < kPfRows) {  // the Q rows this thread copied, made visible to the MMAs
      cp_async_wait_all();
      fence_async_smem();
      mbar_arrive(q_full);
    }
    const int r = 32 * (warp & 3) + lane;
    const int ch = warp >> 2;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int pos = min(first_pos + r, kv_end - 1);  // rows past the last query: any finite result
    float* xch = reinterpret_cast<float*>(sm + S::kXchOff);  // [2 tile parities][2 halves][128 rows]
    float* lx = xch + 4 * kPfRows;                            // [2 halves][128 rows]
    const bool pos_scale = p.scale_log2 > 0.f;
    const float sc = pos_scale ? p.scale_log2 : 1.f;
    float m_use = -INFINITY, l = 0.f;
    bool bad = false;
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1;
      const uint32_t par = (j >> 1) & 1;
      const int t0 = j * kPfTokens + 32 * ch;  // first token of this thread's half
      float x[32];
      float pm = -INFINITY;
      // every wait is made warp-uniform before the warp-collective
      // tensor-memory loads and stores that follow it
      if (__all_sync(kFullMask, !bad && mbar_wait_bounded(&s_full[b], par, p.wait_limit_ns))) {
        tc_fence_after();
        uint32_t u[32];
        tmem_ld32(tbase + lane_base + 64 * b + 32 * ch, u);
        tmem_wait_ld();
        // raw scores: with a positive scale the maximum of the scaled scores
        // is the scaled maximum, so scaling folds into the exponent's FFMA
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = pos_scale ? __uint_as_float(u[i]) : __uint_as_float(u[i]) * p.scale_log2;
        const int vis = pos - t0 + 1;  // visible tokens of this half for this row
        if (vis < 32) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i >= vis) x[i] = -INFINITY;
        }
        float m8[8];  // eight independent partial maxima, then a tree
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = x[k];
#pragma unroll
        for (int i = 8; i < 32; ++i) m8[i & 7] = fmaxf(m8[i & 7], x[i]);
        pm = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      } else {
        bad = true;
      }
      xch[(b * 2 + ch) * kPfRows + r] = pm;
      if (barrier_or(1, kPfSoftThreads, bad)) {
        bad = true;
        break;
      }
      const float mt = sc * fmaxf(pm, xch[(b * 2 + (ch ^ 1)) * kPfRows + r]);
      const bool grow = mt > m_use + kPfRescaleLog2;  // first visible tile: always (m_use = -inf)
      float alpha = 1.f;
      if (grow) {
        alpha = exp2f(m_use - mt);  // 0 while nothing was visible
        m_use = mt;
      }
      if (j > 0 && __any_sync(kFullMask, grow)) {
        // O holds the previous tiles' sums on the old base: rescale this
        // warp's half of its columns once their MMAs are done (S_j
        // completing implies those of tile j-2)
        if (__all_sync(kFullMask, mbar_wait_bounded(o_done, (j - 1) & 1, p.wait_limit_ns))) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t w[16];
            const uint32_t a = tbase + lane_base + 128 + (D / 2) * ch + 16 * c;
            tmem_ld16(a, w);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
            tmem_st16(a, w);
          }
        } else {
          bad = true;
        }
      }
      const float nbase = m_use == -INFINITY ? 0.f : -m_use;
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = ex2_approx(fmaf(x[2 * i], sc, nbase)), p1 = ex2_approx(fmaf(x[2 * i + 1], sc, nbase));
        ps4[i & 3] += p0 + p1;
        hi[i] = P16::pack(p0, p1);
        if constexpr (kPParts == 2) {
          const float2 hv = P16::unpack(hi[i]);
          lo[i] = P16::pack(p0 - hv.x, p1 - hv.y);
        }
      }
      l = l * alpha + ((ps4[0] + ps4[1]) + (ps4[2] + ps4[3]));  // this half's share of the row sum
      // P of this half: packed pairs at columns 16 ch .. (high) and 32 + 16 ch .. (low)
      __syncwarp();
      tmem_st16(tbase + lane_base + 64 * b + 16 * ch, hi);
      if constexpr (kPParts == 2) tmem_st16(tbase + lane_base + 64 * b + 32 + 16 * ch, lo);
      tmem_wait_st();
      if (j == ntiles - 1 && kv_end < j * kPfTokens + kPfTokens) {
        // V rows past the context may hold anything (a NaN would survive a
        // zero probability): zero them once the tile has landed
        if (__all_sync(kFullMask, mbar_wait_bounded(&full_v[b], par, p.wait_limit_ns))) {
          const int z0 = kv_end - j * kPfTokens, per_row = S::kBlocksD * 8;
          unsigned char* vd = sm + S::kVOff + b * S::kTileBytes;
          for (int i = tid; i < (kPfTokens - z0) * per_row; i += kPfSoftThreads) {
            const int row = z0 + i / per_row, rem = i % per_row;
            *reinterpret_cast<uint4*>(vd + (rem >> 3) * S::kColBlock + row * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_async_smem();
        } else {
          bad = true;
        }
      }
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }
    lx[ch * kPfRows + r] = l;
    bad = barrier_or(1, kPfSoftThreads, bad);
    if (!bad && !__all_sync(kFullMask, mbar_wait_bounded(o_last, 0, p.wait_limit_ns))) bad = true;
    if (bad) {
      if (lane == 0) set_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
    } else {
      __syncwarp();
      tc_fence_after();
      const float lt = l + lx[(ch ^ 1) * kPfRows + r];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      T* og = static_cast<T*>(p.out) + ((size_t)(q0 + row0 + r) * p.num_heads + h) * D + (D / 2) * ch;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t w[32];
        tmem_ld32(tbase + lane_base + 128 + (D / 2) * ch + 32 * c, w);
        tmem_wait_ld();
        if (r < rows) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = P16::pack(__uint_as_float(w[2 * i]) * inv, __uint_as_float(w[2 * i + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(og + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
    }
  }

  // ---- tear-down: the TMA warp's boxes have landed and the MMA thread's
  // MMAs have completed (each drain bounded by kDrainLimitNs; if one ran
  // out, the error word already marks this call's outputs as invalid) -----
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, kPfTmemCols);
  }
}

// Rows of a cache pool as a 2-D tensor of 16-bit elements, read in boxes of
// {64 elements, block_size rows} with the 128-byte swizzle.
template <typename T, int D>
cudaError_t encode_pool_map(CUtensorMap* map, const void* base, const PrefillParams& p) {
  return encode_pool_rows_map(map, base, (uint64_t)p.num_blocks * p.num_kv_heads * p.block_size, D, p.block_size,
                              std::is_same<T, __nv_bfloat16>::value);
}

template <typename T, int D>
cudaError_t launch_pa_prefill(const PrefillParams& p, int max_query_len, cudaStream_t stream) {
  using S = PrefillShape<D>;
  // the TMA row coordinate (and one box past the pool) must fit in int32
  if ((long long)p.num_blocks * p.num_kv_heads * p.block_size + kPfTokens > 0x7fffffffLL)
    return cudaErrorNotSupported;
  if (kPfTokens % p.block_size != 0) return cudaErrorNotSupported;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
    e = cudaFuncSetAttribute(pa_prefill_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
  }
  CUtensorMap kmap, vmap;
  e = encode_pool_map<T, D>(&kmap, p.k_cache, p);
  if (e != cudaSuccess) return e;
  e = encode_pool_map<T, D>(&vmap, p.v_cache, p);
  if (e != cudaSuccess) return e;
  if ((max_query_len + kPfRows - 1) / kPfRows > 65535) return cudaErrorNotSupported;
  const dim3 grid(p.num_seqs * p.num_heads, (max_query_len + kPfRows - 1) / kPfRows);
  pa_prefill_kernel<T, D><<<grid, kPfThreads, S::kSmemBytes, stream>>>(kmap, vmap, p);
  return cudaGetLastError();
}

using PrefillLauncher = cudaError_t (*)(const PrefillParams&, int, cudaStream_t);
PrefillLauncher prefill_launcher(int is_bf16, int head_dim);

}  // namespace pkv
