// Paged decode attention kernel (sm_103a).
//
// Operation ("PagedAttention: the KV cache was the bottleneck all along",
// section "Virtual memory for attention"): one query token per sequence
// attends over its context, whose K/V rows sit in fixed-size blocks scattered
// through a pool and are found through the sequence's block table.
//
// Work decomposition (persistent, balanced by construction)
//   Every (sequence s, head group hg) pair is a "segment" of nt_s tiles of 16
//   tokens (an empty context still has one, empty, tile so that its zero
//   output gets written). Segments are laid end to end, sequence-major, into
//   one global sequence of T tiles. The grid is sized to the GPU (blocks that
//   stay resident); its W warps each take one contiguous range of about T/W
//   tiles, so every warp streams the same number of bytes.
//   A warp walks its range tile by tile across segment boundaries. Its lanes
//   issue 1-D bulk copies (cp.async.bulk, completion counted in bytes on an
//   mbarrier; one lane per copy, since copies from one lane queue behind one
//   another) of the next tiles' K rows and V rows (plus the segment's query
//   rows at the first tile of a segment) into the warp's own ring of
//   shared-memory slots, while all lanes compute on the current tile. There
//   is no block-wide barrier after the start-up scan.
//   A segment that lies entirely inside one warp's range is finished by that
//   warp, which writes the output. A segment cut by range boundaries (at most
//   two per warp: its first and its last) gets one partial (m, l, o/l) per
//   piece in the workspace; the last piece to finish (atomic counter) merges
//   them with the log-sum-exp rule, writes the output and re-zeroes the
//   counter.
//
// Per tile and warp: lanes form 4 groups of 8; group g holds tokens g, g+4,
// g+8, g+12 of the tile and lane i of a group owns 16-byte chunks i, i+8, ...
// of every row (a quarter-warp reads 128 contiguous bytes of one row: no
// shared-memory bank conflicts). q.k partial sums are reduced over the 8
// lanes of a group with shuffles; the running max m, exp-sum l and output o
// follow the online softmax in base 2 (q is pre-scaled by scale * log2(e));
// tokens past the context are masked by select, never by multiplication, so
// poisoned rows never reach the result. An fp8 cache read with one query head
// per warp takes the tensor-core tile instead (FpMma below): same ring,
// segments and merges, q.K^T and P.V of each 32-token tile as MMAs.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "tc.cuh"

namespace pkv {

struct DecodeParams {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float scale_log2;  // scale * log2(e)
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int group;        // num_heads / num_kv_heads
  int head_groups;  // num_heads / GPW
  int block_size;
  int max_blocks_per_seq;
  int num_blocks;
  int max_context_len;
  int32_t* ws_counter;  // [num_seqs * head_groups]
  float2* ws_ml;        // [kMaxDecodeWarps][2][GPW]  (m, l)
  float* ws_o;          // [kMaxDecodeWarps][2][GPW][head_dim]
  int32_t* dev_err;
  uint64_t wait_limit_ns;
  float v_scale;  // fp8 caches: stored V times v_scale is the value (1 otherwise)
};

constexpr int kTileTokens = 16;  // tokens of a tile of a 16- or 32-bit cache

// Element tag of a q4_0 cache: each row of D values is D/32 blocks of 32,
// stored as the D/32 binary16 scales d_b, then 16 code bytes per block (byte
// j of block b holds value 32 b + j in its low and 32 b + j + 16 in its high
// four bits); a code q reads back as d_b (q - 8). 9 D / 16 bytes per row.
struct Q4Row {};

template <typename KT>
struct CacheKind {
  static constexpr bool kFp8 = std::is_same<KT, __nv_fp8_e4m3>::value;
  static constexpr bool kQ4 = std::is_same<KT, Q4Row>::value;
  template <int D>
  static constexpr int row_bytes() { return kQ4 ? D / 16 * 9 : D * (int)sizeof(KT); }
};

// Tokens per tile of the plain kernel: fp8 and q4_0 caches take 32-token
// tiles, so a tile carries about as many bytes (and a warp's per-tile work
// as much data) as a 16-token tile of a 16-bit cache.
template <typename KT>
constexpr int tile_tokens_for() {
  return CacheKind<KT>::kQ4 ? 4 * kTileTokens : CacheKind<KT>::kFp8 ? 2 * kTileTokens : kTileTokens;
}
constexpr int kDecodeWarps = 8;  // one resident block of 8 warps per SM (measured best)
// fp8 caches (1 or 2 query heads per warp): a warp's per-tile work is a
// longer latency chain for half the bytes, so more warps share an SM (as many
// as registers allow) with a larger ring budget.
constexpr int kFp8Warps2 = 12;  // two query heads per warp, CUDA cores (register limit)
// One query head per warp: q.K^T and P.V of a tile on tensor cores (FpMma
// below), one 32-token stage per warp. Measured on the LLaMA-13B-shaped step
// (attention, 200 steps): 12 warps (two stages each) 176.7 us, 16 warps
// 170.6 us, 20 warps 182.5 us (registers capped at 96: spills); 16-token
// tiles with three stages per warp 191.2 us at 16 warps.
constexpr int kFp8MmaWarps = 16;
constexpr int kFp8RingBudget = 200 * 1024;
constexpr int kMaxDecodeWarps = 4096;  // bound of the persistent grid (partial slots in the workspace)
constexpr int kMaxGroupPerWarp = 4;    // query heads one warp serves against one kv head
constexpr int kBtChunk = 128;          // block-table entries a warp keeps in shared memory

// Which head dims lane `sub` of an 8-lane row group owns, and how it reads
// them from a cache row (element KT) and from a query / output row (T).
// Same element type: 16-byte chunks sub, sub + 8, ... of the row. fp8
// caches: one run of D / 8 dims starting at dim sub * D / 8 (8 or 16 codes),
// so a quarter-warp still reads one whole cache row.
template <typename T, typename KT, int D>
struct LaneDims {
  static constexpr int kVec = Chunk<T>::kElems;
  static constexpr int kParts = D * (int)sizeof(T) / 16 / 8;  // chunks per lane per row
  static constexpr int kPartElems = kVec;
  __device__ __forceinline__ static int dim(int sub, int k, int e) { return (sub + 8 * k) * kVec + e; }
  __device__ __forceinline__ static void kv(const unsigned char* row, int sub, int k, float (&f)[kPartElems]) {
    Chunk<T>::widen(reinterpret_cast<const uint4*>(row)[sub + 8 * k], f);
  }
  __device__ __forceinline__ static void q(const unsigned char* row, int sub, int k, float (&f)[kPartElems]) {
    Chunk<T>::widen(reinterpret_cast<const uint4*>(row)[sub + 8 * k], f);
  }
  __device__ __forceinline__ static void out(unsigned char* row, int sub, int k, const float (&f)[kPartElems]) {
    reinterpret_cast<uint4*>(row)[sub + 8 * k] = Chunk<T>::narrow(f);
  }
};
template <typename T, int D>
struct LaneDims<T, __nv_fp8_e4m3, D> {
  static_assert(sizeof(T) == 2, "fp8 caches take 16-bit queries");
  static constexpr int kParts = 1;
  static constexpr int kPartElems = D / 8;         // 8 or 16 dims
  static constexpr int kQChunks = kPartElems / 8;  // 16-byte chunks of T per lane
  __device__ __forceinline__ static int dim(int sub, int, int e) { return sub * kPartElems + e; }
  __device__ __forceinline__ static void kv(const unsigned char* row, int sub, int, float (&f)[kPartElems]) {
    const uint2* r = reinterpret_cast<const uint2*>(row + sub * kPartElems);
#pragma unroll
    for (int c = 0; c < kPartElems / 8; ++c) {
      float g[8];
      widen_e4m3x8(r[c], g);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[8 * c + e] = g[e];
    }
  }
  __device__ __forceinline__ static void q(const unsigned char* row, int sub, int, float (&f)[kPartElems]) {
    const uint4* r = reinterpret_cast<const uint4*>(row + sub * kPartElems * 2);
#pragma unroll
    for (int c = 0; c < kQChunks; ++c) {
      float g[8];
      Chunk<T>::widen(r[c], g);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[8 * c + e] = g[e];
    }
  }
  __device__ __forceinline__ static void out(unsigned char* row, int sub, int, const float (&f)[kPartElems]) {
    uint4* r = reinterpret_cast<uint4*>(row + sub * kPartElems * 2);
#pragma unroll
    for (int c = 0; c < kQChunks; ++c) {
      float g[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) g[e] = f[8 * c + e];
      r[c] = Chunk<T>::narrow(g);
    }
  }
};

// q4_0 caches (tensor-core tile, one query head per warp, Q4Mma below): lane
// sub of the CUDA-core layout ends with the head dims of the low (e < DPL/2)
// and high (e >= DPL/2) four bits of its DPL/2 code bytes of one block: two
// runs of DPL/2 contiguous dims.
template <typename T, int D>
struct LaneDims<T, Q4Row, D> {
  static_assert(sizeof(T) == 2, "q4_0 caches take 16-bit queries");
  static constexpr int kParts = 1;
  static constexpr int kPartElems = D / 8;  // 8 or 16 dims
  static constexpr int kHalf = D / 16;      // dims per run
  static constexpr int kLanesPerBlock = 8 / (D / 32);
  __device__ __forceinline__ static int dim(int sub, int, int e) {
    return 32 * (sub / kLanesPerBlock) + (e < kHalf ? 0 : 16) + kHalf * (sub % kLanesPerBlock) + (e % kHalf);
  }
  __device__ __forceinline__ static void q(const unsigned char* row, int sub, int, float (&f)[kPartElems]) {
    const T* r = reinterpret_cast<const T*>(row);
#pragma unroll
    for (int e = 0; e < kPartElems; ++e) f[e] = to_float(r[dim(sub, 0, e)]);
  }
  __device__ __forceinline__ static void out(unsigned char* row, int sub, int, const float (&f)[kPartElems]) {
    T* r = reinterpret_cast<T*>(row);
#pragma unroll
    for (int e = 0; e < kPartElems; ++e) store_elem(r + dim(sub, 0, e), f[e]);
  }
};

// Tensor-core tile of an fp8 cache with one query head per warp (m16n8k16,
// binary16 operands, fp32 accumulation). Every e4m3 value is exactly a
// binary16 value, so K and V enter the MMAs exactly; the query row enters as
// binary16 after scaling by a power of two that brings its largest element
// into [2^14, 2^15) (exact for every element within 2^28 of the largest; the
// power of two is taken back out of the scores), and P as a binary16 high
// part plus a binary16 remainder, about 22 significant bits.
//
// Scores, S^T = K q^T: the tile's tokens are M (two 16-token halves), the
// head dims K, and q fills every column of N, so every lane holds scores.
// The head dims are permuted consistently in K and q (which leaves the dot
// product unchanged) so that lane (g, t) = (lane / 4, lane % 4) finds every A
// element it needs in bytes [t D/4, (t+1) D/4) of its two token rows: k-step
// kk, MMA column 2t + u + 8v is byte t D/4 + 4 kk + 2 v + u. Lane (g, t) holds
// the scores of tokens g and g + 8 of each half.
//
// Output, O^T += V^T P^T: the head dims are M (D / 16 tiles), the tokens K,
// P_hi and P_lo columns 0 and 1 of N (the rest zero). The B fragments of P^T
// are the transposes (movmatrix) of the 8 x 8 matrices [token][column] that
// the score layout gives. MMA row 16 m + g + 8 v is head dim (D/8) g + 2 m + v,
// so lane (g, t) reads bytes [g D/8, (g+1) D/8) of its four token rows 2t,
// 2t + 1, 2t + 8, 2t + 9, and lane 4g ends with the head dims (D/8) g .. + D/8:
// the same dims lane g holds in the CUDA-core layout.
struct FpMma {
  __device__ __forceinline__ static void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  // the two e4m3 codes in the low (high) 16 bits of w as a binary16 pair,
  // the lower byte in the lower half
  __device__ __forceinline__ static uint32_t lo2(uint32_t w) {
    uint32_t r;
    asm("{.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;}" : "=r"(r) : "r"(w));
    return r;
  }
  __device__ __forceinline__ static uint32_t hi2(uint32_t w) {
    uint32_t r;
    asm("{.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;}" : "=r"(r) : "r"(w));
    return r;
  }
  __device__ __forceinline__ static uint32_t pack(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
  }
  __device__ __forceinline__ static float2 unpack(uint32_t u) {
    __half2 h;
    memcpy(&h, &u, 4);
    return __half22float2(h);
  }
  // transpose of an 8 x 8 matrix of 16-bit elements in fragment layout
  __device__ __forceinline__ static uint32_t trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
  }
  // 2^k with k in [-126, 127]
  __device__ __forceinline__ static float pow2(int k) { return __int_as_float((k + 127) << 23); }
};

// Tensor-core tile of a q4_0 cache, one query head per warp (m16n8k16,
// binary16 operands, fp32 accumulation). A code q enters the MMAs as its own
// four bits, masked in place: the binary16 subnormal q 2^-24 (low nibble)
// or 16 q 2^-24 (high nibble), exact; the query operand of high-nibble
// k-steps is scaled by 1/16 to match. The offset 8 and the scales stay out
// of the A operands: sum_j (q_j - 8) x_j = 2^24 sum_j (q_j 2^-24) x_j -
// 8 sum_j x_j, with the sums of the query (scores) and of P (output) kept
// beside the MMAs.
//
// Scores, S^T = K q^T: tokens are M, head dims K. Lane (g, t) supplies the
// A elements of block t (head_dim 128; head_dim 64: half t % 2 of block
// t / 2): k-step kk takes code word kk / 2 of its part, low (kk even) or
// high four bits, bytes 0 and 2 as MMA columns 2t, 2t + 1 and bytes 1 and 3
// as 2t + 8, 2t + 9. Column n of the query operand holds the query only at
// the dims of block n (zero elsewhere), so column n of S^T is 2^-24 times
// the block-n partial sum of q x and the score is sum_n d_n (2^24 S^T[., n]
// - 8 sum_{j in n} x_j) (the scales multiply fp32 partial sums).
//
// Output, O^T += V^T P^T: head dims are M, tokens K; column 2 b + u of P^T
// holds the high (u = 0) or low (u = 1) binary16 part of p d_b (the V row's
// scale of block b), so for a dim of block b the output is 2^24 (2^20 for a
// high nibble) times O^T[dim, 2 b] + O^T[dim, 2 b + 1], less 8 times the sum
// of that column pair over the tokens. Lane (g, t) reads code bytes
// [g D/16, (g + 1) D/16) of its four token rows; byte m gives MMA rows g
// (low bits) and g + 8 (high bits) of m-tile m; lane (g, blk(g)) ends with
// those dims (LaneDims<T, Q4Row, D>).
struct Q4Mma {
  // binary16 pair of the nibbles n0, n1 at bits 0-3 and 16-19 of w, as the
  // subnormals n 2^-24 (the bit pattern n itself: exact)
  __device__ __forceinline__ static uint32_t lo(uint32_t w) { return w & 0x000F000Fu; }
  // the nibbles at bits 4-7 and 20-23, left in place: 16 n 2^-24
  __device__ __forceinline__ static uint32_t hi(uint32_t w) { return w & 0x00F000F0u; }
};

// NWO / BudgetO: explicit warps per block and ring budget (0: the defaults).
template <typename T, int D, int GPW, typename KT = T, int NWO = 0, int BudgetO = 0>
struct DecodeShape {
  static constexpr bool kQ4 = CacheKind<KT>::kQ4;  // q4_0 cache: tensor-core tile, one head per warp
  static constexpr bool kFp8Wide = CacheKind<KT>::kFp8 && GPW <= 2;
  static constexpr bool kFp8Mma = CacheKind<KT>::kFp8 && GPW == 1;
  static constexpr int kWarps =
      NWO ? NWO : ((kFp8Mma || kQ4) ? kFp8MmaWarps : kFp8Wide ? kFp8Warps2 : kDecodeWarps);
  static constexpr int kElemBytes = sizeof(T);
  static constexpr int kRowBytes = D * kElemBytes;                       // query / output row
  static constexpr int kKvRowBytes = CacheKind<KT>::template row_bytes<D>();  // cache row
  static constexpr int kTileTokensT = tile_tokens_for<KT>();
  static constexpr int kTileBytes = kTileTokensT * kKvRowBytes;          // K (or V) rows of one tile
  // the tensor-core fp8 tile at head_dim 128 takes its K and V rows by 2-D
  // TMA with the 128-byte swizzle (conflict-free reads of its fragments):
  // stages start on 1024-byte boundaries
  static constexpr bool kTma = kFp8Mma && D == 128;
  static constexpr int kStageRaw = 2 * kTileBytes + GPW * kRowBytes;     // K, V, query rows
  static constexpr int kStageBytes = kTma ? (kStageRaw + 1023) / 1024 * 1024 : kStageRaw;
  static constexpr int kRingBudget = BudgetO ? BudgetO : ((kFp8Wide || kQ4) ? kFp8RingBudget : 128 * 1024);
  static constexpr int kStagesRaw = kRingBudget / (kWarps * 2 * kTileBytes);
  static constexpr int kStages = kStagesRaw < 1 ? 1 : (kStagesRaw > 4 ? 4 : kStagesRaw);
  static constexpr int kChunksPerRow = kRowBytes / 16;
  static constexpr int kChunksPerLane = kChunksPerRow / 8;
  static constexpr int kVec = Chunk<T>::kElems;
  static constexpr int kDimsPerLane = D / 8;
  static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kBtOff = kBarOff + kWarps * kStages * 8;
  static constexpr int kScanOff = kBtOff + kWarps * kBtChunk * 4;
  static constexpr int kStartOff = kScanOff + kWarps * 8;
  static constexpr int kSmemBytes = kStartOff + kWarps * 16 + (kTma ? 1024 : 0);  // + alignment of the base
  static_assert(!kQ4 || GPW == 1, "q4_0 caches: one query head per warp");
  static_assert(kChunksPerRow % 8 == 0, "row must split into 8 lanes of 16-byte chunks");
  static_assert(kDimsPerLane * 8 == D, "lane mapping");
  static_assert(kStageBytes % 16 == 0 && kRowBytes % 16 == 0 && kTileBytes % 16 == 0, "bulk copy alignment");
};

template <int TT>
__device__ __forceinline__ int tiles_of_t(int L) { return L > 0 ? (L + TT - 1) / TT : 1; }
__device__ __forceinline__ int tiles_of(int L) { return tiles_of_t<kTileTokens>(L); }

// Context length of sequence s, clamped into [0, cap] (out-of-range lengths
// are reported once, by block 0).
__device__ __forceinline__ int load_len(const DecodeParams& p, int s, int cap) {
  int L = __ldg(p.context_lens + s);
  if (L < 0 || L > cap) {
    if (blockIdx.x == 0) set_err(p.dev_err, PKV_DEV_ERR_CONTEXT_LEN);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

// Exclusive scan of one value per thread over a block of NW warps; `total`
// gets the sum.
template <int NW = kDecodeWarps>
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* scratch, long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(kFullMask, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  long long before = 0;
  total = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const long long t = scratch[i];
    if (i < warp) before += t;
    total += t;
  }
  __syncthreads();
  return before + x - v;
}

// Position in the global tile sequence.
struct TileCursor {
  long long g;  // global tile index
  int s, hg, t, nt, L;
};

template <int TT>
__device__ __forceinline__ void cursor_next(TileCursor& c, const DecodeParams& p, int cap) {
  ++c.g;
  if (++c.t < c.nt) return;
  c.t = 0;
  if (++c.hg < p.head_groups) return;
  c.hg = 0;
  if (++c.s < p.num_seqs) {
    c.L = load_len(p, c.s, cap);
    c.nt = tiles_of_t<TT>(c.L);
  }
}

template <typename T, int D, int GPW, typename KT = T>
__global__ void __launch_bounds__(DecodeShape<T, D, GPW, KT>::kWarps * 32)
    pa_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const DecodeParams p) {
  using S = DecodeShape<T, D, GPW, KT>;
  using LD = LaneDims<T, KT, D>;
  constexpr bool kQuant = CacheKind<KT>::kFp8;  // values are codes times p.v_scale
  constexpr bool kQ4 = S::kQ4;
  constexpr bool kMma = S::kFp8Mma || kQ4;     // one query head per warp: tensor-core tiles
  constexpr int NKS = D / 16;          // MMA k-steps of the scores, m-tiles of the output
  constexpr int TT = S::kTileTokensT;  // tokens per tile
  constexpr int RPG = TT / 4;          // rows of a tile per 8-lane group
  constexpr int NW = S::kWarps;
  constexpr int ST = S::kStages;
  constexpr int DPL = S::kDimsPerLane;
  constexpr int CPL = LD::kParts;       // pieces of a row per lane
  constexpr int VEC = LD::kPartElems;  // dims per piece
  constexpr int ROW = S::kRowBytes;    // query / output row bytes
  constexpr int KROW = S::kKvRowBytes; // cache row bytes

  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = S::kTma ? smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u) : smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  long long* scan = reinterpret_cast<long long*>(smem + S::kScanOff);
  longlong2* starts = reinterpret_cast<longlong2*>(smem + S::kStartOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = lane >> 3;  // token sub-index within a 4-row step
  const int sub = lane & 7;   // chunk index within a row
  const int bs = p.block_size;
  const int cap = min(p.max_context_len, p.max_blocks_per_seq * bs);
  const int HG = p.head_groups;

  // ---- start-up: total tiles T, then each warp's first (sequence, offset) --
  long long mine = 0;
  for (int s = threadIdx.x; s < p.num_seqs; s += NW * 32) mine += tiles_of_t<TT>(load_len(p, s, cap));
  long long Ttot;
  block_exclusive_scan<NW>(mine, scan, Ttot);
  Ttot *= HG;
  const long long W = (long long)gridDim.x * NW;
  const long long Weff = W < Ttot ? W : Ttot;  // every active warp gets >= 1 tile
  const long long wid = (long long)blockIdx.x * NW + warp;
  const long long a_begin = wid < Weff ? wid * Ttot / Weff : Ttot;
  const long long a_end = wid < Weff ? (wid + 1) * Ttot / Weff : Ttot;
  if (threadIdx.x < NW) starts[threadIdx.x] = make_longlong2(-1, 0);
  __syncthreads();
  long long carry = 0;
  for (int base = 0; base < p.num_seqs; base += NW * 32) {
    const int s = base + threadIdx.x;
    const long long cnt = s < p.num_seqs ? (long long)tiles_of_t<TT>(load_len(p, s, cap)) * HG : 0;
    long long chunk_total;
    const long long excl = carry + block_exclusive_scan<NW>(cnt, scan, chunk_total);
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const long long w = (long long)blockIdx.x * NW + i;
      if (w < Weff) {
        const long long a = w * Ttot / Weff;
        if (cnt > 0 && a >= excl && a < excl + cnt) starts[i] = make_longlong2(s, a - excl);
      }
    }
    carry += chunk_total;
  }
  __syncthreads();
  if (a_begin >= a_end) return;  // idle warp (more warps than tiles); no block barrier follows

  // ---- per-warp pipeline ------------------------------------------------
  unsigned char* my_ring = smem + warp * ST * S::kStageBytes;
  uint64_t* my_bars = bars + warp * ST;
  int32_t* my_bt = reinterpret_cast<int32_t*>(smem + S::kBtOff) + warp * kBtChunk;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < ST; ++i) mbar_init(&my_bars[i], 1);
    mbar_init_fence();
  }
  __syncwarp();

  TileCursor ci;  // issue cursor
  {
    const longlong2 st0 = starts[warp];
    ci.s = static_cast<int>(st0.x);
    ci.L = load_len(p, ci.s, cap);
    ci.nt = tiles_of_t<TT>(ci.L);
    ci.hg = static_cast<int>(st0.y / ci.nt);
    ci.t = static_cast<int>(st0.y % ci.nt);
    ci.g = a_begin;
  }
  TileCursor cc = ci;  // consume cursor
  int bt_s = -1, bt_j0 = 0;

  const char* kbase = static_cast<const char*>(p.k_cache);
  const char* vbase = static_cast<const char*>(p.v_cache);
  const char* qbase = static_cast<const char*>(p.q);
  const int seg = bs < TT ? bs : TT;  // rows per bulk copy
  const int nseg = TT / seg;

  // Issue the copies of the tile under `c` into slot n % ST (warp-uniform call).
  auto issue = [&](const TileCursor& c, int n) {
    const int t0 = c.t * TT;
    const int nvalid = min(max(c.L - t0, 0), TT);
    const bool with_q = (c.t == 0 || c.g == a_begin) && nvalid > 0;
    if (nvalid > 0) {
      const int j_first = t0 / bs;
      const int j_last = (t0 + nvalid - 1) / bs;
      if (c.s != bt_s || j_first < bt_j0 || j_last >= bt_j0 + kBtChunk) {
        // stage block-table entries [j_first, j_first + kBtChunk) of row c.s
        const int nblk = (c.L + bs - 1) / bs;
        const int32_t* row = p.block_tables + (size_t)c.s * p.max_blocks_per_seq;
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
        bt_s = c.s;
        bt_j0 = j_first;
      }
    }
    // the segments of rows that hold context tokens go from lanes 0 ..
    // 2 nsv - 1 at once (lane 2 c2 the K rows of segment c2, lane 2 c2 + 1 its
    // V rows: copies issued from one lane queue behind one another), the
    // query rows from lane 2 nsv; lane 0 posts the bytes first
    unsigned char* kdst = my_ring + (n % ST) * S::kStageBytes;
    uint64_t* bar = my_bars + (n % ST);
    const int nsv = min(nseg, (nvalid + seg - 1) / seg);
    if (lane == 0) mbar_arrive_expect_tx(bar, (with_q ? GPW * ROW : 0u) + 2u * nsv * seg * KROW);
    __syncwarp();
    if (lane < 2 * nsv) {
      const int c2 = lane >> 1, isv = lane & 1;
      const int t = t0 + c2 * seg;
      const int kvh = (c.hg * GPW) / p.group;
      unsigned char* dst = kdst + isv * S::kTileBytes + c2 * seg * KROW;
      if constexpr (S::kTma) {  // boxes of {128 bytes, seg rows}, swizzled
        const int y = (my_bt[t / bs - bt_j0] * p.num_kv_heads + kvh) * bs + (t % bs);
        tma_load_2d(dst, isv ? &vmap : &kmap, 0, y, bar);
      } else {
        const size_t off = (((size_t)my_bt[t / bs - bt_j0] * p.num_kv_heads + kvh) * bs + (t % bs)) * KROW;
        bulk_copy_g2s(dst, (isv ? vbase : kbase) + off, seg * KROW, bar);
      }
    } else if (lane == 2 * nsv && with_q) {
      bulk_copy_g2s(kdst + 2 * S::kTileBytes, qbase + ((size_t)c.s * p.num_heads + (size_t)c.hg * GPW) * ROW,
                    GPW * ROW, bar);
    }
  };

  int issued = 0;
  for (; issued < ST && ci.g < a_end; ++issued) {
    issue(ci, issued);
    cursor_next<TT>(ci, p, cap);
  }

  float qf[GPW][DPL];
  float m[GPW], l[GPW], o[GPW][DPL];
  // tensor-core state (kMma): the scaled query as B fragments, O^T
  // accumulators, and the scale of the scores
  uint32_t qb[NKS][2];
  float oa[NKS][4];
  float sc_q = 0.f;
  // q4_0: 8 x the query sums of blocks 2t, 2t + 1 (this lane's score
  // columns) and the running sum of this lane's P column pair (block t)
  float q4_corr0 = 0.f, q4_corr1 = 0.f, q4_psum = 0.f;
  bool visit_from_start = true;
  const size_t H = p.num_heads;

  for (int n = 0; cc.g < a_end; ++n) {
    if (!__all_sync(kFullMask, mbar_wait_bounded(my_bars + (n % ST), (n / ST) & 1, p.wait_limit_ns))) {
      // A wait ran out: report it, let this warp's copies in flight land
      // (bounded), and stop. Outputs of this call are not valid.
      if (lane == 0) set_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
      for (int k2 = n; k2 < issued; ++k2) mbar_wait_bounded(my_bars + (k2 % ST), (k2 / ST) & 1, kDrainLimitNs);
      return;
    }
    const unsigned char* ks = my_ring + (n % ST) * S::kStageBytes;
    const unsigned char* vs = ks + S::kTileBytes;
    const int t0 = cc.t * TT;
    const int nvalid = min(max(cc.L - t0, 0), TT);
    const bool first = cc.t == 0 || cc.g == a_begin;
    const bool last = cc.t == cc.nt - 1 || cc.g == a_end - 1;

    if constexpr (kMma) {
      if (first) {
        visit_from_start = cc.t == 0;
        m[0] = -INFINITY;
        l[0] = 0.f;
#pragma unroll
        for (int mm = 0; mm < NKS; ++mm) oa[mm][0] = oa[mm][1] = oa[mm][2] = oa[mm][3] = 0.f;
        q4_psum = 0.f;
        if (kQ4 && nvalid > 0) {
          // lane (g, t): the query dims of its code part (bytes [PB t, PB (t+1))
          // of the row's codes, low then high four bits); nonzero B columns
          // only where the column is the part's block
          constexpr int PB = D / 8;  // code bytes of a lane's part
          const int t = lane & 3, g = lane >> 2;
          const int blk = t / (128 / D);
          const int e0 = 32 * blk + (D == 128 ? 0 : 8 * (t & 1));
          const unsigned char* qrow = ks + 2 * S::kTileBytes;
          float qv[2][PB];
#pragma unroll
          for (int hb = 0; hb < 2; ++hb)
#pragma unroll
            for (int c = 0; c < PB / 8; ++c) {
              float f8[8];
              Chunk<T>::widen(*reinterpret_cast<const uint4*>(qrow + 2 * (e0 + 16 * hb + 8 * c)), f8);
#pragma unroll
              for (int e = 0; e < 8; ++e) qv[hb][8 * c + e] = f8[e];
            }
          float amax = 0.f;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb)
#pragma unroll
            for (int e = 0; e < PB; ++e) amax = fmaxf(amax, fabsf(qv[hb][e]));
          amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
          int k = 0;
          if (amax > 0.f) k = min(141 - ((__float_as_int(amax) >> 23) & 0xff), 127);
          const float sig = FpMma::pow2(max(k, -126));
          sc_q = ldexpf(p.scale_log2, -max(k, -126));
          const bool mine = g == blk;
#pragma unroll
          for (int kk = 0; kk < NKS; ++kk) {  // code word kk / 2, four bits kk % 2 (high: times 1/16)
            const int hb = kk & 1, j = 4 * (kk >> 1);
            const float sk = hb ? sig * 0.0625f : sig;
            qb[kk][0] = mine ? FpMma::pack(qv[hb][j] * sk, qv[hb][j + 2] * sk) : 0u;
            qb[kk][1] = mine ? FpMma::pack(qv[hb][j + 1] * sk, qv[hb][j + 3] * sk) : 0u;
          }
          // 8 x the sum of each block's scaled query (as the MMAs see it),
          // to the lanes whose score columns hold blocks 2t and 2t + 1
          float qs = 0.f;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb)
#pragma unroll
            for (int e = 0; e < PB; ++e) qs += FpMma::unpack(FpMma::pack(qv[hb][e] * sig, 0.f)).x;
          if (D == 64) qs += __shfl_xor_sync(kFullMask, qs, 1);  // two lanes per block
          const int per = 128 / D;                                // lanes per block
          const float s0 = __shfl_sync(kFullMask, qs, (lane & ~3) | ((2 * t * per) & 3));
          const float s1 = __shfl_sync(kFullMask, qs, (lane & ~3) | (((2 * t + 1) * per) & 3));
          q4_corr0 = 2 * t < D / 32 ? 8.f * s0 : 0.f;
          q4_corr1 = 2 * t + 1 < D / 32 ? 8.f * s1 : 0.f;
        } else if (nvalid > 0) {
          // lane (g, t) takes query dims [t D/4, (t+1) D/4) as its B
          // fragments (the query fills every column of N)
          constexpr int QPL = D / 4;
          const int t = lane & 3;
          const uint4* qr = reinterpret_cast<const uint4*>(ks + 2 * S::kTileBytes + t * QPL * (int)sizeof(T));
          float qv[QPL];
#pragma unroll
          for (int c = 0; c < QPL / 8; ++c) {
            float f8[8];
            Chunk<T>::widen(qr[c], f8);
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[8 * c + e] = f8[e];
          }
          float amax = 0.f;
#pragma unroll
          for (int e = 0; e < QPL; ++e) amax = fmaxf(amax, fabsf(qv[e]));
          amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
          // largest element times 2^k in [2^14, 2^15)
          int k = 0;
          if (amax > 0.f) k = min(141 - ((__float_as_int(amax) >> 23) & 0xff), 127);
          const float sig = FpMma::pow2(max(k, -126));
          sc_q = ldexpf(p.scale_log2, -max(k, -126));
#pragma unroll
          for (int kk = 0; kk < NKS; ++kk) {  // the same query in every column
            qb[kk][0] = FpMma::pack(qv[4 * kk] * sig, qv[4 * kk + 1] * sig);
            qb[kk][1] = FpMma::pack(qv[4 * kk + 2] * sig, qv[4 * kk + 3] * sig);
          }
        }
      }
    }
    if constexpr (!kMma) if (first) {
      visit_from_start = cc.t == 0;
#pragma unroll
      for (int g = 0; g < GPW; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[g][e] = 0.f;
      }
      if (nvalid > 0) {
        const unsigned char* qs = ks + 2 * S::kTileBytes;
#pragma unroll
        for (int g = 0; g < GPW; ++g) {
#pragma unroll
          for (int k = 0; k < CPL; ++k) {
            float f[VEC];
            LD::q(qs + g * ROW, sub, k, f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) qf[g][k * VEC + e] = f[e] * p.scale_log2;
          }
        }
      }
    }

    if constexpr (kQ4) {
      if (nvalid > 0) {
        // ---- tensor-core tile of q4_0 rows (layouts: Q4Mma) --------------------
        const int g = lane >> 2, t = lane & 3;
        constexpr int MT = TT / 16;
        constexpr int NBK = D / 32;  // blocks (scales) per row
        constexpr int SCB = D / 16;  // scale bytes per row
        constexpr int PB = D / 8;    // code bytes of a lane's part (scores)
        constexpr int VB = D / 16;   // code bytes a lane reads per row (output)
        float sacc[MT][4];
        float x[MT][2];
        float mx = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          sacc[mt][0] = sacc[mt][1] = sacc[mt][2] = sacc[mt][3] = 0.f;
          uint32_t cw[2][PB / 4];  // code words of the lane's part
          uint32_t wst[2];          // the rows' scale words of blocks 2t, 2t + 1
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const unsigned char* row = ks + (16 * mt + g + 8 * v) * KROW;
            uint32_t sw[NBK / 2];
            if constexpr (D == 128) {
              const uint2 s2 = *reinterpret_cast<const uint2*>(row);
              const uint2 a0 = *reinterpret_cast<const uint2*>(row + SCB + PB * t);
              const uint2 a1 = *reinterpret_cast<const uint2*>(row + SCB + PB * t + 8);
              cw[v][0] = a0.x, cw[v][1] = a0.y, cw[v][2] = a1.x, cw[v][3] = a1.y;
              sw[0] = s2.x, sw[1] = s2.y;
            } else {
              sw[0] = *reinterpret_cast<const uint32_t*>(row);
              cw[v][0] = *reinterpret_cast<const uint32_t*>(row + SCB + PB * t);
              cw[v][1] = *reinterpret_cast<const uint32_t*>(row + SCB + PB * t + 4);
            }
            wst[v] = sw[0];
#pragma unroll
            for (int i = 1; i < NBK / 2; ++i) wst[v] = t == i ? sw[i] : wst[v];
          }
#pragma unroll
          for (int w = 0; w < PB / 4; ++w) {  // k-steps 2w (low four bits) and 2w + 1 (high)
            const uint32_t x0 = cw[0][w], x1 = cw[1][w], y0 = x0 >> 8, y1 = x1 >> 8;
            FpMma::mma(sacc[mt], Q4Mma::lo(x0), Q4Mma::lo(x1), Q4Mma::lo(y0), Q4Mma::lo(y1), qb[2 * w][0],
                       qb[2 * w][1]);
            FpMma::mma(sacc[mt], Q4Mma::hi(x0), Q4Mma::hi(x1), Q4Mma::hi(y0), Q4Mma::hi(y1), qb[2 * w + 1][0],
                       qb[2 * w + 1][1]);
          }
          // columns 2t, 2t + 1 are the partial sums of blocks 2t, 2t + 1
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const auto half_at = [](uint32_t w, int hi) {
              return __half2float(__ushort_as_half((unsigned short)(hi ? w >> 16 : w & 0xffffu)));
            };
            float part = 0.f;
            if (2 * t < NBK)
              part = half_at(wst[v], 0) * fmaf(sacc[mt][2 * v], 16777216.f, -q4_corr0) +
                     half_at(wst[v], 1) * fmaf(sacc[mt][2 * v + 1], 16777216.f, -q4_corr1);
            part += __shfl_xor_sync(kFullMask, part, 1);
            part += __shfl_xor_sync(kFullMask, part, 2);
            const int tok = 16 * mt + g + 8 * v;
            x[mt][v] = tok < nvalid ? part * sc_q : -INFINITY;
            mx = fmaxf(mx, x[mt][v]);
          }
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, off));
        const float mn = fmaxf(m[0], mx);
        const float alpha = exp2f(m[0] - mn);  // 0 on the first tile (m = -inf)
        m[0] = mn;
        float pv[MT][2], ps = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            pv[mt][v] = exp2f(x[mt][v] - mn);
            ps += pv[mt][v];
          }
        l[0] = l[0] * alpha + ps;
        if (alpha != 1.f) {  // warp-uniform
          q4_psum *= alpha;
#pragma unroll
          for (int mm = 0; mm < NKS; ++mm)
#pragma unroll
            for (int e = 0; e < 4; ++e) oa[mm][e] *= alpha;
        }
#pragma unroll
        for (int ks2 = 0; ks2 < MT; ++ks2) {
          // column pair 2t, 2t + 1: p d_t of tokens 16 ks2 + g (+ 8), d_t the
          // V row's scale of block t, as a binary16 high part and remainder
          // (rows past the context: 0, whatever their scale bytes hold)
          uint32_t mv[2];
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const int tok = 16 * ks2 + g + 8 * v;
            const float dvt = t < NBK ? __half2float(*reinterpret_cast<const __half*>(vs + tok * KROW + 2 * t)) : 0.f;
            const float pd = tok < nvalid ? pv[ks2][v] * dvt : 0.f;
            const float ph = __half2float(__float2half_rn(pd));
            mv[v] = t < NBK ? FpMma::pack(ph, pd - ph) : 0u;
            const float2 fed = FpMma::unpack(mv[v]);
            q4_psum += fed.x + fed.y;  // the column pair's sum as the MMAs see it
          }
          const uint32_t b0 = FpMma::trans(mv[0]), b1 = FpMma::trans(mv[1]);
          // code bytes [g VB, (g+1) VB) of token rows 2t, 2t + 1, 2t + 8, 2t + 9
          uint32_t vr[4][VB / 4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tok = 16 * ks2 + 2 * t + (i & 1) + 8 * (i >> 1);
            const unsigned char* vrow = vs + tok * KROW + SCB + VB * g;
            if constexpr (VB == 8) {
              const uint2 a = *reinterpret_cast<const uint2*>(vrow);
              vr[i][0] = a.x, vr[i][1] = a.y;
            } else {
              vr[i][0] = *reinterpret_cast<const uint32_t*>(vrow);
            }
          }
#pragma unroll
          for (int mm = 0; mm < NKS; ++mm) {
            // byte mm of the two token rows of a pair into bytes 0 and 2
            const uint32_t sel = 0x4400u + 0x1111u * (uint32_t)(mm & 3);
            const uint32_t y01 = __byte_perm(vr[0][mm >> 2], vr[1][mm >> 2], sel);
            const uint32_t y23 = __byte_perm(vr[2][mm >> 2], vr[3][mm >> 2], sel);
            FpMma::mma(oa[mm], Q4Mma::lo(y01), Q4Mma::hi(y01), Q4Mma::lo(y23), Q4Mma::hi(y23), b0, b1);
          }
        }
      }
    } else if constexpr (kMma) {
      if (nvalid > 0) {
        // ---- tensor-core tile (layouts: FpMma) --------------------------------
        const int g = lane >> 2, t = lane & 3;
        constexpr int MT = TT / 16;  // 16-token row blocks of the tile
        float sacc[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          sacc[mt][0] = sacc[mt][1] = sacc[mt][2] = sacc[mt][3] = 0.f;
          // bytes [t D/4, (t+1) D/4) of token rows 16 mt + g and 16 mt + g + 8
          uint32_t w0[NKS], w1[NKS];
          const unsigned char* r0 = ks + (16 * mt + g) * KROW;
          const unsigned char* r1 = ks + (16 * mt + g + 8) * KROW;
#pragma unroll
          for (int c = 0; c < NKS / 4; ++c) {
            // 16-byte chunk (D/64) t + c of the rows (stored at chunk ^ (row & 7)
            // when the tile came by swizzled TMA; rows g and g + 8 share row & 7)
            const int ch = (D / 64) * t + c;
            const int pc = S::kTma ? (ch ^ g) : ch;
            const uint4 a = *reinterpret_cast<const uint4*>(r0 + 16 * pc);
            const uint4 b = *reinterpret_cast<const uint4*>(r1 + 16 * pc);
            w0[4 * c] = a.x, w0[4 * c + 1] = a.y, w0[4 * c + 2] = a.z, w0[4 * c + 3] = a.w;
            w1[4 * c] = b.x, w1[4 * c + 1] = b.y, w1[4 * c + 2] = b.z, w1[4 * c + 3] = b.w;
          }
#pragma unroll
          for (int kk = 0; kk < NKS; ++kk)
            FpMma::mma(sacc[mt], FpMma::lo2(w0[kk]), FpMma::lo2(w1[kk]), FpMma::hi2(w0[kk]),
                       FpMma::hi2(w1[kk]), qb[kk][0], qb[kk][1]);
        }
        // every lane (g, t) holds the scores of tokens 16 mt + g + 8 v (all
        // columns are equal)
        float x[MT][2];
        float mx = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const int tok = 16 * mt + g + 8 * v;
            x[mt][v] = tok < nvalid ? sacc[mt][2 * v] * sc_q : -INFINITY;
            mx = fmaxf(mx, x[mt][v]);
          }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, off));
        const float mn = fmaxf(m[0], mx);
        const float alpha = exp2f(m[0] - mn);  // 0 on the first tile (m = -inf)
        m[0] = mn;
        float pv[MT][2], ps = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            pv[mt][v] = exp2f(x[mt][v] - mn);
            ps += pv[mt][v];
          }
        l[0] = l[0] * alpha + ps;  // this lane's tokens (each counted by the 4 lanes of its row)
        if (alpha != 1.f) {        // warp-uniform
#pragma unroll
          for (int mm = 0; mm < NKS; ++mm)
#pragma unroll
            for (int e = 0; e < 4; ++e) oa[mm][e] *= alpha;
        }
        // O^T += V^T P^T, one 16-token k-step at a time
#pragma unroll
        for (int ks2 = 0; ks2 < MT; ++ks2) {
          // P of tokens 16 ks2 + g (+ 8) as a binary16 high part and remainder,
          // as the 8 x 8 matrices M[token][column] (column 0 P_hi, 1 P_lo, the
          // rest 0) in MMA fragment layout; transposed, they are the B fragments
          // of P^T (lane (g, t): column g, tokens 2t, 2t + 1)
          uint32_t mv[2];
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const float ph = __half2float(__float2half_rn(pv[ks2][v]));
            mv[v] = t == 0 ? FpMma::pack(ph, pv[ks2][v] - ph) : 0u;
          }
          const uint32_t b0 = FpMma::trans(mv[0]), b1 = FpMma::trans(mv[1]);
          // bytes [g D/8, (g+1) D/8) of token rows 2t, 2t + 1, 2t + 8, 2t + 9; rows
          // past the context may hold anything (NaN codes): zeros instead
          constexpr int VW = D / 32;  // words per row
          uint32_t vr[4][VW];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tok = 16 * ks2 + 2 * t + (i & 1) + 8 * (i >> 1);
            const unsigned char* vrow = vs + tok * KROW + g * (D / 8);
            if constexpr (VW == 4) {
              // chunk g of the row (at chunk g ^ (tok & 7) when swizzled)
              const uint4 a = *reinterpret_cast<const uint4*>(
                  S::kTma ? vs + tok * KROW + 16 * (g ^ (tok & 7)) : vrow);
              vr[i][0] = a.x, vr[i][1] = a.y, vr[i][2] = a.z, vr[i][3] = a.w;
            } else {
              const uint2 a = *reinterpret_cast<const uint2*>(vrow);
              vr[i][0] = a.x, vr[i][1] = a.y;
            }
            if (tok >= nvalid) {
#pragma unroll
              for (int w = 0; w < VW; ++w) vr[i][w] = 0u;
            }
          }
#pragma unroll
          for (int mm = 0; mm < NKS; ++mm) {
            // head dim bytes 2 mm, 2 mm + 1 of the token pairs, interleaved by token
            const uint32_t sel = (mm & 1) ? 0x7362u : 0x5140u;
            const uint32_t u01 = __byte_perm(vr[0][mm >> 1], vr[1][mm >> 1], sel);
            const uint32_t u23 = __byte_perm(vr[2][mm >> 1], vr[3][mm >> 1], sel);
            FpMma::mma(oa[mm], FpMma::lo2(u01), FpMma::hi2(u01), FpMma::lo2(u23), FpMma::hi2(u23), b0, b1);
          }
        }
      }
    }

    if constexpr (!kMma) if (nvalid > 0) {
      // logits of rows grp, grp+4, grp+8, grp+12
      float x[GPW][RPG];
#pragma unroll
      for (int it = 0; it < RPG; ++it) {
        const int r = it * 4 + grp;
        const unsigned char* krow = ks + r * KROW;
        float acc[GPW];
#pragma unroll
        for (int g = 0; g < GPW; ++g) acc[g] = 0.f;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          float f[VEC];
          LD::kv(krow, sub, k, f);
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
      float pw[GPW][RPG];
#pragma unroll
      for (int g = 0; g < GPW; ++g) {
        float mt = x[g][0];
#pragma unroll
        for (int it = 1; it < RPG; ++it) mt = fmaxf(mt, x[g][it]);
        mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 16));
        const float mn = fmaxf(m[g], mt);
        const float alpha = exp2f(m[g] - mn);  // 0 on the first tile (m = -inf)
        float ps = 0.f;
#pragma unroll
        for (int it = 0; it < RPG; ++it) {
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
      for (int it = 0; it < RPG; ++it) {
        const int r = it * 4 + grp;
        if (r < nvalid) {
          const unsigned char* vrow = vs + r * KROW;
#pragma unroll
          for (int k = 0; k < CPL; ++k) {
            float f[VEC];
            LD::kv(vrow, sub, k, f);
#pragma unroll
            for (int g = 0; g < GPW; ++g)
#pragma unroll
              for (int e = 0; e < VEC; ++e) o[g][k * VEC + e] = fmaf(pw[g][it], f[e], o[g][k * VEC + e]);
          }
        }
      }
    }
    __syncwarp();  // every lane is done with this slot before it is refilled
    if (ci.g < a_end) {
      issue(ci, issued++);
      cursor_next<TT>(ci, p, cap);
    }

    if (last) {
      // ---- end of this warp's visit of segment (cc.s, cc.hg) -----------
      if constexpr (kMma) {
        // into the CUDA-core layout: lane g < 8 holds the row sum and head
        // dims (D/8) g .. + D/8 (lane 4g's columns 0 + 1), the other lanes zeros
        float lt = l[0];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) lt += __shfl_xor_sync(kFullMask, lt, off);
        l[0] = lane < 8 ? lt : 0.f;
        if constexpr (kQ4) {
          // lane g < 8 takes its dims from lane (g, block of g): low bits of
          // byte e (e < DPL/2) are row g, high bits row g + 8 of m-tile e % (DPL/2)
          // (codes entered as q 2^-24 and 16 q 2^-24: scale back, less 8 x
          // the P column pair's sum)
          constexpr int HALF = DPL / 2;
          const int src = 4 * (lane & 7) + (lane & 7) / (256 / D);
          float ps8 = q4_psum;
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) ps8 += __shfl_xor_sync(kFullMask, ps8, off);
          ps8 *= 8.f;
#pragma unroll
          for (int e = 0; e < DPL; ++e) {
            const int mm = e % HALF;
            const float v = e < HALF ? fmaf(oa[mm][0] + oa[mm][1], 16777216.f, -ps8)
                                     : fmaf(oa[mm][2] + oa[mm][3], 1048576.f, -ps8);
            const float w = __shfl_sync(kFullMask, v, src);
            o[0][e] = lane < 8 ? w : 0.f;
          }
        } else {
#pragma unroll
          for (int e = 0; e < DPL; ++e) {
            const float v = oa[e >> 1][2 * (e & 1)] + oa[e >> 1][2 * (e & 1) + 1];
            const float w = __shfl_sync(kFullMask, v, 4 * (lane & 7));
            o[0][e] = lane < 8 ? w : 0.f;
          }
        }
      }
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
      const size_t row0 = (size_t)cc.s * H + (size_t)cc.hg * GPW;
      if (visit_from_start && cc.t == cc.nt - 1) {
        // the whole segment was ours: write the output rows
        if (grp == 0) {
#pragma unroll
          for (int g = 0; g < GPW; ++g) {
            float inv = cc.L > 0 ? 1.f / l[g] : 0.f;
            if constexpr (kQuant) inv *= p.v_scale;
            unsigned char* orow = static_cast<unsigned char*>(p.out) + (row0 + g) * ROW;
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
              float f[VEC];
#pragma unroll
              for (int e = 0; e < VEC; ++e) f[e] = o[g][k * VEC + e] * inv;
              LD::out(orow, sub, k, f);
            }
          }
        }
      } else {
        // one piece of a segment shared with neighbouring warps
        const int slot = cc.g - cc.t <= a_begin ? 0 : 1;  // segment is this warp's first visit -> 0
        const size_t base = ((size_t)wid * 2 + slot) * GPW;
        if (grp == 0) {
#pragma unroll
          for (int g = 0; g < GPW; ++g) {
            const float inv = 1.f / l[g];
            float4* po = reinterpret_cast<float4*>(p.ws_o + (base + g) * D);
#pragma unroll
            for (int k = 0; k < CPL; ++k)
#pragma unroll
              for (int e = 0; e < VEC; e += 4)
                po[LD::dim(sub, k, e) / 4] =
                    make_float4(o[g][k * VEC + e] * inv, o[g][k * VEC + e + 1] * inv,
                                o[g][k * VEC + e + 2] * inv, o[g][k * VEC + e + 3] * inv);
          }
        }
        if (lane == 0) {
#pragma unroll
          for (int g = 0; g < GPW; ++g) p.ws_ml[base + g] = make_float2(m[g], l[g]);
        }
        __syncwarp();  // the partial's writes precede lane 0's release below
        const long long seg_start = cc.g - cc.t;
        const long long seg_end = seg_start + cc.nt;
        // warps whose ranges meet this segment: w(x) = ceil((x+1) Weff / T) - 1
        const long long w_first = ((seg_start + 1) * Weff + Ttot - 1) / Ttot - 1;
        const long long w_last = (seg_end * Weff + Ttot - 1) / Ttot - 1;
        int is_last = 0;
        if (lane == 0) {
          int32_t* ctr = p.ws_counter + (size_t)cc.s * HG + cc.hg;
          const int prev = atomic_add_acq_rel_gpu(ctr, 1);
          is_last = prev == (int)(w_last - w_first);
          if (is_last) *ctr = 0;  // every piece has counted: leave the counter zero
        }
        is_last = __shfl_sync(kFullMask, is_last, 0);
        if (is_last) {
          __syncwarp();  // the other pieces' partials, acquired by lane 0, are visible to all lanes
          constexpr int DL = D / 32;  // output dims per lane in the merge
#pragma unroll
          for (int g = 0; g < GPW; ++g) {
            float M = -INFINITY;
            for (long long w = w_first; w <= w_last; ++w) {
              const int sl = (w == w_first && w * Ttot / Weff < seg_start) ? 1 : 0;
              M = fmaxf(M, __ldcg(p.ws_ml + ((size_t)w * 2 + sl) * GPW + g).x);
            }
            float Ls = 0.f, O[DL];
#pragma unroll
            for (int e = 0; e < DL; ++e) O[e] = 0.f;
            for (long long w = w_first; w <= w_last; ++w) {
              const int sl = (w == w_first && w * Ttot / Weff < seg_start) ? 1 : 0;
              const size_t idx = ((size_t)w * 2 + sl) * GPW + g;
              const float2 v = __ldcg(p.ws_ml + idx);
              const float wt = v.y * exp2f(v.x - M);  // l_j 2^(m_j - M); partials hold o_j / l_j
              Ls += wt;
              const float* po = p.ws_o + idx * D + lane * DL;
#pragma unroll
              for (int e = 0; e < DL; ++e) O[e] += __ldcg(po + e) * wt;
            }
            T* orow = static_cast<T*>(p.out) + (row0 + g) * D + lane * DL;
            if constexpr (kQuant) {
              const float vs_l = p.v_scale / Ls;
#pragma unroll
              for (int e = 0; e < DL; ++e) store_elem(orow + e, O[e] * vs_l);
            } else {
#pragma unroll
              for (int e = 0; e < DL; ++e) store_elem(orow + e, O[e] / Ls);
            }
          }
        }
      }
    }
    cursor_next<TT>(cc, p, cap);
  }
}

// Launch one instantiation as a persistent grid sized to the device.
template <typename T, int D, int GPW, typename KT = T>
cudaError_t launch_pa_decode(const DecodeParams& p, cudaStream_t stream) {
  using S = DecodeShape<T, D, GPW, KT>;
  static int grid_of_device[64] = {0};  // cached per device ordinal (0 = not yet known)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int grid = (dev >= 0 && dev < 64) ? __atomic_load_n(&grid_of_device[dev], __ATOMIC_ACQUIRE) : 0;
  if (grid == 0) {
    e = cudaFuncSetAttribute(pa_decode_kernel<T, D, GPW, KT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::kSmemBytes);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pa_decode_kernel<T, D, GPW, KT>,
                                                      S::kWarps * 32, S::kSmemBytes);
    if (e != cudaSuccess) return e;
    grid = sms * (per_sm > 0 ? per_sm : 1);
    if (grid > kMaxDecodeWarps / S::kWarps) grid = kMaxDecodeWarps / S::kWarps;
    if (dev >= 0 && dev < 64) __atomic_store_n(&grid_of_device[dev], grid, __ATOMIC_RELEASE);
  }
  CUtensorMap kmap, vmap;
  memset(&kmap, 0, sizeof(kmap));
  memset(&vmap, 0, sizeof(vmap));
  if constexpr (S::kTma) {
    const uint64_t rows = (uint64_t)p.num_blocks * p.num_kv_heads * p.block_size;
    // the TMA row coordinate (one box past the pool included) must fit in int32
    if (rows + S::kTileTokensT > 0x7fffffffull) return cudaErrorNotSupported;
    const int box_rows = p.block_size < S::kTileTokensT ? p.block_size : S::kTileTokensT;
    e = encode_pool_bytes_map(&kmap, p.k_cache, rows, box_rows);
    if (e != cudaSuccess) return e;
    e = encode_pool_bytes_map(&vmap, p.v_cache, rows, box_rows);
    if (e != cudaSuccess) return e;
  }
  pa_decode_kernel<T, D, GPW, KT><<<grid, S::kWarps * 32, S::kSmemBytes, stream>>>(kmap, vmap, p);
  return cudaGetLastError();
}

using DecodeLauncher = cudaError_t (*)(const DecodeParams&, cudaStream_t);

// Per-dtype tables, defined in decode_<dtype>.cu. gpw_index: 0 -> 1, 1 -> 2, 2 -> 4.
DecodeLauncher decode_launcher_f32(int head_dim, int gpw_index);
DecodeLauncher decode_launcher_f16(int head_dim, int gpw_index);
DecodeLauncher decode_launcher_bf16(int head_dim, int gpw_index);
// fp8 e4m3 caches with 16-bit queries (decode_fp8.cu): q_is_bf16 0 -> fp16 queries.
DecodeLauncher decode_launcher_fp8(int q_is_bf16, int head_dim, int gpw_index);
// q4_0 caches with 16-bit queries, one query head per warp (decode_q4.cu).
DecodeLauncher decode_launcher_q4(int q_is_bf16, int head_dim);

}  // namespace pkv
