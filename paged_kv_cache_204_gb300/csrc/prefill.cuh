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
// Work: one CTA of 8 warps per (128-query tile, sequence, query head); a warp
// owns 16 query rows. K/V tiles of 64 tokens are gathered through the block
// table with 16-byte cp.async copies into a double-buffered, XOR-swizzled
// shared-memory layout (rows past the context are zero-filled without a
// read) and fed to the tensor cores with ldmatrix:
//   S = Q K^T   mma.sync m16n8k16, fp32 accumulation;
//   online softmax in base 2 on the accumulators (causal mask by select);
//   O += P V    P from the S accumulators as a high + low 16-bit pair (two
//               MMAs) so that the probabilities keep fp32-level accuracy.
#pragma once

#include "common.cuh"

namespace pkv {

constexpr int kPfRows = 128;   // query rows per CTA (8 warps x 16)
constexpr int kPfTokens = 64;  // K/V tokens per tile
constexpr int kPfWarps = 8;

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
};

template <typename T>
struct PfMma;
template <>
struct PfMma<__half> {
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
template <>
struct PfMma<__nv_bfloat16> {
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

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
// 16-byte asynchronous copy; src_bytes 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16_zfill(void* smem, const void* gmem, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte chunk c of row r in a [rows][D] tile: chunks are
// XOR-swizzled by the row's low 3 bits so that 8 consecutive rows at the same
// chunk fall on different banks (ldmatrix reads them conflict-free).
template <int D>
__device__ __forceinline__ int pf_off(int r, int c) {
  return r * (D * 2) + ((c ^ (r & 7)) << 4);
}

template <typename T, int D>
struct PrefillShape {
  static constexpr int kTileBytes = kPfTokens * D * 2;
  static constexpr int kQBytes = kPfRows * D * 2;
  static constexpr int kSmemBytes = kQBytes + 4 * kTileBytes;  // Q, then K and V for two stages
  static_assert(D % 64 == 0, "head_dim 64 or 128");
};

template <typename T, int D>
__global__ void __launch_bounds__(kPfWarps * 32, 2) pa_prefill_kernel(const PrefillParams p) {
  using S = PrefillShape<T, D>;
  using M = PfMma<T>;
  constexpr int CH = D / 8;   // 16-byte chunks per row
  constexpr int KS = D / 16;  // k-steps of q.k
  constexpr int NT = D / 8;   // n-tiles of the output
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* qs = smem;
  unsigned char* kv = smem + S::kQBytes;  // stage s: K at kv + 2s*tile, V at kv + (2s+1)*tile

  const int tile = blockIdx.x, s = blockIdx.y, h = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int L = __ldg(p.context_lens + s);
  const int q0 = __ldg(p.query_start + s), n = __ldg(p.query_start + s + 1) - q0;
  if (L < 0 || L > p.max_blocks_per_seq * p.block_size || n < 0 || n > L) {
    if (tid == 0 && tile == 0 && h == 0) set_err(p.dev_err, PKV_DEV_ERR_CONTEXT_LEN);
    return;
  }
  const int row0 = tile * kPfRows;
  if (row0 >= n) return;  // this tile has no queries
  const int rows = min(kPfRows, n - row0);
  const int first_pos = L - n + row0;         // position of the tile's first query
  const int kv_end = first_pos + rows;        // tokens the tile's queries can see
  const int ntiles = (kv_end + kPfTokens - 1) / kPfTokens;
  const int kvh = h / p.group;
  const T* qg = static_cast<const T*>(p.q);
  const T* kg = static_cast<const T*>(p.k_cache);
  const T* vg = static_cast<const T*>(p.v_cache);
  const int32_t* bt = p.block_tables + (size_t)s * p.max_blocks_per_seq;
  const int bs = p.block_size;

  // ---- async loads -----------------------------------------------------------
  for (int i = tid; i < kPfRows * CH; i += kPfWarps * 32) {
    const int r = i / CH, c = i % CH;
    const bool ok = r < rows;
    const T* src = qg + ((size_t)(q0 + row0 + (ok ? r : 0)) * p.num_heads + h) * D + c * 8;
    cp_async16_zfill(qs + pf_off<D>(r, c), src, ok ? 16 : 0);
  }
  auto load_kv = [&](int j, int stage) {
    unsigned char* kd = kv + (2 * stage) * S::kTileBytes;
    unsigned char* vd = kd + S::kTileBytes;
    for (int i = tid; i < kPfTokens * CH; i += kPfWarps * 32) {
      const int r = i / CH, c = i % CH;
      const int t = j * kPfTokens + r;
      int id = 0;
      bool ok = t < kv_end;
      if (ok) {
        id = __ldg(bt + t / bs);
        if (id < 0 || id >= p.num_blocks) {
          set_err(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
          ok = false;
          id = 0;
        }
      }
      const size_t off = (((size_t)id * p.num_kv_heads + kvh) * bs + (ok ? t % bs : 0)) * D + c * 8;
      cp_async16_zfill(kd + pf_off<D>(r, c), kg + off, ok ? 16 : 0);
      cp_async16_zfill(vd + pf_off<D>(r, c), vg + off, ok ? 16 : 0);
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  // ---- per-warp state: rows w*16 + g and w*16 + g + 8 --------------------------
  const int wr = warp * 16;
  const int pos_a = first_pos + wr + g, pos_b = pos_a + 8;  // query positions of this thread's rows
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

  for (int j = 0; j < ntiles; ++j) {
    if (j + 1 < ntiles) {
      load_kv(j + 1, (j + 1) & 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    const unsigned char* ks = kv + (2 * (j & 1)) * S::kTileBytes;
    const unsigned char* vs = ks + S::kTileBytes;
    const int t0 = j * kPfTokens;

    // S = Q K^T over the tile's 64 tokens: 8 n-tiles of 8 tokens
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t qa[4];  // this k-step's query fragment, reloaded per tile (keeps registers for occupancy)
      {
        const int r = wr + (lane & 15), c = 2 * kk + (lane >> 4);
        ldsm_x4(qa, qs + pf_off<D>(r, c));
      }
#pragma unroll
      for (int np = 0; np < 4; ++np) {  // pairs of n-tiles
        uint32_t b[4];
        const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3), c = 2 * kk + ((lane >> 3) & 1);
        ldsm_x4(b, ks + pf_off<D>(r, c));
        M::run(sc[2 * np], qa, b[0], b[1]);
        M::run(sc[2 * np + 1], qa, b[2], b[3]);
      }
    }
    // scale, causal mask, running max
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = t0 + nt * 8 + 2 * t4 + e;
        sc[nt][e] = t <= pos_a ? sc[nt][e] * p.scale_log2 : -INFINITY;
        sc[nt][2 + e] = t <= pos_b ? sc[nt][2 + e] * p.scale_log2 : -INFINITY;
        mx_a = fmaxf(mx_a, sc[nt][e]);
        mx_b = fmaxf(mx_b, sc[nt][2 + e]);
      }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(kFullMask, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(kFullMask, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(kFullMask, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(kFullMask, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    // a row with nothing visible yet keeps m = -inf: subtract 0 instead
    const float base_a = mn_a == -INFINITY ? 0.f : mn_a, base_b = mn_b == -INFINITY ? 0.f : mn_b;
    const float al_a = exp2f(m_a - base_a), al_b = exp2f(m_b - base_b);
    m_a = mn_a;
    m_b = mn_b;
    float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      sc[nt][0] = exp2f(sc[nt][0] - base_a);
      sc[nt][1] = exp2f(sc[nt][1] - base_a);
      sc[nt][2] = exp2f(sc[nt][2] - base_b);
      sc[nt][3] = exp2f(sc[nt][3] - base_b);
      ps_a += sc[nt][0] + sc[nt][1];
      ps_b += sc[nt][2] + sc[nt][3];
    }
    l_a = l_a * al_a + ps_a;  // per-thread partial sums; the quad is summed at the end
    l_b = l_b * al_b + ps_b;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      o[nt][0] *= al_a;
      o[nt][1] *= al_a;
      o[nt][2] *= al_b;
      o[nt][3] *= al_b;
    }
    // O += P V: k-steps of 16 tokens (n-tiles 2k, 2k+1 of S), P as hi + lo
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) {
      uint32_t ph[4], pl[4];
      const float* p0 = sc[2 * k2];
      const float* p1 = sc[2 * k2 + 1];
      const float src[4][2] = {{p0[0], p0[1]}, {p0[2], p0[3]}, {p1[0], p1[1]}, {p1[2], p1[3]}};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ph[i] = M::pack(src[i][0], src[i][1]);
        const float2 hv = M::unpack(ph[i]);
        pl[i] = M::pack(src[i][0] - hv.x, src[i][1] - hv.y);
      }
#pragma unroll
      for (int cp = 0; cp < NT / 2; ++cp) {  // pairs of output n-tiles (chunks 2cp, 2cp+1)
        uint32_t b[4];
        const int r = k2 * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), c = 2 * cp + (lane >> 4);
        ldsm_x4_trans(b, vs + pf_off<D>(r, c));
        M::run(o[2 * cp], ph, b[0], b[1]);  // high halves first: dependent MMAs two apart
        M::run(o[2 * cp + 1], ph, b[2], b[3]);
        M::run(o[2 * cp], pl, b[0], b[1]);
        M::run(o[2 * cp + 1], pl, b[2], b[3]);
      }
    }
    __syncthreads();  // every warp is done with this stage before it is refilled
  }

  // ---- normalise and store ---------------------------------------------------------
  l_a += __shfl_xor_sync(kFullMask, l_a, 1);
  l_a += __shfl_xor_sync(kFullMask, l_a, 2);
  l_b += __shfl_xor_sync(kFullMask, l_b, 1);
  l_b += __shfl_xor_sync(kFullMask, l_b, 2);
  const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f, inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
  const int ra = wr + g, rb = ra + 8;
  T* og = static_cast<T*>(p.out);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int d = nt * 8 + 2 * t4;
    if (ra < rows) {
      const uint32_t u = M::pack(o[nt][0] * inv_a, o[nt][1] * inv_a);
      *reinterpret_cast<uint32_t*>(og + ((size_t)(q0 + row0 + ra) * p.num_heads + h) * D + d) = u;
    }
    if (rb < rows) {
      const uint32_t u = M::pack(o[nt][2] * inv_b, o[nt][3] * inv_b);
      *reinterpret_cast<uint32_t*>(og + ((size_t)(q0 + row0 + rb) * p.num_heads + h) * D + d) = u;
    }
  }
}

template <typename T, int D>
cudaError_t launch_pa_prefill(const PrefillParams& p, int max_query_len, cudaStream_t stream) {
  using S = PrefillShape<T, D>;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
    e = cudaFuncSetAttribute(pa_prefill_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
  }
  const dim3 grid((max_query_len + kPfRows - 1) / kPfRows, p.num_seqs, p.num_heads);
  pa_prefill_kernel<T, D><<<grid, kPfWarps * 32, S::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

using PrefillLauncher = cudaError_t (*)(const PrefillParams&, int, cudaStream_t);
PrefillLauncher prefill_launcher(int is_bf16, int head_dim);

}  // namespace pkv
