// Instantiations of the paged decode kernel for q4_0 caches read with
// binary16 or bfloat16 queries (outputs in the query type), one query head
// per warp.
#include "decode.cuh"

namespace pkv {

DecodeLauncher decode_launcher_q4(int q_is_bf16, int head_dim) {
  using H = __half;
  using B = __nv_bfloat16;
  if (head_dim == 64) return q_is_bf16 ? launch_pa_decode<B, 64, 1, Q4Row> : launch_pa_decode<H, 64, 1, Q4Row>;
  if (head_dim == 128) return q_is_bf16 ? launch_pa_decode<B, 128, 1, Q4Row> : launch_pa_decode<H, 128, 1, Q4Row>;
  return nullptr;
}

}  // namespace pkv
