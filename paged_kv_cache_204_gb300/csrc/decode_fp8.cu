// Instantiations of the paged decode kernel for fp8 e4m3 caches read with
// binary16 or bfloat16 queries (outputs in the query type).
#include "decode.cuh"

namespace pkv {

DecodeLauncher decode_launcher_fp8(int q_is_bf16, int head_dim, int gpw_index) {
  using E = __nv_fp8_e4m3;
  using H = __half;
  using B = __nv_bfloat16;
  static const DecodeLauncher h64[3] = {launch_pa_decode<H, 64, 1, E>, launch_pa_decode<H, 64, 2, E>,
                                         launch_pa_decode<H, 64, 4, E>};
  static const DecodeLauncher h128[3] = {launch_pa_decode<H, 128, 1, E>, launch_pa_decode<H, 128, 2, E>,
                                          launch_pa_decode<H, 128, 4, E>};
  static const DecodeLauncher b64[3] = {launch_pa_decode<B, 64, 1, E>, launch_pa_decode<B, 64, 2, E>,
                                         launch_pa_decode<B, 64, 4, E>};
  static const DecodeLauncher b128[3] = {launch_pa_decode<B, 128, 1, E>, launch_pa_decode<B, 128, 2, E>,
                                          launch_pa_decode<B, 128, 4, E>};
  if (gpw_index < 0 || gpw_index > 2) return nullptr;
  if (head_dim == 64) return q_is_bf16 ? b64[gpw_index] : h64[gpw_index];
  if (head_dim == 128) return q_is_bf16 ? b128[gpw_index] : h128[gpw_index];
  return nullptr;
}

}  // namespace pkv
