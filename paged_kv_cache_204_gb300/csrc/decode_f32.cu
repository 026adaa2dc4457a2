// Instantiations of the paged decode kernel for float storage.
#include "decode.cuh"
#include "decode_grouped.cuh"

namespace pkv {

DecodeLauncher decode_launcher_f32(int head_dim, int gpw_index) {
  using T = float;
  static const DecodeLauncher d64[3] = {launch_pa_decode<T, 64, 1>, launch_pa_decode<T, 64, 2>,
                                         launch_pa_decode<T, 64, 4>};
  static const DecodeLauncher d128[3] = {launch_pa_decode<T, 128, 1>, launch_pa_decode<T, 128, 2>,
                                          launch_pa_decode<T, 128, 4>};
  if (gpw_index < 0 || gpw_index > 2) return nullptr;
  if (head_dim == 64) return d64[gpw_index];
  if (head_dim == 128) return d128[gpw_index];
  return nullptr;
}

GroupedLauncher grouped_launcher_f32(int head_dim, int gpw_index) {
  using T = float;
  static const GroupedLauncher d64[3] = {launch_pa_decode_grouped<T, 64, 1>, launch_pa_decode_grouped<T, 64, 2>,
                                          launch_pa_decode_grouped<T, 64, 4>};
  static const GroupedLauncher d128[3] = {launch_pa_decode_grouped<T, 128, 1>,
                                           launch_pa_decode_grouped<T, 128, 2>,
                                           launch_pa_decode_grouped<T, 128, 4>};
  if (gpw_index < 0 || gpw_index > 2) return nullptr;
  if (head_dim == 64) return d64[gpw_index];
  if (head_dim == 128) return d128[gpw_index];
  return nullptr;
}

}  // namespace pkv
