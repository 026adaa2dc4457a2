// Instantiations of the paged prefill kernel (binary16 and bfloat16).
#include "prefill.cuh"

namespace pkv {

PrefillLauncher prefill_launcher(int is_bf16, int head_dim) {
  if (head_dim == 64) return is_bf16 ? launch_pa_prefill<__nv_bfloat16, 64> : launch_pa_prefill<__half, 64>;
  if (head_dim == 128) return is_bf16 ? launch_pa_prefill<__nv_bfloat16, 128> : launch_pa_prefill<__half, 128>;
  return nullptr;
}

}  // namespace pkv
