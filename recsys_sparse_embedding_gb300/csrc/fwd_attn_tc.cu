// Instantiations of the forward kernel with the bf16 tcgen05 attention MLP.
#include "launch.cuh"

namespace dsf {

int launch_attn_tc(int D, bool bf16, const FwdParams& p, cudaStream_t s) {
  if (D == 16 && !bf16) return launch_fwd<Cfg<16, false, 0, true>>(p, s);
  if (D == 16 && bf16) return launch_fwd<Cfg<16, true, 0, true>>(p, s);
  if (D == 64 && bf16) return launch_fwd<Cfg<64, true, 0, true>>(p, s);
  return 2;
}

int grid_attn_tc(int D, bool bf16, int dev) {
  if (D == 16 && !bf16) return grid_for_device<Cfg<16, false, 0, true>>(dev);
  if (D == 16 && bf16) return grid_for_device<Cfg<16, true, 0, true>>(dev);
  if (D == 64 && bf16) return grid_for_device<Cfg<64, true, 0, true>>(dev);
  return 0;
}

}  // namespace dsf
