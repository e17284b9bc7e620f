// Instantiations of the forward kernel without attention (EmbeddingBag only).
#include "launch.cuh"

namespace dsf {

int launch_pool(int D, bool bf16, const FwdParams& p, cudaStream_t s) {
  if (D == 16 && !bf16) return launch_fwd<Cfg<16, false, 1, false>>(p, s);
  if (D == 16 && bf16) return launch_fwd<Cfg<16, true, 1, false>>(p, s);
  if (D == 64 && !bf16) return launch_fwd<Cfg<64, false, 1, false>>(p, s);
  if (D == 64 && bf16) return launch_fwd<Cfg<64, true, 1, false>>(p, s);
  return 2;
}

int grid_pool(int D, bool bf16, int dev) {
  if (D == 16 && !bf16) return grid_for_device<Cfg<16, false, 1, false>>(dev);
  if (D == 16 && bf16) return grid_for_device<Cfg<16, true, 1, false>>(dev);
  if (D == 64 && !bf16) return grid_for_device<Cfg<64, false, 1, false>>(dev);
  if (D == 64 && bf16) return grid_for_device<Cfg<64, true, 1, false>>(dev);
  return 0;
}

}  // namespace dsf
