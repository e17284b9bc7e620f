// Launch of the EmbeddingBag pooling kernels (emb_bag_pool and its no-alloc
// variant): the range totals, then the pooling, with the same grid (one wave
// of resident CTAs), on the caller's stream.
#include <atomic>

#include "bag_kernel.cuh"
#include "launch.cuh"

namespace dsf {
namespace {

template <class C>
int bag_grid(int dev) {
  static std::atomic<int> cache[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return 0;
  const int known = cache[dev].load(std::memory_order_acquire);
  if (known > 0) return known;
  int nsm = 0, occ = 0;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, bag::bag_kernel<C>, bag::kThreads, 0) != cudaSuccess)
    return 0;
  if (occ < 1) return 0;
  long long g = (long long)nsm * occ;
  if (g > bag::kMaxWords) g = bag::kMaxWords;
  cache[dev].store(int(g), std::memory_order_release);
  return int(g);
}

template <class C>
int bag_launch(const FwdParams& p, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 3;
  const int G = bag_grid<C>(dev);
  if (G <= 0) return 2;
  bag::bag_totals_kernel<<<G, bag::kThreads, 0, stream>>>(p);
  bag::bag_kernel<C><<<G, bag::kThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace

int launch_pool(int D, bool bf16, const FwdParams& p, cudaStream_t s) {
  if (D == 16 && !bf16) return bag_launch<bag::Cfg<16, false>>(p, s);
  if (D == 16 && bf16) return bag_launch<bag::Cfg<16, true>>(p, s);
  if (D == 64 && !bf16) return bag_launch<bag::Cfg<64, false>>(p, s);
  if (D == 64 && bf16) return bag_launch<bag::Cfg<64, true>>(p, s);
  return 2;
}

int grid_pool(int D, bool bf16, int dev) {
  if (D == 16 && !bf16) return bag_grid<bag::Cfg<16, false>>(dev);
  if (D == 16 && bf16) return bag_grid<bag::Cfg<16, true>>(dev);
  if (D == 64 && !bf16) return bag_grid<bag::Cfg<64, false>>(dev);
  if (D == 64 && bf16) return bag_grid<bag::Cfg<64, true>>(dev);
  return 0;
}

}  // namespace dsf
