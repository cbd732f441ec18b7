// t3_tc_fwd.cu -- instantiates and launches the pair pipeline for the forward
// product (its own translation unit, so that the products compile in parallel).
#include <atomic>

#include "t3_tc2_launch.cuh"

namespace t3 {

int launch_tc2_fwd(const tc2::Params& p, const CUtensorMap& ma, const CUtensorMap& mw,
                   const CUtensorMap& mo, int grid, cudaStream_t s) {
  return launch_tc2_op<kOpFwd>(p, ma, mw, mo, grid, s);
}

int prepare_tc2_fwd() { return prepare_tc2_op<kOpFwd>(); }

int launch_tc2_fwd_bf16(const tc2::Params& p, const CUtensorMap& ma, const CUtensorMap& mw,
                        const CUtensorMap& mo, int grid, cudaStream_t s) {
  constexpr int kSmem = tc2::Layout<kOpFwd, 2>::smem_alloc;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return T3_ECUDA;
  static std::atomic<bool> attr_done[64];
  if (dev < 0 || dev >= 64) return T3_EDEVICE;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(tc2::tc2_kernel<kOpFwd, tc2::kModeBf16, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
      return T3_ECUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  tc2::tc2_kernel<kOpFwd, tc2::kModeBf16, false><<<grid, tc2::kThreads, kSmem, s>>>(p, ma, mw, mo);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
