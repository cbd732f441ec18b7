// t3_tc_fwd.cu -- instantiates and launches the pair pipeline for one product.
#include <atomic>
#include "t3_internal.h"
#include "t3.h"

namespace t3 {

int launch_tc2_fwd(const tc2::Params& p, const CUtensorMap& ma, const CUtensorMap& mw,
                   const CUtensorMap& mo, int grid, cudaStream_t s) {
  constexpr int kSmem = tc2::Layout<kOpFwd>::smem_alloc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return T3_ECUDA;
  static std::atomic<bool> attr_done[64];
  if (dev < 0 || dev >= 64) return T3_EDEVICE;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(tc2::tc2_kernel<kOpFwd, tc2::kModeTma>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(tc2::tc2_kernel<kOpFwd, tc2::kModeWGlobal>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(tc2::tc2_kernel<kOpFwd, tc2::kModeAGlobal>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
      return T3_ECUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  if (p.mode == tc2::kModeTma)
    tc2::tc2_kernel<kOpFwd, tc2::kModeTma><<<grid, tc2::kThreads, kSmem, s>>>(p, ma, mw, mo);
  else if (p.mode == tc2::kModeWGlobal)
    tc2::tc2_kernel<kOpFwd, tc2::kModeWGlobal><<<grid, tc2::kThreads, kSmem, s>>>(p, ma, mw, mo);
  else
    tc2::tc2_kernel<kOpFwd, tc2::kModeAGlobal><<<grid, tc2::kThreads, kSmem, s>>>(p, ma, mw, mo);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
