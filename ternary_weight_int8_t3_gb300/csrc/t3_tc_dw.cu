// t3_tc_dw.cu -- instantiates and launches the pair pipeline for one product.
#include <atomic>
#include "t3_internal.h"
#include "t3.h"

namespace t3 {

int launch_dw2(const dw2::Params& p, const CUtensorMap& ma, const CUtensorMap& mdy,
               const CUtensorMap& mo, int grid, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return T3_ECUDA;
  static std::atomic<bool> attr_done[64];
  if (dev < 0 || dev >= 64) return T3_EDEVICE;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(dw2::dw2_kernel<dw2::kChunkElems, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dw2::SMEM_ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(dw2::dw2_kernel<dw2::kChunkElems, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dw2::SMEM_ALLOC) != cudaSuccess)
      return T3_ECUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(dw2::kThreads, 1, 1);
  cfg.dynamicSmemBytes = dw2::SMEM_ALLOC;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le =
      p.global_ops ? cudaLaunchKernelEx(&cfg, dw2::dw2_kernel<dw2::kChunkElems, true>, p, ma, mdy, mo)
                   : cudaLaunchKernelEx(&cfg, dw2::dw2_kernel<dw2::kChunkElems, false>, p, ma, mdy,
                                        mo);
  if (le != cudaSuccess) return T3_ECUDA;
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
