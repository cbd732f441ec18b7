// t3_tc2_launch.cuh -- launches the fwd/dX pair pipeline for one product: the
// kernel instantiation for the operands' load mode, or, when the schedule is
// split (stream-K pieces add onto rows a zeroing grid clears just before), the
// split instantiation with the programmatic-dependent-launch attribute, so
// that it overlaps the zeroing grid and waits for it only before its first
// output write.
#pragma once
#include <atomic>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {

// Sets the kernels' shared-memory attributes, once per device.
template <int OP>
int prepare_tc2_op() {
  constexpr int kSmem = tc2::Layout<OP>::smem_alloc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return T3_ECUDA;
  static std::atomic<bool> attr_done[64];
  if (dev < 0 || dev >= 64) return T3_EDEVICE;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(tc2::tc2_kernel<OP, tc2::kModeTma, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(tc2::tc2_kernel<OP, tc2::kModeTma, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(tc2::tc2_kernel<OP, tc2::kModeWGlobal, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(tc2::tc2_kernel<OP, tc2::kModeAGlobal, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
      return T3_ECUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  return T3_OK;
}

template <int OP>
int launch_tc2_op(const tc2::Params& p, const CUtensorMap& ma, const CUtensorMap& mw,
                  const CUtensorMap& mo, int grid, cudaStream_t s) {
  constexpr int kSmem = tc2::Layout<OP>::smem_alloc;
  const int st = prepare_tc2_op<OP>();
  if (st != T3_OK) return st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(tc2::kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.dp_tiles < p.tiles_r * p.tiles_c) {
    if (p.mode != tc2::kModeTma) return T3_EINVAL;  // the split schedule takes TMA operands
    if (cudaLaunchKernelEx(&cfg, tc2::tc2_kernel<OP, tc2::kModeTma, true>, p, ma, mw, mo) !=
        cudaSuccess)
      return T3_ECUDA;
    return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
  }
  if (p.mode == tc2::kModeTma)
    tc2::tc2_kernel<OP, tc2::kModeTma, false><<<grid, tc2::kThreads, kSmem, s>>>(p, ma, mw, mo);
  else if (p.mode == tc2::kModeWGlobal)
    tc2::tc2_kernel<OP, tc2::kModeWGlobal, false><<<grid, tc2::kThreads, kSmem, s>>>(p, ma, mw, mo);
  else
    tc2::tc2_kernel<OP, tc2::kModeAGlobal, false><<<grid, tc2::kThreads, kSmem, s>>>(p, ma, mw, mo);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
