// t3_internal.h -- declarations shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include "t3_tc_gemm.cuh"

namespace t3 {

// Launch the tensor-core pipeline for one product.  Returns a t3_status.
int launch_tc_fwd(const tc::Params& p, const CUtensorMap& ma, const CUtensorMap& mb,
                  const CUtensorMap& mo, int grid, cudaStream_t s);
int launch_tc_dx(const tc::Params& p, const CUtensorMap& ma, const CUtensorMap& mb,
                  const CUtensorMap& mo, int grid, cudaStream_t s);
int launch_tc_dw(const tc::Params& p, const CUtensorMap& ma, const CUtensorMap& mb,
                  const CUtensorMap& mo, int grid, cudaStream_t s);

}  // namespace t3
