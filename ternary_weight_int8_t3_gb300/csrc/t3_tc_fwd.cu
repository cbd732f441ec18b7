// t3_tc_fwd.cu -- instantiates and launches the pair pipeline for the forward
// product (its own translation unit, so that the products compile in parallel).
#include "t3_tc2_launch.cuh"

namespace t3 {

int launch_tc2_fwd(const tc2::Params& p, const CUtensorMap& ma, const CUtensorMap& mw,
                   const CUtensorMap& mo, int grid, cudaStream_t s) {
  return launch_tc2_op<kOpFwd>(p, ma, mw, mo, grid, s);
}

int prepare_tc2_fwd() { return prepare_tc2_op<kOpFwd>(); }

}  // namespace t3
