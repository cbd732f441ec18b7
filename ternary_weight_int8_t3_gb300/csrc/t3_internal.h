// t3_internal.h -- declarations shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include "t3_common.cuh"
#include "t3_tc2.cuh"
#include "t3_tc2_dw.cuh"

namespace t3 {

// Tensor maps for 2-D row-major matrices (row stride = cols elements).  They
// return false, leaving *map zeroed, when TMA cannot be used (base or row
// stride not 16-byte aligned, or the driver refuses).
bool make_u8_map_tiled(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                       int box_rows, int box_cols, bool swizzle128 = false);
bool make_i32_map_tiled(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                        int box_rows, int box_cols, bool swizzle128);

// CTA-pair pipeline for the forward and dX products.  With a split schedule
// (p.dp_tiles below the tile count) the rows the stream-K pieces add into must
// have been zeroed by launch_zero_pdl just before on `s`.
int launch_tc2_fwd(const tc2::Params& p, const CUtensorMap& ma, const CUtensorMap& mw,
                   const CUtensorMap& mo, int grid, cudaStream_t s);
int launch_tc2_dx(const tc2::Params& p, const CUtensorMap& ma, const CUtensorMap& mw,
                  const CUtensorMap& mo, int grid, cudaStream_t s);
// The same kernels' launch attributes, set once per device (launch_tc2_* call
// these too); the split schedule calls them before it queues its zeroing grid.
int prepare_tc2_fwd();
int prepare_tc2_dx();

// The forward on bf16 activations quantized in the pair pipeline's converters
// (tc2::kModeBf16; p.row_inv holds the rows' inverse scales).
int launch_tc2_fwd_bf16(const tc2::Params& p, const CUtensorMap& ma, const CUtensorMap& mw,
                        const CUtensorMap& mo, int grid, cudaStream_t s);

// Zeroes out[0, n) on `s` as a programmatic dependent of the work before it:
// it waits for that work to complete, then lets the next grid launch early.
int launch_zero_pdl(int32_t* out, int64_t n, int sms, cudaStream_t s);

// CTA-pair pipeline for dW (A, dY and dW all TMA-able).  Adds onto dW, which
// launch_zero_pdl has cleared just before on `s`; launched as its programmatic
// dependent.
int launch_dw2(const dw2::Params& p, const CUtensorMap& ma, const CUtensorMap& mdy,
               const CUtensorMap& mo, int grid, cudaStream_t s);

// Device packer: int8 w [K][N] -> Wp [N][ceil(K/4)] on `s`; a value outside
// {-1, 0, +1} packs as 0 and records (9 << 8) | 6 in *err.
int launch_pack_device(const int8_t* w, uint8_t* wp, int64_t K, int64_t N, int sms, int* err,
                       cudaStream_t s);

// bf16 x [M][K] -> int8 q [M][K] and a float scale per row (absmax), on `s`.
int launch_quant_rows(const void* x, int8_t* q, float* scale, int64_t M, int64_t K, int sms,
                      cudaStream_t s);

// The row quantizer's scales only: scale = amax / 127 and inv = 127 / amax per
// row of bf16 x [M][K] (0 and 0 for a zero row), on `s`.
int launch_row_scales(const void* x, float* scale, float* inv, int64_t M, int64_t K, int sms,
                      cudaStream_t s);

// out[r][c] = scaled int32 x[r][c] (T3_OUT_* kind), on `s`.
int launch_dequant(const int32_t* x, void* out, int64_t rows, int64_t cols, const float* row_scale,
                   const float* col_scale, int kind, int sms, cudaStream_t s);

// Forward for M <= 8 on the CUDA cores (t3_gemv.cu); T3_EINVAL, with nothing
// launched, when A's copy would not fit its shared-memory budget.
int launch_gemv_fwd(const int8_t* A, const uint8_t* Wp, int32_t* C, int64_t M, int64_t N,
                    int64_t K, int sms, cudaStream_t s);

// The three products on the CUDA cores for small problems, any alignment
// (t3_small.cu): op 1 C = A.W (x = A, wp = Wp), 2 dX = dY.Wᵀ (x = dY, wp = Wp),
// 3 dW = Aᵀ.dY (x = A, y = dY); int32 output, written whole (zeroed first
// when the reduction is split over CTAs).
int launch_small(int op, const int8_t* x, const int8_t* y, const uint8_t* wp, int32_t* out,
                 int64_t M, int64_t N, int64_t K, int sms, cudaStream_t s);

// Small-M forward (M <= 32) on the tensor cores.
int launch_skinny_fwd(const int8_t* A, const uint8_t* Wp, int32_t* C, int64_t M, int64_t N,
                      int64_t K, int sms, int* err, cudaStream_t s);

}  // namespace t3
