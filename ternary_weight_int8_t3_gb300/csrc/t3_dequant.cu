// t3_dequant.cu -- scaling an exact int32 product into float or bf16 output.
//
// What it computes: the step right after the products in "spec(igla):
// hslm_bwd_ptx -- HSLM backward dX and dW as int8 tensor-core PTX written by
// t27", where the host rescales the integer results (dX by a scale per row,
// dW by scales per column of X and of dY), and the "+=" forms of the products
// named there.  Written out: y = ((float)x * row_scale[r]) * col_scale[c],
// each product rounded to the nearest float (ties to even), a NULL scale
// vector standing for ones; the output is y as float, y rounded to bf16
// (nearest, ties to even), or old + y as float (one rounding).
//
// Why this shape.  One read of x (and of the old output for "+="), one write:
// HBM-bound.  Each thread handles four consecutive elements of a row (16-byte
// loads and stores where the row allows), grid-stride over the matrix.  x and
// out may be the same buffer (float output): every element is read and then
// written by the same thread.
#include <cuda_bf16.h>

#include <cstdint>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {
namespace dq {

constexpr int kThreads = 256;

__device__ __forceinline__ float scaled(int32_t x, float rs, float cs) {
  // explicit roundings: no fused multiply-add may merge these steps
  return __fmul_rn(__fmul_rn(__int2float_rn(x), rs), cs);
}

template <int KIND>
__device__ __forceinline__ void put(void* out, int64_t i, float y) {
  if (KIND == T3_OUT_F32) {
    static_cast<float*>(out)[i] = y;
  } else if (KIND == T3_OUT_BF16) {
    static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(y);
  } else {
    float* o = static_cast<float*>(out);
    o[i] = __fadd_rn(o[i], y);
  }
}

// Groups of four consecutive elements of one row; `vec` when every row starts
// 16-byte aligned in x and in out (then cols % 4 == 0 and a group never
// crosses a row).
template <int KIND>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const int32_t* x, void* out,
                                                           int64_t rows, int64_t cols,
                                                           const float* row_scale,
                                                           const float* col_scale, int vec) {
  const int64_t total = rows * cols;
  const int64_t groups = (total + 3) / 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
       g += stride) {
    const int64_t i0 = 4 * g;
    if (vec) {
      const int64_t r = i0 / cols, c = i0 - r * cols;
      const float rs = row_scale ? __ldg(row_scale + r) : 1.0f;
      const int4 xv = *reinterpret_cast<const int4*>(x + i0);
      float4 cs = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
      if (col_scale) cs = *reinterpret_cast<const float4*>(col_scale + c);
      float4 y = make_float4(scaled(xv.x, rs, cs.x), scaled(xv.y, rs, cs.y),
                             scaled(xv.z, rs, cs.z), scaled(xv.w, rs, cs.w));
      if (KIND == T3_OUT_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + i0) = y;
      } else if (KIND == T3_OUT_F32_ADD) {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + i0);
        const float4 old = *o;
        *o = make_float4(__fadd_rn(old.x, y.x), __fadd_rn(old.y, y.y), __fadd_rn(old.z, y.z),
                         __fadd_rn(old.w, y.w));
      } else {
        __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(out) + i0);
        o[0] = __nv_bfloat162(__float2bfloat16_rn(y.x), __float2bfloat16_rn(y.y));
        o[1] = __nv_bfloat162(__float2bfloat16_rn(y.z), __float2bfloat16_rn(y.w));
      }
    } else {
      for (int64_t i = i0; i < i0 + 4 && i < total; ++i) {
        const int64_t r = i / cols, c = i - r * cols;
        const float rs = row_scale ? __ldg(row_scale + r) : 1.0f;
        const float cs = col_scale ? __ldg(col_scale + c) : 1.0f;
        put<KIND>(out, i, scaled(x[i], rs, cs));
      }
    }
  }
}

}  // namespace dq

int launch_dequant(const int32_t* x, void* out, int64_t rows, int64_t cols, const float* row_scale,
                   const float* col_scale, int kind, int sms, cudaStream_t s) {
  const int64_t total = rows * cols;
  const int64_t groups = (total + 3) / 4;
  const int out_align = (kind == T3_OUT_BF16) ? 8 : 16;
  const int vec = (cols % 4 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(out) % out_align == 0) &&
                  (col_scale == nullptr || reinterpret_cast<uintptr_t>(col_scale) % 16 == 0);
  const int64_t cap = 8 * static_cast<int64_t>(sms > 0 ? sms : 1) * (2048 / dq::kThreads);
  int64_t grid = (groups + dq::kThreads - 1) / dq::kThreads;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const unsigned g = static_cast<unsigned>(grid);
  if (kind == T3_OUT_F32)
    dq::dequant_kernel<T3_OUT_F32><<<g, dq::kThreads, 0, s>>>(x, out, rows, cols, row_scale,
                                                              col_scale, vec);
  else if (kind == T3_OUT_BF16)
    dq::dequant_kernel<T3_OUT_BF16><<<g, dq::kThreads, 0, s>>>(x, out, rows, cols, row_scale,
                                                               col_scale, vec);
  else
    dq::dequant_kernel<T3_OUT_F32_ADD><<<g, dq::kThreads, 0, s>>>(x, out, rows, cols, row_scale,
                                                                  col_scale, vec);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
