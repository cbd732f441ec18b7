// t3_quant.cu -- bf16 activations to int8 with one scale per row.
//
// What it computes: the step before the products.  "spec(igla): hslm_bwd_ptx
// -- HSLM backward dX and dW as int8 tensor-core PTX written by t27" feeds the
// int8 kernels from quantized tensors and names the scales the host must use
// (dX per row); the quantizer itself is not given.  The plainest reading,
// symmetric absmax per row, written out:
//   amax[m]  = max_k |x[m][k]|
//   scale[m] = amax[m] / 127,   inv = 127 / amax[m]   (each a float division,
//                                                      rounded to nearest)
//   q[m][k]  = rint(x[m][k] * inv), the product rounded to a float first,
//              rint to nearest with ties to even, clamped to [-127, 127]
// and a row of zeros gives q = 0, scale = 0.  x * scale[m] then reproduces
// q's row scale in the scaled products (t3_dequant_i32).
//
// Why this shape.  It reads 2 bytes and writes 1 byte per element: HBM-bound.
// One warp per row: the first pass takes the row's absolute maximum (16-byte
// loads of 8 bf16 where rows allow, a warp shuffle reduction), the second
// reads the row again (now in L1/L2) and writes 8 int8 per 8-byte store.
#include <cuda_bf16.h>

#include <cstdint>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {
namespace qz {

constexpr int kWarps = 8;

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ int8_t quant1(float x, float inv) {
  int q = __float2int_rn(__fmul_rn(x, inv));  // nearest, ties to even
  q = q > 127 ? 127 : (q < -127 ? -127 : q);
  return static_cast<int8_t>(q);
}

// kCodes: write the int8 codes (else only the scales, and `inv`: the inverse
// scales 127 / amax of the same division, for a product that quantizes the
// rows itself).
template <bool kCodes>
__global__ void __launch_bounds__(32 * kWarps) quant_rows_kernel(const uint16_t* __restrict__ x,
                                                                 int8_t* __restrict__ q,
                                                                 float* __restrict__ scale,
                                                                 float* __restrict__ inv_out,
                                                                 int64_t M, int64_t K, int vec) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t m = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); m < M;
       m += warps) {
    const uint16_t* row = x + m * K;
    int8_t* qrow = q + m * K;
    float amax = 0.0f;
    if (vec) {
      for (int64_t k = 8 * lane; k < K; k += 256) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + k));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[j] & 0xFFFFu)));
          amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[j] >> 16)));
        }
      }
    } else {
      for (int64_t k = lane; k < K; k += 32) amax = fmaxf(amax, fabsf(bf16_bits_to_f32(row[k])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float inv = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
    if (lane == 0) scale[m] = amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 0.0f;
    if (!kCodes) {
      if (lane == 0) inv_out[m] = inv;
      continue;
    }
    if (vec) {
      for (int64_t k = 8 * lane; k < K; k += 256) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + k));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t lo = static_cast<uint8_t>(quant1(bf16_bits_to_f32(w[j] & 0xFFFFu), inv));
          const uint32_t hi = static_cast<uint8_t>(quant1(bf16_bits_to_f32(w[j] >> 16), inv));
          out[j >> 1] |= (lo | (hi << 8)) << (16 * (j & 1));
        }
        *reinterpret_cast<uint2*>(qrow + k) = make_uint2(out[0], out[1]);
      }
    } else {
      for (int64_t k = lane; k < K; k += 32) qrow[k] = quant1(bf16_bits_to_f32(row[k]), inv);
    }
  }
}

}  // namespace qz

int launch_quant_rows(const void* x, int8_t* q, float* scale, int64_t M, int64_t K, int sms,
                      cudaStream_t s) {
  const int vec = (K % 8 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(q) % 8 == 0);
  const int64_t blocks = (M + qz::kWarps - 1) / qz::kWarps;
  const int64_t cap = 8 * static_cast<int64_t>(sms > 0 ? sms : 1);
  const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
  qz::quant_rows_kernel<true><<<grid, 32 * qz::kWarps, 0, s>>>(static_cast<const uint16_t*>(x), q,
                                                              scale, nullptr, M, K, vec);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

int launch_row_scales(const void* x, float* scale, float* inv, int64_t M, int64_t K, int sms,
                      cudaStream_t s) {
  const int vec = (K % 8 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0);
  const int64_t blocks = (M + qz::kWarps - 1) / qz::kWarps;
  const int64_t cap = 8 * static_cast<int64_t>(sms > 0 ? sms : 1);
  const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
  qz::quant_rows_kernel<false><<<grid, 32 * qz::kWarps, 0, s>>>(static_cast<const uint16_t*>(x),
                                                               nullptr, scale, inv, M, K, vec);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
