// t3_common.cuh -- definitions shared by the tensor-core pipelines.
//
// The products are those of "t27c PTX backend: ternary x int8 GEMM kernel
// emitted by a .t27 spec (int8 mma.sync), ptx-run glue" ("What this adds":
// C = A.W, W from 2-bit codes decoded as (c & 1) - ((c >> 1) & 1)) and of
// "spec(igla): hslm_bwd_ptx -- HSLM backward dX and dW as int8 tensor-core
// PTX written by t27" (kernels 1 and 2: dX = dY.W^T, dW = A^T.dY).  This file
// holds the product tags and the small device helpers the pair pipelines
// (t3_tc2.cuh, t3_tc2_dw.cuh) and the small-M kernel (t3_skinny.cu) share.
#pragma once
#include <cstdint>
#include "t3_ptx.cuh"

namespace t3 {

enum OpKind : int { kOpFwd = 1, kOpDx = 2, kOpDw = 3 };

namespace tc {

// Plain-load copy of one box (rows x cols bytes) into shared memory with zero
// fill outside the source: the producer's fallback when TMA is not allowed
// (rows of any alignment, so single-byte loads).  Each lane gathers 8 words
// before storing any of them, so that their loads are in flight together
// instead of one global round trip per word.
__device__ __forceinline__ void manual_box(uint8_t* dst, const uint8_t* src, int64_t ld,
                                           int64_t src_rows, int64_t src_cols, int64_t y0,
                                           int64_t x0, int box_rows, int box_cols, int lane) {
  constexpr int kBatch = 8;
  const int wpr = box_cols / 4;
  const int total = box_rows * wpr;
  for (int base = lane; base < total; base += 32 * kBatch) {
    uint32_t words[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int idx = base + 32 * b;
      const int r = idx / wpr, cw = idx % wpr;
      const int64_t y = y0 + r, x = x0 + 4 * cw;
      uint32_t word = 0;
      if (idx < total && y < src_rows) {
        const uint8_t* rowp = src + y * ld;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (x + j < src_cols) word |= static_cast<uint32_t>(__ldg(rowp + x + j)) << (8 * j);
      }
      words[b] = word;
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int idx = base + 32 * b;
      if (idx < total) {
        const int r = idx / wpr, cw = idx % wpr;
        *reinterpret_cast<uint32_t*>(dst + r * box_cols + 4 * cw) = words[b];
      }
    }
  }
}

// Four int8 (one word) -> two f16x2 words, exact: bias each byte to
// u = b + 128, place it under the f16 exponent of 1024 (0x64uu is 1024 + u)
// and subtract 1152.
__device__ __forceinline__ void s8x4_to_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
  const uint32_t y = x ^ 0x80808080u;
  lo = hsub2(prmt(y, 0x64646464u, 0x4140u), 0x64806480u);
  hi = hsub2(prmt(y, 0x64646464u, 0x4342u), 0x64806480u);
}

// High byte of the f16 weight for code c = byte c of this word: 0 -> 0x00,
// 1 -> 0x3C (+1.0), 2 -> 0xBC (-1.0), 3 -> 0x00; the low byte is always 0.
constexpr uint32_t kF16HiTable = 0x00BC3C00u;

// Byte offset of 16-byte chunk c of row r in a tile of 128-byte rows in the
// 128-byte swizzle (chunk c of row r sits at c ^ (r mod 8)).
__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// f32 accumulator bits -> int32.
__device__ __forceinline__ int32_t f32_bits_to_i32(uint32_t bits) {
  return __float2int_rn(__uint_as_float(bits));  // the value is an exact integer
}

// How out_block32 writes: store, add into elements only this warp writes
// (read, add, write), or add atomically (other CTAs add into the same ones).
enum OutBlockKind { kOutStore = 0, kOutAdd = 1, kOutAtomicAdd = 2 };

// The row pass of out_block32, out of line: it runs only for outputs TMA
// cannot address, and kept inline its loop adds to the register pressure of
// every pipeline instantiation.
static __device__ __noinline__ void out_rows32(const uint32_t* scratch, int lane, int32_t* out, int64_t ld,
                                               int64_t row0, int64_t rows, int64_t col0, int64_t cols,
                                               int kind) {
  const bool col_ok = col0 + lane < cols;
  const int64_t left = rows - row0;
  const int nrows = left < 32 ? static_cast<int>(left) : 32;
  int32_t* dst = out + row0 * ld + col0 + lane;
  for (int r = 0; r < nrows; ++r, dst += ld) {
    const int32_t x = f32_bits_to_i32(scratch[r * 33 + lane]);
    if (!col_ok) continue;
    if (kind == kOutStore)
      *dst = x;
    else if (kind == kOutAdd)
      *dst += x;
    else
      atomicAdd(dst, x);
  }
}

// A warp's 32 x 32 block of exact sums (f32 bit patterns) into int32 rows of
// any alignment: lane l holds row row0 + l, columns col0 .. col0 + 31, in v.
// The block is transposed through `scratch` (33 x 32 words of this warp's
// own shared memory; the odd pitch keeps both passes free of bank conflicts)
// so that each instruction writes 32 consecutive columns of one row, one or
// two memory transactions, instead of touching 32 rows.  Rows from `rows`
// on and columns from `cols` on are left alone.
__device__ __forceinline__ void out_block32(uint32_t* scratch, const uint32_t (&v)[32], int lane,
                                            int32_t* out, int64_t ld, int64_t row0, int64_t rows,
                                            int64_t col0, int64_t cols, int kind) {
  __syncwarp();  // the previous block's reads of scratch are done
#pragma unroll
  for (int j = 0; j < 32; ++j) scratch[lane * 33 + j] = v[j];
  __syncwarp();
  out_rows32(scratch, lane, out, ld, row0, rows, col0, cols, kind);
}

}  // namespace tc
}  // namespace t3
