// t3_small.cu -- the three products for small problems on the CUDA cores,
// for operands of any alignment.
//
// What it computes: the forward of "t27c PTX backend: ternary x int8 GEMM
// kernel emitted by a .t27 spec (int8 mma.sync), ptx-run glue" (section "What
// this adds": C[m][n] = sum_k A[m][k] W[k][n], W from 2-bit codes) and kernels
// 1 and 2 of "spec(igla): hslm_bwd_ptx -- HSLM backward dX and dW as int8
// tensor-core PTX written by t27" (dX[m][k] = sum_n dY[m][n] W[k][n] on the same
// codes, dW[k][n] = sum_m A[m][k] dY[m][n]), exactly in int32.
//
// Why this shape.  The CTA-pair pipelines move 256-row tiles through 128-
// element stages; a product of a few hundred million multiply-adds, such as
// the pages' HSLM layers (widths 243 and 729 at 27 and 1782 rows), leaves
// most of their tiles, stages and SMs idle, and rows of 243 or 729 bytes are
// not TMA-addressable, so their operands arrive through byte-wise loads.
// Here every CTA owns a 64 x 64 output tile and a contiguous range of the
// reduction (split over several CTAs, which add atomically onto a zeroed
// output, when the tiles alone would not fill the GPU):
//   * per 64-element chunk of the reduction it stages both operands in shared
//     memory as rows of int8 words along the reduction: the output's rows as
//     X, its columns as Y.  fwd: X = A (reordered within each 16-element group
//     as the decode orders the codes), Y = W decoded with one byte permute per
//     4 codes on the table {0, +1, -1, 0}.  dX: X = dY, Y = Wᵀ: four packed
//     rows at a time, the codes of one k gathered into a word.  dW: X = Aᵀ,
//     Y = dYᵀ through 4 x 4 byte transposes (byte permutes);
//   * each of the 256 threads keeps a 4 x 4 block of int32 sums and adds four
//     products per dp4a;
//   * staged rows are 80 bytes apart, so that the 16 rows a warp reads at once
//     fall on distinct 16-byte bank groups in pairs.
#include <atomic>
#include <cstdint>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {
namespace smp {

constexpr int kTile = 64;           // output rows and columns per CTA
constexpr int kChunk = 64;          // reduction elements per staged chunk
constexpr int kWords = kChunk / 4;  // int8x4 words per staged row
constexpr int kPitch = kWords + 4;  // words between staged rows (80 bytes)
constexpr int kThreads = 256;

// The product a launch computes.
enum Op { kFwd = 1, kDx = 2, kDw = 3 };

struct Params {
  const int8_t* x;     // fwd: A [M][K]; dX: dY [M][N]; dW: A [M][K]
  const int8_t* y;     // dW: dY [M][N]
  const uint8_t* wp;   // fwd, dX: Wp [N][KB]
  int32_t* out;        // fwd: C [M][N]; dX: dX [M][K]; dW: dW [K][N]
  int64_t M, N, K, KB;
  int64_t rows, cols;  // the output's shape
  int64_t red;         // the reduction's length
  int64_t tiles_c;     // tiles along the output's columns
  int64_t chunks;      // 64-element chunks of the reduction
  int split;           // CTAs per output tile (> 1: atomic adds onto zeros)
  int x_vec;           // fwd/dX: rows of x as 16-byte loads; dW: rows of A as words
  int y_vec;           // dW: rows of dY as words
};

// 16 bytes of row `row` (of `len` bytes, `nrows` rows) from column c; 0 past
// the rows or the row's end.
__device__ __forceinline__ uint4 load16(const int8_t* base, int64_t nrows, int64_t len, int vec,
                                        int64_t row, int64_t c) {
  uint32_t b[4] = {0u, 0u, 0u, 0u};
  if (row < nrows) {
    const int8_t* p = base + row * len + c;
    if (vec && c + 16 <= len) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
      return v;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (c + j < len) b[j >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(__ldg(p + j))) << (8 * (j & 3));
  }
  return make_uint4(b[0], b[1], b[2], b[3]);
}

// 4 bytes of row `row` from column c (a multiple of 4); 0 past the edges.
__device__ __forceinline__ uint32_t load4(const int8_t* base, int64_t nrows, int64_t len, int vec,
                                          int64_t row, int64_t c) {
  if (row >= nrows) return 0u;
  const int8_t* p = base + row * len + c;
  if (vec && c + 4 <= len) return __ldg(reinterpret_cast<const uint32_t*>(p));
  uint32_t w = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (c + j < len) w |= static_cast<uint32_t>(static_cast<uint8_t>(__ldg(p + j))) << (8 * j);
  return w;
}

// 4 bytes of packed weights, row n, bytes [b, b + 4); 0 past the edges.
__device__ __forceinline__ uint32_t load_codes4(const uint8_t* wp, int64_t N, int64_t KB, int64_t n,
                                                int64_t b) {
  if (n >= N) return 0u;
  const uint8_t* p = wp + n * KB + b;
  uint32_t w = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (b + j < KB) w |= static_cast<uint32_t>(__ldg(p + j)) << (8 * j);
  return w;
}

// Four 2-bit codes, one per byte (bits 0-1) -> four int8 weights: 1 -> +1,
// 2 -> -1, 0 and 3 -> 0.
__device__ __forceinline__ uint32_t codes_to_s8x4(uint32_t c) {
  const uint32_t lo = c & 0x01010101u, hi = (c >> 1) & 0x01010101u;
  return (lo & ~hi) | ((hi & ~lo) * 0xFFu);
}

// Column j of the 4 x 4 byte block whose rows are r0..r3 (byte j of each).
__device__ __forceinline__ void transpose4x4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3,
                                             uint32_t (&c)[4]) {
  const uint32_t lo01 = prmt(r0, r1, 0x5140u), lo23 = prmt(r2, r3, 0x5140u);
  const uint32_t hi01 = prmt(r0, r1, 0x7362u), hi23 = prmt(r2, r3, 0x7362u);
  c[0] = prmt(lo01, lo23, 0x5410u);
  c[1] = prmt(lo01, lo23, 0x7632u);
  c[2] = prmt(hi01, hi23, 0x5410u);
  c[3] = prmt(hi01, hi23, 0x7632u);
}

// The four int8-weight words of 16 codes (code i at bits 2i of x), in the
// order even codes 0..6 | 8..14, odd codes 1..7 | 9..15.
__device__ __forceinline__ void decode16_s8(uint32_t x, uint32_t (&w)[4]) {
  const uint32_t ev = x & 0x33333333u, od = (x >> 2) & 0x33333333u;
  w[0] = prmt(0x00FF0100u, 0u, ev);
  w[1] = prmt(0x00FF0100u, 0u, ev >> 16);
  w[2] = prmt(0x00FF0100u, 0u, od);
  w[3] = prmt(0x00FF0100u, 0u, od >> 16);
}

// Stages chunk [r0, r0 + 64) of the reduction for output rows [row0, +64) (X)
// and columns [col0, +64) (Y).
template <int OP>
__device__ __forceinline__ void stage(const Params& p, int64_t row0, int64_t col0, int64_t r0,
                                      uint32_t (*xs)[kPitch], uint32_t (*ys)[kPitch], int t) {
  if constexpr (OP == kFwd || OP == kDx) {
    // X: row t/4, 16 reduction elements from 16 (t % 4)
    const int row = t >> 2, seg = t & 3;
    const int64_t len = (OP == kFwd) ? p.K : p.N;
    const uint4 v = load16(p.x, p.M, len, p.x_vec, row0 + row, r0 + 16 * seg);
    uint4* dst = reinterpret_cast<uint4*>(&xs[row][4 * seg]);
    if constexpr (OP == kFwd)  // the decode's order: even elements, then odd
      *dst = make_uint4(prmt(v.x, v.y, 0x6420u), prmt(v.z, v.w, 0x6420u), prmt(v.x, v.y, 0x7531u),
                        prmt(v.z, v.w, 0x7531u));
    else
      *dst = v;
  }
  if constexpr (OP == kFwd) {
    // Y: weight row col0 + t/4, its codes for k in [r0 + 16 (t % 4), +16)
    const int row = t >> 2, seg = t & 3;
    uint32_t w[4];
    decode16_s8(load_codes4(p.wp, p.N, p.KB, col0 + row, r0 / 4 + 4 * seg), w);
    *reinterpret_cast<uint4*>(&ys[row][4 * seg]) = make_uint4(w[0], w[1], w[2], w[3]);
  } else if constexpr (OP == kDx) {
    // Y: k in [col0, +64) as rows, n along the words: packed rows n0 + 4 g .. +3,
    // byte col0/4 + b (k = col0 + 4 b .. +3)
    const int g = t >> 4, b = t & 15;
    const int64_t n = r0 + 4 * g, kb = col0 / 4 + b;
    uint32_t x = 0u;
#pragma unroll
    for (int r = 0; r < 4; ++r)
      if (n + r < p.N && kb < p.KB) x |= static_cast<uint32_t>(__ldg(p.wp + (n + r) * p.KB + kb)) << (8 * r);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) ys[4 * b + kk][g] = codes_to_s8x4((x >> (2 * kk)) & 0x03030303u);
  } else {
    // dW: X = Aᵀ (k as rows), Y = dYᵀ (n as rows): a 4 m x 4 k (or 4 n) block
    // per thread, transposed so that each word holds four consecutive m
    const int g = t >> 4, b = t & 15;
    const int64_t m = r0 + 4 * g;
    uint32_t c[4];
    transpose4x4(load4(p.x, p.M, p.K, p.x_vec, m, row0 + 4 * b),
                 load4(p.x, p.M, p.K, p.x_vec, m + 1, row0 + 4 * b),
                 load4(p.x, p.M, p.K, p.x_vec, m + 2, row0 + 4 * b),
                 load4(p.x, p.M, p.K, p.x_vec, m + 3, row0 + 4 * b), c);
#pragma unroll
    for (int j = 0; j < 4; ++j) xs[4 * b + j][g] = c[j];
    transpose4x4(load4(p.y, p.M, p.N, p.y_vec, m, col0 + 4 * b),
                 load4(p.y, p.M, p.N, p.y_vec, m + 1, col0 + 4 * b),
                 load4(p.y, p.M, p.N, p.y_vec, m + 2, col0 + 4 * b),
                 load4(p.y, p.M, p.N, p.y_vec, m + 3, col0 + 4 * b), c);
#pragma unroll
    for (int j = 0; j < 4; ++j) ys[4 * b + j][g] = c[j];
  }
}

template <int OP>
__global__ void __launch_bounds__(kThreads) small_kernel(const Params p) {
  __shared__ __align__(16) uint32_t xs[kTile][kPitch];
  __shared__ __align__(16) uint32_t ys[kTile][kPitch];
  const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
  const int64_t tile = static_cast<int64_t>(blockIdx.x) / p.split;
  const int part = static_cast<int>(static_cast<int64_t>(blockIdx.x) % p.split);
  const int64_t row0 = (tile / p.tiles_c) * kTile, col0 = (tile % p.tiles_c) * kTile;
  const int64_t c0 = p.chunks * part / p.split, c1 = p.chunks * (part + 1) / p.split;
  int32_t acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0;
  for (int64_t c = c0; c < c1; ++c) {
    stage<OP>(p, row0, col0, c * kChunk, xs, ys, t);
    __syncthreads();
#pragma unroll
    for (int w4 = 0; w4 < kWords / 4; ++w4) {
      uint4 xv[4], yv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = *reinterpret_cast<const uint4*>(&xs[ty + 16 * i][4 * w4]);
#pragma unroll
      for (int j = 0; j < 4; ++j) yv[j] = *reinterpret_cast<const uint4*>(&ys[tx + 16 * j][4 * w4]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = __dp4a(static_cast<int>(xv[i].x), static_cast<int>(yv[j].x), acc[i][j]);
          acc[i][j] = __dp4a(static_cast<int>(xv[i].y), static_cast<int>(yv[j].y), acc[i][j]);
          acc[i][j] = __dp4a(static_cast<int>(xv[i].z), static_cast<int>(yv[j].z), acc[i][j]);
          acc[i][j] = __dp4a(static_cast<int>(xv[i].w), static_cast<int>(yv[j].w), acc[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = row0 + ty + 16 * i;
    if (r >= p.rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t col = col0 + tx + 16 * j;
      if (col >= p.cols) continue;
      int32_t* dst = p.out + r * p.cols + col;
      if (p.split > 1)
        atomicAdd(dst, acc[i][j]);
      else
        *dst = acc[i][j];
    }
  }
}

}  // namespace smp

int launch_small(int op, const int8_t* x, const int8_t* y, const uint8_t* wp, int32_t* out,
                 int64_t M, int64_t N, int64_t K, int sms, cudaStream_t s) {
  smp::Params p{};
  p.x = x;
  p.y = y;
  p.wp = wp;
  p.out = out;
  p.M = M;
  p.N = N;
  p.K = K;
  p.KB = (K + 3) / 4;
  p.rows = (op == smp::kDw) ? K : M;
  p.cols = (op == smp::kFwd || op == smp::kDw) ? N : K;
  p.red = (op == smp::kFwd) ? K : (op == smp::kDx) ? N : M;
  p.tiles_c = (p.cols + smp::kTile - 1) / smp::kTile;
  const int64_t tiles = (p.rows + smp::kTile - 1) / smp::kTile * p.tiles_c;
  p.chunks = (p.red + smp::kChunk - 1) / smp::kChunk;
  // enough CTAs for about four per SM, each at least two chunks of the
  // reduction when the tiles alone fall short
  int64_t split = 1;
  if (tiles < 4 * static_cast<int64_t>(sms)) {
    split = (4 * static_cast<int64_t>(sms) + tiles - 1) / tiles;
    const int64_t most = p.chunks / 2 > 1 ? p.chunks / 2 : 1;
    if (split > most) split = most;
  }
  if (tiles * split > 2147483647LL) return T3_EINVAL;
  p.split = static_cast<int>(split);
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x);
  if (op == smp::kDw) {
    p.x_vec = (K % 4 == 0) && (xa % 4 == 0);
    p.y_vec = (N % 4 == 0) && (reinterpret_cast<uintptr_t>(y) % 4 == 0);
  } else {
    const int64_t len = (op == smp::kFwd) ? K : N;
    p.x_vec = (len % 16 == 0) && (xa % 16 == 0);
  }
  if (split > 1 &&
      cudaMemsetAsync(out, 0, static_cast<size_t>(p.rows) * p.cols * sizeof(int32_t), s) !=
          cudaSuccess)
    return T3_ECUDA;
  const dim3 grid(static_cast<unsigned>(tiles * split));
  if (op == smp::kFwd)
    smp::small_kernel<smp::kFwd><<<grid, smp::kThreads, 0, s>>>(p);
  else if (op == smp::kDx)
    smp::small_kernel<smp::kDx><<<grid, smp::kThreads, 0, s>>>(p);
  else
    smp::small_kernel<smp::kDw><<<grid, smp::kThreads, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
