// t3_gemv.cu -- the forward for a few activation rows (M <= 8) on the CUDA
// cores: C = A . W at the rate of reading the packed weights.
//
// What it computes: the forward product of "t27c PTX backend: ternary x int8
// GEMM kernel emitted by a .t27 spec (int8 mma.sync), ptx-run glue", section
// "What this adds": C[m][n] = sum_k A[m][k] W[k][n], W from 2-bit codes.
//
// Why this shape.  With one to eight activation rows the product is a matrix-
// vector product: a byte of packed weights carries 4 weights and 4 M
// multiply-adds.  The tensor-core path (t3_skinny.cu) pays a fixed cost per
// 16 KB unit (decode into TMEM, barrier hand-offs between producer, decoders
// and MMA issuers) and per call (TMEM, clusters, the partial exchange) that a
// few rows do not need.  Here:
//   * every SM takes an equal contiguous share of the weight rows; each warp
//     takes 4 of them at a time (2 for more than 4 activation rows): lane l
//     reads the 16-byte chunks l, l + 32, ... of each row's ceil(K/4) bytes (each load instruction reads 512 contiguous bytes of a
//     row), 64 codes per chunk, and one read of the activations serves all
//     the rows;
//   * a 16-code word becomes four words of int8 weights with one byte permute
//     each on the table {0, +1, -1, 0}: its even codes (k = 0, 2, .., 14), then
//     its odd codes, selected by the 2-bit codes as nibbles;
//   * every CTA first copies A into shared memory in that same order within
//     each 16-element group, zero past K (so pad codes and code 3 meet a zero
//     or a zero weight), and each lane multiplies with dp4a: four int8 x int8
//     products summed into an int32, exactly;
//   * the lanes' int32 sums of a row are added with warp shuffles and one lane
//     per (row, m) stores C[m][n].
// Launch: a programmatic dependent of whatever precedes it on the stream; it
// reads A and Wp and writes C only after griddepcontrol.wait, and before the
// wait asks its share of 16-byte aligned packed rows into L2.
#include <atomic>
#include <cstdint>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {
namespace gv {

constexpr int kWarps = 16;                 // 512 threads, one CTA per SM
constexpr uint32_t kWeightTable = 0x00FF0100u;  // code c -> byte c: 0, +1, -1, 0
constexpr int64_t kMaxSmem = 64 * 1024;    // A's copy: M * ceil(K/64) * 64 bytes at most
constexpr int64_t kPrefetchBytes = 48ll << 20;  // weights asked into L2 ahead, per call
constexpr uint32_t kPrefetchPiece = 16384;

// The four int8-weight words of 16 codes (code i at bits 2i of x), in the
// order even codes 0..6 | 8..14, odd codes 1..7 | 9..15.
__device__ __forceinline__ void decode16_s8(uint32_t x, uint32_t (&w)[4]) {
  const uint32_t ev = x & 0x33333333u, od = (x >> 2) & 0x33333333u;
  w[0] = prmt(kWeightTable, 0u, ev);
  w[1] = prmt(kWeightTable, 0u, ev >> 16);
  w[2] = prmt(kWeightTable, 0u, od);
  w[3] = prmt(kWeightTable, 0u, od >> 16);
}

// Each warp takes R weight rows at a time, so that one read of A's copy from
// shared memory serves R rows.  kVec: packed rows of a multiple of 16 bytes
// at a 16-byte aligned base (16-byte loads); else the chunks are assembled
// from single bytes.
template <int MR, bool kVec>
__global__ void __launch_bounds__(32 * kWarps, 1)
    gemv_kernel(const int8_t* __restrict__ A, const uint8_t* __restrict__ Wp,
                int32_t* __restrict__ C, int M, int N, int K, int64_t KB, int groups) {
  constexpr int R = MR <= 4 ? 4 : 2;
  // A's copy, [MR][4][chunks]: entry (m, q, j) holds the 16 activations of
  // 16-k group 4 j + q in the decode's order, so that consecutive lanes (chunks
  // j) read consecutive 16-byte entries
  extern __shared__ uint4 sa[];
  const int chunks4 = groups / 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // this CTA's rows: an equal contiguous share [nb, ne), taken R at a time by
  // its warps in turn
  const int64_t nb = static_cast<int64_t>(N) * blockIdx.x / gridDim.x;
  const int64_t ne = static_cast<int64_t>(N) * (blockIdx.x + 1) / gridDim.x;
  launch_dependents();
  if (kVec) {
    // the share's packed rows are contiguous: ask them into L2 while the grid
    // before is still running (a hint only; the loads come after the wait)
    int64_t bytes = (ne - nb) * KB;
    const int64_t cap = kPrefetchBytes / gridDim.x / 16 * 16;
    if (bytes > cap) bytes = cap;
    const uint8_t* base = Wp + nb * KB;
    for (int64_t off = static_cast<int64_t>(tid) * kPrefetchPiece; off < bytes;
         off += static_cast<int64_t>(32 * kWarps) * kPrefetchPiece)
      bulk_prefetch_l2(base + off, static_cast<uint32_t>(bytes - off < kPrefetchPiece ? bytes - off
                                                                                      : kPrefetchPiece));
  }
  grid_dependency_wait();  // A and Wp exist, and C is no longer read by the grid before
  // rows of A in 16-byte pieces where they allow (K a multiple of 16, aligned)
  const bool a_vec = (K % 16 == 0) && (reinterpret_cast<uintptr_t>(A) % 16 == 0);
  for (int idx = tid; idx < MR * groups; idx += 32 * kWarps) {
    const int m = idx / groups, g = idx - m * groups;
    uint32_t b[4] = {0u, 0u, 0u, 0u};  // elements 16 g .. 16 g + 15, natural order
    const int64_t k0 = static_cast<int64_t>(g) * 16;
    const int8_t* row = A + static_cast<int64_t>(m) * K;
    if (m < M && a_vec && k0 < K) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + k0));
      b[0] = v.x;
      b[1] = v.y;
      b[2] = v.z;
      b[3] = v.w;
    } else if (m < M) {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (k0 + j < K)
          b[j >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(__ldg(row + k0 + j))) << (8 * (j & 3));
    }
    // even elements 0, 2, 4, 6 | 8, 10, 12, 14, then odd 1, 3, 5, 7 | 9, .., 15
    sa[m * groups + (g & 3) * chunks4 + (g >> 2)] =
        make_uint4(prmt(b[0], b[1], 0x6420u), prmt(b[2], b[3], 0x6420u),
                   prmt(b[0], b[1], 0x7531u), prmt(b[2], b[3], 0x7531u));
  }
  __syncthreads();
  const int64_t chunks = (KB + 15) / 16;
  for (int64_t n0 = nb + static_cast<int64_t>(warp) * R; n0 < ne; n0 += kWarps * R) {
    int32_t acc[R][MR];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MR; ++m) acc[r][m] = 0;
#pragma unroll 2
    for (int64_t j = lane; j < chunks; j += 32) {
      uint32_t c[R][4];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int64_t n = n0 + r < ne ? n0 + r : n0;  // rows past the share repeat row n0, unused
        const uint8_t* wrow = Wp + n * KB;
        if (kVec) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(wrow) + j);
          c[r][0] = v.x;
          c[r][1] = v.y;
          c[r][2] = v.z;
          c[r][3] = v.w;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            c[r][q] = 0u;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int64_t off = 16 * j + 4 * q + t;
              if (off < KB) c[r][q] |= static_cast<uint32_t>(__ldg(wrow + off)) << (8 * t);
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r) decode16_s8(c[r][q], w[r]);
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          const uint4 a = sa[m * groups + q * chunks4 + static_cast<int>(j)];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            acc[r][m] = __dp4a(static_cast<int>(w[r][0]), static_cast<int>(a.x), acc[r][m]);
            acc[r][m] = __dp4a(static_cast<int>(w[r][1]), static_cast<int>(a.y), acc[r][m]);
            acc[r][m] = __dp4a(static_cast<int>(w[r][2]), static_cast<int>(a.z), acc[r][m]);
            acc[r][m] = __dp4a(static_cast<int>(w[r][3]), static_cast<int>(a.w), acc[r][m]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MR; ++m)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], o);
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MR; ++m)
        if (lane == r * MR + m && m < M && n0 + r < ne)
          C[static_cast<int64_t>(m) * N + n0 + r] = acc[r][m];
  }
}

template <int MR>
int set_attrs() {
  return (cudaFuncSetAttribute(gemv_kernel<MR, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kMaxSmem)) == cudaSuccess &&
          cudaFuncSetAttribute(gemv_kernel<MR, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kMaxSmem)) == cudaSuccess)
             ? T3_OK
             : T3_ECUDA;
}

template <int MR>
int launch_mr(const int8_t* A, const uint8_t* Wp, int32_t* C, int M, int N, int K, int64_t KB,
              int groups, int64_t smem, int grid, bool vec, cudaStream_t s) {
  auto fn = vec ? gemv_kernel<MR, true> : gemv_kernel<MR, false>;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(32 * kWarps, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fn, A, Wp, C, M, N, K, KB, groups) != cudaSuccess) return T3_ECUDA;
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace gv

int launch_gemv_fwd(const int8_t* A, const uint8_t* Wp, int32_t* C, int64_t M, int64_t N,
                    int64_t K, int sms, cudaStream_t s) {
  const int64_t KB = (K + 3) / 4;
  // 16-k groups, padded to whole 16-byte chunks of codes (64 k)
  const int64_t groups = (K + 63) / 64 * 4;
  const int mr = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
  const int64_t smem = static_cast<int64_t>(mr) * groups * 16;
  if (M < 1 || M > 8 || smem > gv::kMaxSmem || N > 2147483647LL) return T3_EINVAL;
  const bool vec = (KB % 16 == 0) && (reinterpret_cast<uintptr_t>(Wp) % 16 == 0);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return T3_ECUDA;
  static std::atomic<bool> attr_done[64];
  if (dev < 0 || dev >= 64) return T3_EDEVICE;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (gv::set_attrs<1>() != T3_OK || gv::set_attrs<2>() != T3_OK || gv::set_attrs<4>() != T3_OK ||
        gv::set_attrs<8>() != T3_OK)
      return T3_ECUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  // one CTA per SM, each an equal share of the rows (one CTA per row when
  // there are fewer rows than SMs)
  const int grid = static_cast<int>(N < sms ? N : sms);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const int gr = static_cast<int>(groups);
  switch (mr) {
    case 1: return gv::launch_mr<1>(A, Wp, C, m, n, k, KB, gr, smem, grid, vec, s);
    case 2: return gv::launch_mr<2>(A, Wp, C, m, n, k, KB, gr, smem, grid, vec, s);
    case 4: return gv::launch_mr<4>(A, Wp, C, m, n, k, KB, gr, smem, grid, vec, s);
    default: return gv::launch_mr<8>(A, Wp, C, m, n, k, KB, gr, smem, grid, vec, s);
  }
}

}  // namespace t3
