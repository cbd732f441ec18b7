// t3_pack.cu -- the 2-bit weight packer on the device.
//
// What it computes: the weight codes of "t27c PTX backend: ternary x int8 GEMM
// kernel emitted by a .t27 spec (int8 mma.sync), ptx-run glue", section "What
// this adds": w in {-1, 0, +1} becomes code 1 for +1, 2 for -1 and 0 for 0;
// the code of element k sits at bits 2 (k % 4) of byte k / 4 of its row, and
// the packed matrix Wp [N][ceil(K/4)] holds one row per output column n of
// W [K][N] (so the packer transposes).  Codes past K in a row's last byte are 0.
//
// Why this shape.  The packer moves K*N bytes in and K*N/4 out and does no
// arithmetic to speak of: it should be bound by HBM, so it is written to keep
// the instruction count per weight low.  A CTA takes a tile of 64 k x 256 n: it
// reads the tile's 64 rows with coalesced loads (16 bytes per thread where
// every row is 16-byte aligned, single bytes otherwise) into shared memory.
// Each thread then owns 4 columns x 16 k: per 4 rows it reads four 32-bit
// words (64 threads read a row's 256 bytes, conflict-free), transposes the
// 4 x 4 bytes with byte permutes so that each word holds 4 k of one column,
// and turns that word into one packed byte with a few bitwise operations
// (SWAR), checking the four values at once.  The packed words are staged in
// shared memory so that each column's 16 packed bytes leave as one 16-byte
// store.
#include <cstdint>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {
namespace pack {

constexpr int TK = 64;    // k per tile (16 packed bytes per row of Wp)
constexpr int TN = 256;   // n per tile
constexpr int kThreads = 256;
constexpr int kErrInvalid = (9 << 8) | 6;  // kernel 9 (device packer), role 6 (invalid value)

__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Four int8 weights (one per byte) -> their four 2-bit codes in one byte
// (byte j's code at bits 2j); a byte other than 0x00, 0x01, 0xFF packs as
// code 0 and sets `bad`.
__device__ __forceinline__ uint32_t pack4(uint32_t x, bool& bad) {
  // bytewise x + 1 (no carries between bytes): valid bytes become 0, 1 or 2,
  // i.e. bits 2-7 clear and not both bits 0 and 1 set
  const uint32_t inc = ((x & 0x7F7F7F7Fu) + 0x01010101u) ^ (x & 0x80808080u);
  if (((inc & 0xFCFCFCFCu) | (inc & (inc >> 1) & 0x01010101u)) != 0u) {
    bad = true;  // rare: byte by byte, invalid bytes as code 0
    uint32_t r = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = static_cast<int8_t>(x >> (8 * j));
      r |= (v == 1 ? 1u : (v == -1 ? 2u : 0u)) << (2 * j);
    }
    return r;
  }
  const uint32_t b0 = x & 0x01010101u, b1 = (x >> 1) & 0x01010101u;
  const uint32_t c = (b0 & ~b1) | (b1 << 1);  // +1 -> 1, -1 -> 2, 0 -> 0, per byte
  return (c | (c >> 6) | (c >> 12) | (c >> 18)) & 0xFFu;
}

// Tiles are numbered n-block fastest and walked grid-stride.
__global__ void __launch_bounds__(kThreads) pack_kernel(const int8_t* __restrict__ w,
                                                        uint8_t* __restrict__ wp, int64_t K,
                                                        int64_t N, int64_t KB, int64_t tiles_n,
                                                        int64_t tiles, int vec_in, int vec_out,
                                                        int* err) {
  __shared__ __align__(16) int8_t tile[TK][TN];
  // packed rows of the tile: 16 bytes per column n, padded to 5 words so that
  // the 4-byte stores of consecutive column groups spread over the banks
  __shared__ uint32_t packed[TN][5];
  const int t = threadIdx.x;
  // thread -> columns 4 cg .. 4 cg + 3 of the tile, k rows 16 kq .. 16 kq + 15
  const int cg = t % (TN / 4), kq = t / (TN / 4);
  bool bad = false;
  for (int64_t tix = blockIdx.x; tix < tiles; tix += gridDim.x) {
    const int64_t tk = tix / tiles_n;
    const int64_t k0 = tk * TK;
    const int64_t n0 = (tix - tk * tiles_n) * TN;
    __syncthreads();  // the previous tile's reads are done
    if (vec_in) {
      // 64 rows x 16 chunks of 16 bytes; N % 16 == 0 so a chunk is in or out whole
      for (int i = t; i < TK * (TN / 16); i += kThreads) {
        const int r = i / (TN / 16), c = i % (TN / 16);
        const int64_t k = k0 + r, n = n0 + 16 * c;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (k < K && n < N) v = __ldg(reinterpret_cast<const uint4*>(w + k * N + n));
        *reinterpret_cast<uint4*>(&tile[r][16 * c]) = v;
      }
    } else {
      for (int i = t; i < TK * TN; i += kThreads) {
        const int r = i / TN, c = i % TN;
        const int64_t k = k0 + r, n = n0 + c;
        tile[r][c] = (k < K && n < N) ? w[k * N + n] : static_cast<int8_t>(0);
      }
    }
    __syncthreads();
    // rows past K hold 0 and pack as code 0
    uint32_t out[4] = {0u, 0u, 0u, 0u};  // per column: 4 packed bytes = 16 k
#pragma unroll
    for (int sb = 0; sb < 4; ++sb) {
      const int r = 16 * kq + 4 * sb;
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(&tile[r][4 * cg]);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(&tile[r + 1][4 * cg]);
      const uint32_t w2 = *reinterpret_cast<const uint32_t*>(&tile[r + 2][4 * cg]);
      const uint32_t w3 = *reinterpret_cast<const uint32_t*>(&tile[r + 3][4 * cg]);
      // 4 x 4 byte transpose: col[i] = byte i of w0, w1, w2, w3 (4 k of column i)
      const uint32_t a = byte_perm(w0, w1, 0x5140u), b = byte_perm(w2, w3, 0x5140u);
      const uint32_t c = byte_perm(w0, w1, 0x7362u), d = byte_perm(w2, w3, 0x7362u);
      const uint32_t col[4] = {byte_perm(a, b, 0x5410u), byte_perm(a, b, 0x7632u),
                               byte_perm(c, d, 0x5410u), byte_perm(c, d, 0x7632u)};
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i] |= pack4(col[i], bad) << (8 * sb);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) packed[4 * cg + i][kq] = out[i];
    __syncthreads();
    // one thread per column: its 16 packed bytes in one store where aligned
    {
      const int64_t n = n0 + t;
      const int64_t b0 = tk * (TK / 4);
      if (n < N) {
        uint8_t* dst = wp + n * KB + b0;
        const uint32_t* row = packed[t];
        if (vec_out && b0 + 16 <= KB) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(row[0], row[1], row[2], row[3]);
        } else {
          for (int b = 0; b < 16 && b0 + b < KB; ++b)
            dst[b] = static_cast<uint8_t>(row[b >> 2] >> (8 * (b & 3)));
        }
      }
    }
  }
  if (__any_sync(0xffffffffu, bad) && (t & 31) == 0) atomicCAS(err, 0, kErrInvalid);
}

}  // namespace pack

int launch_pack_device(const int8_t* w, uint8_t* wp, int64_t K, int64_t N, int sms, int* err,
                       cudaStream_t s) {
  const int64_t KB = (K + 3) / 4;
  const int64_t tiles_n = (N + pack::TN - 1) / pack::TN, tiles_k = (K + pack::TK - 1) / pack::TK;
  const int64_t tiles = tiles_n * tiles_k;
  const int vec_in = (N % 16 == 0) && (reinterpret_cast<uintptr_t>(w) % 16 == 0);
  const int vec_out = (KB % 16 == 0) && (reinterpret_cast<uintptr_t>(wp) % 16 == 0);
  // enough CTAs to keep every SM's loads in flight, each walking several tiles
  const int64_t cap = 16 * static_cast<int64_t>(sms > 0 ? sms : 1);
  const int64_t grid = tiles < cap ? tiles : cap;
  pack::pack_kernel<<<static_cast<unsigned>(grid), pack::kThreads, 0, s>>>(
      w, wp, K, N, KB, tiles_n, tiles, vec_in, vec_out, err);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
