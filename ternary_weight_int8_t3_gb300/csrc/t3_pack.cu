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
// Each thread then owns 4 columns x 16 k: it reads one 32-bit word per row
// (64 threads read a row's 256 bytes, conflict-free), turns each word into
// the four columns' 2-bit codes with a few bitwise operations (SWAR), which
// also check the four values at once, ORs the codes of 4 rows into one word
// of 4 packed bytes, and transposes the resulting 4 x 4 bytes once.  The packed words are staged in
// shared memory so that each column's 16 packed bytes leave as one 16-byte
// store.
//
// Where w can be a TMA source (rows of a multiple of 16 bytes, 16-byte aligned
// base), one CTA per SM walks tiles of 128 k x 128 n with the loads decoupled
// from the packing: a producer warp streams them by TMA into a ring of nine
// stages (~144 KB per SM in flight), and three groups of eight warps pack the
// tiles in turn, each group on its own three stages, with the same per-thread
// work as above.  A column's 32 packed bytes of a tile fill one sector of its
// Wp row, written by two neighbouring lanes.  Tiles past K or N arrive
// zero-filled (code 0, as the pad positions want).
#include <atomic>
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

// The 2-bit codes of four int8 weights (one per byte), each in the low bits
// of its byte: +1 -> 1, -1 -> 2, 0 -> 0.  Per byte, lo = bit 0 and sg = the
// sign bit; the valid bytes are exactly the ones rebuilt by lo | (sg ? 0xFF :
// 0) -- 0x00, 0x01 and 0xFF (sg * 0xFF stays inside its byte) -- and their
// codes are lo + sg.  A word with another byte takes the byte-by-byte path
// (rare): invalid bytes get code 0 and set `bad`.
__device__ __forceinline__ uint32_t codes4(uint32_t x, bool& bad) {
  const uint32_t lo = x & 0x01010101u, sg = (x >> 7) & 0x01010101u;
  if ((lo | (sg * 0xFFu)) == x) return lo + sg;
  bad = true;
  uint32_t r = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int v = static_cast<int8_t>(x >> (8 * j));
    r |= (v == 1 ? 1u : (v == -1 ? 2u : 0u)) << (8 * j);
  }
  return r;
}

// The packing of one [TK][TN] tile by one thread: columns 4 cg .. 4 cg + 3,
// k rows 16 kq .. 16 kq + 15.  A row's word holds the four columns' weights
// at one k; the code words of four consecutive rows, shifted by 0, 2, 4 and
// 6 bits, OR into one word whose byte i is column i's packed byte for those
// four k (codes fill 2 bits, so nothing crosses into the next byte).  A 4 x 4
// byte transpose of the four such words gives out[i], column i's 4 packed
// bytes (16 k).
template <int kRow>
__device__ __forceinline__ void pack_tile(const int8_t (*tile)[kRow], int cg, int kq,
                                          uint32_t (&out)[4], bool& bad) {
  uint32_t q[4];
  // per byte lo = bit 0 and sg = the sign bit of every word; the code words
  // of four rows (lo + sg in bits 2 rr of each byte) add up as lo0 + sg0 +
  // 4 (lo1 + sg1) + 16 (..) + 64 (..), the fields never overlapping, so the
  // merge is multiply-adds; one validity word collects every byte that lo |
  // (sg * 0xFF) does not rebuild, and only a tile part with such a byte
  // takes the byte-by-byte path (invalid values as code 0)
  uint32_t x[16], any_bad = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = *reinterpret_cast<const uint32_t*>(&tile[16 * kq + i][4 * cg]);
#pragma unroll
  for (int sb = 0; sb < 4; ++sb) {
    uint32_t word = 0u;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const uint32_t xv = x[4 * sb + rr];
      const uint32_t lo = xv & 0x01010101u, sg = (xv >> 7) & 0x01010101u;
      any_bad |= (lo | (sg * 0xFFu)) ^ xv;
      word += (lo + sg) * (1u << (2 * rr));
    }
    q[sb] = word;
  }
  if (any_bad != 0u) {
#pragma unroll
    for (int sb = 0; sb < 4; ++sb) {
      uint32_t word = 0u;
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) word |= codes4(x[4 * sb + rr], bad) << (2 * rr);
      q[sb] = word;
    }
  }
  const uint32_t a = byte_perm(q[0], q[1], 0x5140u), b = byte_perm(q[2], q[3], 0x5140u);
  const uint32_t c = byte_perm(q[0], q[1], 0x7362u), d = byte_perm(q[2], q[3], 0x7362u);
  out[0] = byte_perm(a, b, 0x5410u);
  out[1] = byte_perm(a, b, 0x7632u);
  out[2] = byte_perm(c, d, 0x5410u);
  out[3] = byte_perm(c, d, 0x7632u);
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
    uint32_t out[4];  // per column: 4 packed bytes = 16 k
    pack_tile<TN>(tile, cg, kq, out, bad);
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

constexpr int kGroups = 3;                          // consumer groups, tiles in turn
// Tile i goes to stage i % kStages and to group i % kGroups; with kStages a
// multiple of kGroups every stage belongs to one group, which consumes its
// stages in order.  A group can then never wait on a stage whose previous
// tile (another group's) has not landed yet, where the parity wait would
// match the completion two phases back and pass early.
constexpr int kStages = 3 * kGroups;
constexpr int kTmaThreads = kGroups * kThreads + 32;  // + the producer warp
// the TMA path's tiles: 128 k x 128 n (16 KB), so that a column's packed
// bytes of a tile (32) fill a sector of its Wp row, written by two lanes
constexpr int TK2 = 128, TN2 = 128;
constexpr int kTileBytes = TK2 * TN2;
constexpr int kTmaSmem = kStages * kTileBytes + 128;
constexpr int kRowWords = TK2 / 16;                 // packed words per column per tile
static_assert(kStages % kGroups == 0, "each stage belongs to one consumer group");
static_assert((TN2 / 4) * (TK2 / 16) == kThreads, "a thread packs 4 columns x 16 k");

// Tiles of 128 k x 128 n, numbered n-block fastest; each column of a tile
// makes 32 packed bytes of its Wp row.
__global__ void __launch_bounds__(kTmaThreads, 1)
    pack_tma_kernel(const __grid_constant__ CUtensorMap map_w, uint8_t* __restrict__ wp,
                    int64_t N, int64_t KB, int64_t tiles_n, int64_t tiles, int vec_out,
                    int* err) {
  extern __shared__ uint8_t smem_raw[];
  int8_t (*ring)[TK2][TN2] = reinterpret_cast<int8_t (*)[TK2][TN2]>(
      smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u));
  // a group's packed rows (two buffers), padded by one word
  __shared__ uint32_t packed[kGroups][2][TN2][kRowWords + 1];
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kThreads / 32);  // the warps of the group that packed the stage
    }
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  const int64_t my_tiles = blockIdx.x < tiles ? (tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  constexpr int code = (9 << 8) | 1;
  if (warp == kGroups * (kThreads / 32)) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&map_w);
      int64_t j = 0;
      for (; j < my_tiles; ++j) {
        const int s = static_cast<int>(j % kStages);
        if (!mbar_wait(&empty[s], static_cast<uint32_t>((j / kStages) & 1) ^ 1u, &abort_flag, err,
                       code))
          break;
        const int64_t tix = blockIdx.x + j * gridDim.x;
        const int64_t tk = tix / tiles_n;
        mbar_arrive_expect_tx(&full[s], kTileBytes);
        tma_load_2d(ring[s], &map_w, &full[s], static_cast<int32_t>((tix - tk * tiles_n) * TN2),
                    static_cast<int32_t>(tk * TK2));
      }
      // no copy is left in flight when the CTA ends, whatever the consumers
      // did (a wait of its own, bounded, that an abort does not cut short)
      int keep_waiting = 0;
      for (int64_t q = j - kStages < 0 ? 0 : j - kStages; q < j; ++q)
        mbar_wait(&full[q % kStages], static_cast<uint32_t>((q / kStages) & 1), &keep_waiting, err,
                  code);
    }
    return;
  }
  // ------------------------------------------------------------- consumers
  const int grp = warp / (kThreads / 32);
  const int t = threadIdx.x - grp * kThreads;
  const int cg = t % (TN2 / 4), kq = t / (TN2 / 4);
  bool bad = false;
  for (int64_t i = grp; i < my_tiles; i += kGroups) {
    uint32_t out[4] = {0u, 0u, 0u, 0u};
    const int s = static_cast<int>(i % kStages);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>((i / kStages) & 1),
                                                     &abort_flag, err, code + 1));
    if (ok) {
      pack_tile<TN2>(ring[s], cg, kq, out, bad);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    const int64_t tix = blockIdx.x + i * gridDim.x;
    const int64_t tk = tix / tiles_n;
    const int64_t n0 = (tix - tk * tiles_n) * TN2;
    // two staging buffers per group, so that one barrier per tile separates
    // this tile's stores from its reads, and the reads of the tile before
    // (the other buffer) from the stores of the tile after; the barrier also
    // takes the group's decision to stop (a wait that gave up), so that all
    // its warps leave together and none is left at a later barrier
    uint32_t (*pk)[kRowWords + 1] = packed[grp][(i / kGroups) & 1];
#pragma unroll
    for (int c = 0; c < 4; ++c) pk[4 * cg + c][kq] = out[c];
    if (!named_bar_and(1 + grp, kThreads, ok)) break;
    // lanes 2 c and 2 c + 1: the two 16-byte halves of column c's 32 bytes
    const int64_t n = n0 + (t >> 1);
    const int hh = t & 1;
    const int64_t off = tk * (TK2 / 4) + 16 * hh;
    if (t < 2 * TN2 && n < N) {
      uint8_t* dst = wp + n * KB + off;
      const uint32_t* row = pk[t >> 1] + 4 * hh;
      if (vec_out && off + 16 <= KB) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(row[0], row[1], row[2], row[3]);
      } else {
        for (int b = 0; b < 16 && off + b < KB; ++b) dst[b] = static_cast<uint8_t>(row[b >> 2] >> (8 * (b & 3)));
      }
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(err, 0, kErrInvalid);
}

}  // namespace pack

int launch_pack_device(const int8_t* w, uint8_t* wp, int64_t K, int64_t N, int sms, int* err,
                       cudaStream_t s) {
  const int64_t KB = (K + 3) / 4;
  const int64_t tiles_n = (N + pack::TN - 1) / pack::TN, tiles_k = (K + pack::TK - 1) / pack::TK;
  const int64_t tiles = tiles_n * tiles_k;
  const int vec_in = (N % 16 == 0) && (reinterpret_cast<uintptr_t>(w) % 16 == 0);
  const int vec_out = (KB % 16 == 0) && (reinterpret_cast<uintptr_t>(wp) % 16 == 0);
  CUtensorMap map;
  if (vec_in && make_u8_map_tiled(&map, w, K, N, N, pack::TK2, pack::TN2, false)) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return T3_ECUDA;
    static std::atomic<bool> attr_done[64];
    if (dev < 0 || dev >= 64) return T3_EDEVICE;
    if (!attr_done[dev].load(std::memory_order_acquire)) {
      if (cudaFuncSetAttribute(pack::pack_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               pack::kTmaSmem) != cudaSuccess)
        return T3_ECUDA;
      attr_done[dev].store(true, std::memory_order_release);
    }
    const int64_t tiles_n2 = (N + pack::TN2 - 1) / pack::TN2, tiles_k2 = (K + pack::TK2 - 1) / pack::TK2;
    const int64_t tiles2 = tiles_n2 * tiles_k2;
    const int64_t grid = tiles2 < sms ? tiles2 : sms;
    pack::pack_tma_kernel<<<static_cast<unsigned>(grid > 0 ? grid : 1), pack::kTmaThreads,
                            pack::kTmaSmem, s>>>(map, wp, N, KB, tiles_n2, tiles2, vec_out, err);
    return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
  }
  // enough CTAs to keep every SM's loads in flight, each walking several tiles
  const int64_t cap = 16 * static_cast<int64_t>(sms > 0 ? sms : 1);
  const int64_t grid = tiles < cap ? tiles : cap;
  pack::pack_kernel<<<static_cast<unsigned>(grid), pack::kThreads, 0, s>>>(
      w, wp, K, N, KB, tiles_n, tiles, vec_in, vec_out, err);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
