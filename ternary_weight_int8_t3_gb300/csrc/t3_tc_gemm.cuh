// t3_tc_gemm.cuh -- the tensor-core pipeline shared by the forward, dX and dW
// products of a ternary-weight layer (sm_103a, tcgen05 + TMA + mbarrier).
//
// What it computes (web pages, by title and section):
//   forward  "t27c PTX backend: ternary x int8 GEMM kernel emitted by a .t27
//            spec (int8 mma.sync), ptx-run glue", "What this adds":
//            C[m][n] = sum_k A[m][k] W[k][n], W from 2-bit codes decoded as
//            (c & 1) - ((c >> 1) & 1).
//   dX, dW   "spec(igla): hslm_bwd_ptx -- HSLM backward dX and dW as int8
//            tensor-core PTX written by t27", kernels 1 and 2:
//            dX[m][k] = sum_n dY[m][n] W[k][n],  dW[k][n] = sum_m A[m][k] dY[m][n].
//
// How (GB300 design, not the pages' sm_89 one):
//   sm_103a has no int8 tcgen05 kind, so operands are carried as f16, which
//   holds every int8 and every ternary value exactly, and the tensor core
//   accumulates in f32 in TMEM.  A sum of integers stays exact in f32 while
//   its magnitude stays <= 2^23 (below 2^24 with a bit of margin for the
//   hardware's alignment), so the reduction is cut into chunks of
//   2^23 / max|product| elements: 65536 for the ternary products (|a w| <=
//   128) and 512 for dW (|a dy| <= 16384).  Each chunk's f32 sum is converted
//   to int32 exactly in the epilogue and added in integer arithmetic.
//
//   One CTA per SM, persistent over output tiles of 128 x 256, 10 warps:
//     warps 0-3  converters: raw int8 / packed 2-bit tiles -> f16 tiles in the
//                128-byte-swizzled K-major layout the tensor core reads; the
//                packed weights are decoded once per tile load with byte
//                permutes on the table {0, +1.0, -1.0, 0}.
//     warp 4     producer: TMA (cp.async.bulk.tensor) of the raw tiles into a
//                4-stage ring; a plain-load fallback when a row stride or base
//                is not 16-byte aligned.
//     warp 5     tensor-core issuer: tcgen05.mma kind::f16, M=128 N=256 K=16,
//                into one of two TMEM accumulators (2 x 256 columns).
//     warps 6-9  epilogue: tcgen05.ld -> int32 -> predicated global stores,
//                overlapping the next tile's main loop.
#pragma once
#include <cstdint>
#include "t3_ptx.cuh"

namespace t3 {

enum OpKind : int { kOpFwd = 1, kOpDx = 2, kOpDw = 3 };

namespace tc {

constexpr int BM = 128;  // output rows per tile (TMEM lanes)
constexpr int BN = 256;  // output columns per tile (MMA N)
constexpr int BK = 64;   // reduction elements per pipeline stage (128 B of f16)
constexpr int UK = 16;   // reduction elements per tcgen05.mma (kind::f16)
// Raw stages in flight: enough bytes to cover L2/HBM latency at the MMA rate.
template <int OP> struct RawStages { static constexpr int value = 6; };
constexpr int OP_STAGES = 2;
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = ACC_BUFS * BN;  // 512
constexpr int kConvWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kProducerWarp = kConvWarps;
constexpr int kMmaWarp = kConvWarps + 1;
constexpr int kEpiWarp0 = kConvWarps + 2;
constexpr int kThreads = 32 * (kConvWarps + 2 + 4);
constexpr int OPA_BYTES = BM * BK * 2;
constexpr int OPB_BYTES = BN * BK * 2;

// Exact-f32 chunk lengths, in pipeline stages.
constexpr int64_t kChunkKbTernary = 65536 / BK;  // |product| <= 128
constexpr int64_t kChunkKbInt8 = 512 / BK;       // |product| <= 16384

// Raw (pre-conversion) box shapes in bytes: rows x columns.
template <int OP> struct Raw;
template <> struct Raw<kOpFwd> {  // A [BM m][BK k];  Wp [BN n][BK/4 bytes]
  static constexpr int a_rows = BM, a_cols = BK, b_rows = BN, b_cols = BK / 4;
};
template <> struct Raw<kOpDx> {   // dY [BM m][BK n]; Wp [BK n][BN/4 bytes]
  static constexpr int a_rows = BM, a_cols = BK, b_rows = BK, b_cols = BN / 4;
};
template <> struct Raw<kOpDw> {   // A [BK m][BM k];  dY [BK m][BN n]
  static constexpr int a_rows = BK, a_cols = BM, b_rows = BK, b_cols = BN;
};

template <> struct RawStages<kOpDw> { static constexpr int value = 3; };

// Output staging for the bulk-store epilogue: two [128 rows][32 int32]
// buffers in the 128-byte swizzle layout.
constexpr int STAGE_OUT_BYTES = BM * 32 * 4;
constexpr int kEpiBarrier = 1;  // named barrier of the 4 epilogue warps

template <int OP> struct Layout {
  static constexpr int RAW_STAGES = RawStages<OP>::value;
  static constexpr int raw_a = Raw<OP>::a_rows * Raw<OP>::a_cols;
  static constexpr int raw_b = Raw<OP>::b_rows * Raw<OP>::b_cols;
  static constexpr int raw_stage = raw_a + raw_b;
  static constexpr int off_opa = 0;
  static constexpr int off_opb = off_opa + OP_STAGES * OPA_BYTES;
  static constexpr int off_raw = off_opb + OP_STAGES * OPB_BYTES;
  static constexpr int off_out = off_raw + RAW_STAGES * raw_stage;
  static constexpr int off_bar = off_out + 2 * STAGE_OUT_BYTES;
  static constexpr int n_bars = 2 * RAW_STAGES + 2 * OP_STAGES + 2 * ACC_BUFS + 1;
  static constexpr int off_misc = off_bar + 8 * n_bars;
  static constexpr int bytes = off_misc + 16;
  static constexpr int smem_alloc = bytes + 1024;  // slack to align the base to 1024
};

struct Params {
  const uint8_t* a_src;  // fwd: A, dX: dY, dW: A
  int64_t a_ld, a_rows, a_cols;
  const uint8_t* b_src;  // fwd: Wp, dX: Wp, dW: dY
  int64_t b_ld, b_rows, b_cols;
  int32_t* out;
  int64_t out_rows, out_cols;
  int64_t num_kb;    // pipeline stages along the reduction
  int64_t chunk_kb;  // stages per exact f32 chunk
  int tiles_r, tiles_c;
  int use_tma_a, use_tma_b;
  int use_tma_out;  // output written with bulk tensor stores (needs out_cols % 4 == 0)
  int* err;  // device error word
  int op_code;
};

// ---------------------------------------------------------------- helpers

template <int OP>
__device__ __forceinline__ void box_coords(int tr, int tcol, int64_t kb, int& ax, int& ay,
                                           int& bx, int& by) {
  if (OP == kOpFwd) {
    ax = static_cast<int>(kb * BK); ay = tr * BM;
    bx = static_cast<int>(kb * (BK / 4)); by = tcol * BN;
  } else if (OP == kOpDx) {
    ax = static_cast<int>(kb * BK); ay = tr * BM;
    bx = tcol * (BN / 4); by = static_cast<int>(kb * BK);
  } else {
    ax = tr * BM; ay = static_cast<int>(kb * BK);
    bx = tcol * BN; by = static_cast<int>(kb * BK);
  }
}

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

// 8 codes in bits 0..15 -> each code in its own nibble.
__device__ __forceinline__ uint32_t spread_codes_to_nibbles(uint32_t v) {
  v = (v | (v << 8)) & 0x00FF00FFu;
  v = (v | (v << 4)) & 0x0F0F0F0Fu;
  v = (v | (v << 2)) & 0x33333333u;
  return v;
}

// 8 codes (one per nibble) -> 8 f16 weights in reduction order.
__device__ __forceinline__ uint4 decode8_nibbles(uint32_t nib) {
  const uint32_t h0 = prmt(kF16HiTable, 0u, nib);
  const uint32_t h1 = prmt(kF16HiTable, 0u, nib >> 16);
  uint4 o;
  o.x = prmt(h0, 0u, 0x1404u);
  o.y = prmt(h0, 0u, 0x3424u);
  o.z = prmt(h1, 0u, 0x1404u);
  o.w = prmt(h1, 0u, 0x3424u);
  return o;
}

// Y[b] = byte b of a0..a3, in that order.
__device__ __forceinline__ void transpose4x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t (&Y)[4]) {
  const uint32_t t0 = prmt(a0, a1, 0x5140u), t1 = prmt(a2, a3, 0x5140u);
  const uint32_t t2 = prmt(a0, a1, 0x7362u), t3 = prmt(a2, a3, 0x7362u);
  Y[0] = prmt(t0, t1, 0x5410u);
  Y[1] = prmt(t0, t1, 0x7632u);
  Y[2] = prmt(t2, t3, 0x5410u);
  Y[3] = prmt(t2, t3, 0x7632u);
}

// Byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled tile.
__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// ------------------------------------------------------------- converters

// int8 rows [128][64] (reduction contiguous) -> f16 rows [128][64].
__device__ __forceinline__ void convert_rows_s8(const uint8_t* raw, uint8_t* op, int tid) {
#pragma unroll
  for (int i = 0; i < 512 / kConvThreads; ++i) {
    const int u = tid + kConvThreads * i, r = u >> 2, c = u & 3;
    const uint4 x = *reinterpret_cast<const uint4*>(raw + r * 64 + c * 16);
    uint4 o0, o1;
    s8x4_to_f16(x.x, o0.x, o0.y);
    s8x4_to_f16(x.y, o0.z, o0.w);
    s8x4_to_f16(x.z, o1.x, o1.y);
    s8x4_to_f16(x.w, o1.z, o1.w);
    *reinterpret_cast<uint4*>(op + sw128(r, 2 * c)) = o0;
    *reinterpret_cast<uint4*>(op + sw128(r, 2 * c + 1)) = o1;
  }
}

// Forward weights: packed rows [256 n][16 bytes = 64 codes along k] -> f16
// rows [256 n][64 k].
__device__ __forceinline__ void decode_rows_w(const uint8_t* raw, uint8_t* op, int tid) {
#pragma unroll
  for (int i = 0; i < 1024 / kConvThreads; ++i) {
    const int u = tid + kConvThreads * i, r = u >> 2, w = u & 3;
    const uint32_t x = *reinterpret_cast<const uint32_t*>(raw + r * 16 + w * 4);
    *reinterpret_cast<uint4*>(op + sw128(r, 2 * w)) =
        decode8_nibbles(spread_codes_to_nibbles(x & 0xFFFFu));
    *reinterpret_cast<uint4*>(op + sw128(r, 2 * w + 1)) =
        decode8_nibbles(spread_codes_to_nibbles(x >> 16));
  }
}

// dX weights: packed [64 n][64 bytes = 256 codes along k] -> f16 rows
// [256 k][64 n]: a transposing decode.  Unit = (word column w, group of 8
// n-rows g), split across kConvThreads/128 threads by byte b; g is rotated by
// w so that each 8-thread store phase hits 8 distinct bank groups.
__device__ __forceinline__ void decode_cols_w(const uint8_t* raw, uint8_t* op, int tid) {
  constexpr int kParts = kConvThreads / 128, kBytes = 4 / kParts;
  const int t = tid & 127, part = tid >> 7;
  const int w = t & 15, g = ((t >> 4) + w) & 7;
  const uint32_t* rw = reinterpret_cast<const uint32_t*>(raw);
  uint32_t x[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = rw[(8 * g + i) * 16 + w];
  uint32_t Y[4], Z[4];
  transpose4x4(x[0], x[1], x[2], x[3], Y);
  transpose4x4(x[4], x[5], x[6], x[7], Z);
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    if (b / kBytes != part) continue;  // warp-uniform; keeps Y[b] statically indexed
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int krow = 16 * w + 4 * b + j;
      const uint32_t sy = Y[b] >> (2 * j), sz = Z[b] >> (2 * j);
      uint4 o;
      o.x = prmt(kF16HiTable, 0u, ((sy << 4) & 0x3030u) | 0x0404u);
      o.y = prmt(kF16HiTable, 0u, ((sy >> 12) & 0x3030u) | 0x0404u);
      o.z = prmt(kF16HiTable, 0u, ((sz << 4) & 0x3030u) | 0x0404u);
      o.w = prmt(kF16HiTable, 0u, ((sz >> 12) & 0x3030u) | 0x0404u);
      *reinterpret_cast<uint4*>(op + sw128(krow, g)) = o;
    }
  }
}

// dW operands: int8 [64 m][ROW_WORDS*4 columns] (reduction m is the row) ->
// f16 rows [ROW_WORDS*4][64 m]: a transposing conversion.
template <int ROW_WORDS>
__device__ __forceinline__ void convert_cols_s8(const uint8_t* raw, uint8_t* op, int tid) {
  constexpr int kUnits = ROW_WORDS * 8 / kConvThreads;
  static_assert(kUnits >= 1, "one unit per thread at least");
  const uint32_t* rw = reinterpret_cast<const uint32_t*>(raw);
#pragma unroll
  for (int i = 0; i < kUnits; ++i) {
    const int u = tid + kConvThreads * i, w = u % ROW_WORDS, g = ((u / ROW_WORDS) + w) & 7;
    uint32_t x[8];
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) x[ii] = rw[(8 * g + ii) * ROW_WORDS + w];
    uint32_t Y[4], Z[4];
    transpose4x4(x[0], x[1], x[2], x[3], Y);
    transpose4x4(x[4], x[5], x[6], x[7], Z);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int row = 4 * w + b;
      uint4 o;
      s8x4_to_f16(Y[b], o.x, o.y);
      s8x4_to_f16(Z[b], o.z, o.w);
      *reinterpret_cast<uint4*>(op + sw128(row, g)) = o;
    }
  }
}

template <int OP>
__device__ __forceinline__ void convert_stage(const uint8_t* raw, uint8_t* opa, uint8_t* opb,
                                              int tid) {
  const uint8_t* ra = raw;
  const uint8_t* rb = raw + Layout<OP>::raw_a;
  if (OP == kOpFwd) {
    convert_rows_s8(ra, opa, tid);
    decode_rows_w(rb, opb, tid);
  } else if (OP == kOpDx) {
    convert_rows_s8(ra, opa, tid);
    decode_cols_w(rb, opb, tid);
  } else {
    convert_cols_s8<BM / 4>(ra, opa, tid);
    convert_cols_s8<BN / 4>(rb, opb, tid);
  }
}

// ------------------------------------------------------------- epilogue

__device__ __forceinline__ int32_t f32_bits_to_i32(uint32_t bits) {
  return __float2int_rn(__uint_as_float(bits));  // the value is an exact integer
}

// Writes (first chunk) or adds (later chunks) 32 values of one output row.
__device__ __forceinline__ void store_row32(int32_t* dst, const uint32_t (&v)[32], int valid,
                                            bool first, bool vec_ok) {
  if (vec_ok && valid == 32) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      int4 val = make_int4(f32_bits_to_i32(v[i]), f32_bits_to_i32(v[i + 1]),
                           f32_bits_to_i32(v[i + 2]), f32_bits_to_i32(v[i + 3]));
      int4* p = reinterpret_cast<int4*>(dst + i);
      if (!first) {
        const int4 old = *p;
        val.x += old.x; val.y += old.y; val.z += old.z; val.w += old.w;
      }
      *p = val;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < valid) {
        const int32_t val = f32_bits_to_i32(v[i]);
        dst[i] = first ? val : dst[i] + val;
      }
    }
  }
}

// ------------------------------------------------------------------ kernel

template <int OP>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const Params p, const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_out) {
  using L = Layout<OP>;
  using R = Raw<OP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((base_addr + 1023u) & ~1023u) - base_addr);

  uint8_t* opa = smem + L::off_opa;
  uint8_t* opb = smem + L::off_opb;
  uint8_t* raw = smem + L::off_raw;
  uint8_t* stage_out = smem + L::off_out;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::off_bar);
  uint64_t* raw_full = bars;
  constexpr int RAW_STAGES = L::RAW_STAGES;
  uint64_t* raw_empty = raw_full + RAW_STAGES;
  uint64_t* op_full = raw_empty + RAW_STAGES;
  uint64_t* op_empty = op_full + OP_STAGES;
  uint64_t* acc_full = op_empty + OP_STAGES;
  uint64_t* acc_empty = acc_full + ACC_BUFS;
  uint64_t* drain_bar = acc_empty + ACC_BUFS;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::off_misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = p.tiles_r * p.tiles_c;
  const int code_base = p.op_code << 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW_STAGES; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kConvWarps);
    }
    for (int s = 0; s < OP_STAGES; ++s) {
      mbar_init(&op_full[s], kConvWarps);
      mbar_init(&op_empty[s], 1);
    }
    for (int s = 0; s < ACC_BUFS; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp < kConvWarps) {
    // ---------------------------------------------------------- converters
    const int tid = threadIdx.x;
    uint32_t rs = 0, rph = 0, os = 0, oph = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      bool ok = true;
      for (int64_t kb = 0; kb < p.num_kb; ++kb) {
        ok = mbar_wait(&raw_full[rs], rph, abort_flag, p.err, code_base | 2) &&
             mbar_wait(&op_empty[os], oph ^ 1u, abort_flag, p.err, code_base | 2);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        convert_stage<OP>(raw + rs * L::raw_stage, opa + os * OPA_BYTES, opb + os * OPB_BYTES,
                          tid);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&raw_empty[rs]);
          mbar_arrive(&op_full[os]);
        }
        if (++rs == RAW_STAGES) { rs = 0; rph ^= 1u; }
        if (++os == OP_STAGES) { os = 0; oph ^= 1u; }
      }
      if (!ok) break;
    }
  } else if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if (p.use_tma_a) prefetch_tensormap(&map_a);
      if (p.use_tma_b) prefetch_tensormap(&map_b);
    }
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, issued_phase = 0;  // stages with a copy possibly in flight
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const int tr = tile / p.tiles_c, tcol = tile % p.tiles_c;
      for (int64_t kb = 0; kb < p.num_kb; ++kb) {
        ok = mbar_wait(&raw_empty[stage], phase ^ 1u, abort_flag, p.err, code_base | 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        int ax, ay, bx, by;
        box_coords<OP>(tr, tcol, kb, ax, ay, bx, by);
        uint8_t* ra = raw + stage * L::raw_stage;
        uint8_t* rb = ra + L::raw_a;
        if (!p.use_tma_a)
          manual_box(ra, p.a_src, p.a_ld, p.a_rows, p.a_cols, ay, ax, R::a_rows, R::a_cols, lane);
        if (!p.use_tma_b)
          manual_box(rb, p.b_src, p.b_ld, p.b_rows, p.b_cols, by, bx, R::b_rows, R::b_cols, lane);
        __threadfence_block();
        __syncwarp();
        if (lane == 0) {
          const uint32_t tx = (p.use_tma_a ? L::raw_a : 0) + (p.use_tma_b ? L::raw_b : 0);
          if (tx) {
            mbar_arrive_expect_tx(&raw_full[stage], tx);
            if (p.use_tma_a) tma_load_2d(ra, &map_a, &raw_full[stage], ax, ay);
            if (p.use_tma_b) tma_load_2d(rb, &map_b, &raw_full[stage], bx, by);
          } else {
            mbar_arrive(&raw_full[stage]);
          }
        }
        issued_mask |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == RAW_STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      // Let every copy this warp started land before the CTA exits.
      for (int s = 0; s < RAW_STAGES; ++s) {
        if (!(issued_mask & (1u << s))) continue;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&raw_full[s], (issued_phase >> s) & 1u) &&
               global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      uint32_t os = 0, oph = 0, ab = 0, aph = 0;
      bool ok = true;
      bool issued_any = false;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        for (int64_t c0 = 0; ok && c0 < p.num_kb; c0 += p.chunk_kb) {
          const int64_t c1 = (p.num_kb < c0 + p.chunk_kb) ? p.num_kb : c0 + p.chunk_kb;
          if (!mbar_wait(&acc_empty[ab], aph ^ 1u, abort_flag, p.err, code_base | 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + ab * BN;
          for (int64_t kb = c0; kb < c1; ++kb) {
            if (!mbar_wait(&op_full[os], oph, abort_flag, p.err, code_base | 3)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_addr(opa + os * OPA_BYTES);
            const uint32_t b0 = smem_addr(opb + os * OPB_BYTES);
#pragma unroll
            for (int j = 0; j < BK / UK; ++j) {
              umma_f16_ss(d_tmem, smem_desc_k_sw128(a0 + 32 * j), smem_desc_k_sw128(b0 + 32 * j),
                          idesc, (kb > c0 || j > 0) ? 1u : 0u);
            }
            issued_any = true;
            umma_commit(&op_empty[os]);
            if (++os == OP_STAGES) { os = 0; oph ^= 1u; }
          }
          if (!ok) break;
          umma_commit(&acc_full[ab]);
          if (++ab == ACC_BUFS) { ab = 0; aph ^= 1u; }
        }
      }
      if (!ok && issued_any) {
        // Let the tensor core finish what was issued before TMEM is released.
        umma_commit(drain_bar);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int epi_tid = threadIdx.x - kEpiWarp0 * 32;
    const bool vec_ok = (p.out_cols % 4 == 0) &&
                        (reinterpret_cast<uintptr_t>(p.out) % 16 == 0);
    const int srow = q * 32 + lane;  // staging row = TMEM lane = tile row
    uint32_t ab = 0, aph = 0, slab = 0;
    bool ok = true;
    if (p.use_tma_out && epi_tid == 0) prefetch_tensormap(&map_out);
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const int tr = tile / p.tiles_c, tcol = tile % p.tiles_c;
      const int64_t row = static_cast<int64_t>(tr) * BM + srow;
      for (int64_t c0 = 0; c0 < p.num_kb; c0 += p.chunk_kb) {
        ok = mbar_wait(&acc_full[ab], aph, abort_flag, p.err, code_base | 4);
        // One decision for all four epilogue warps: they share named barriers below.
        ok = named_bar_and(kEpiBarrier, 128, __all_sync(0xffffffffu, ok));
        if (!ok) break;
        tc_fence_after();
        const bool first = (c0 == 0);
        // A later chunk adds into what the first one stored: let those
        // stores land before the first add is issued.
        if (p.use_tma_out && c0 == p.chunk_kb && epi_tid == 0) bulk_wait_group<0>();
        for (int cb = 0; cb < BN / 32; ++cb) {
          const int64_t col0 = static_cast<int64_t>(tcol) * BN + cb * 32;
          if (col0 >= p.out_cols) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * BN + cb * 32,
                             v);
          tmem_wait_ld();
          if (p.use_tma_out) {
            uint8_t* buf = stage_out + (slab & 1) * STAGE_OUT_BYTES;
            if (epi_tid == 0) bulk_wait_group_read<1>();  // the store 2 slabs ago has read buf
            named_bar_sync(kEpiBarrier, 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const int4 val = make_int4(f32_bits_to_i32(v[4 * c]), f32_bits_to_i32(v[4 * c + 1]),
                                         f32_bits_to_i32(v[4 * c + 2]),
                                         f32_bits_to_i32(v[4 * c + 3]));
              *reinterpret_cast<int4*>(buf + sw128(srow, c)) = val;
            }
            fence_proxy_async_smem();
            named_bar_sync(kEpiBarrier, 128);
            if (epi_tid == 0) {
              if (first)
                tma_store_2d(&map_out, buf, static_cast<int>(col0), tr * BM);
              else
                tma_reduce_add_2d(&map_out, buf, static_cast<int>(col0), tr * BM);
              bulk_commit_group();
            }
            ++slab;
          } else if (row < p.out_rows) {
            const int64_t rem = p.out_cols - col0;
            store_row32(p.out + row * p.out_cols + col0, v, rem < 32 ? static_cast<int>(rem) : 32,
                        first, vec_ok);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
        if (++ab == ACC_BUFS) { ab = 0; aph ^= 1u; }
      }
    }
    if (p.use_tma_out && epi_tid == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace tc
}  // namespace t3
