// t3_tc2.cuh -- CTA-pair tensor-core pipeline for the forward and dX products
// (sm_103a: tcgen05 cta_group::2, TMEM A operand, TMA, mbarrier).
//
// What it computes: the forward product of "t27c PTX backend: ternary x int8
// GEMM kernel emitted by a .t27 spec (int8 mma.sync), ptx-run glue" ("What
// this adds": C = A.W, W from 2-bit codes decoded as (c & 1) - ((c >> 1) & 1))
// and kernel 1 of "spec(igla): hslm_bwd_ptx -- HSLM backward dX and dW as
// int8 tensor-core PTX written by t27" (dX = dY.W^T with the same codes).
//
// Why this shape.  On sm_103a the tensor core has no int8 kind, so both
// operands travel as exact f16 values.  Expanding them in shared memory costs
// more shared-memory bandwidth than the tensor core leaves free, so:
//   * two CTAs on two SMs issue one M=256 MMA (cta_group::2); each CTA holds
//     128 activation rows and half of the 192 weight rows, halving the weight
//     operand each SM must write and read;
//   * the activations are converted in registers and stored into TMEM with
//     tcgen05.st (the MMA's A operand comes from TMEM), never into shared memory;
//   * the packed weights are decoded once per tile load into the 128-byte-
//     swizzled K-major layout the tensor core reads from shared memory;
//   * stages of 128 reduction elements keep the per-stage control overhead of
//     the single-thread issue loops below the MMA time.
// Exactness: the f32 accumulator holds integers of magnitude <= 128 * 65536 =
// 2^23 per chunk of 65536 reduction elements; chunks are added in int32 by TMA
// bulk reduce-add.
//
// Roles per CTA (704 threads): warps 0-7 convert activations into TMEM, warps
// 8-15 decode weights into shared memory, warp 16 is the TMA producer, warp
// 17 issues the MMAs in the even CTA and, in the odd CTA, forwards "stage
// ready" to the even CTA (one cluster-scope arrive per stage instead of one
// per converter warp: a cluster-scope release costs the issuing thread
// hundreds of nanoseconds), warps 18-21 are the epilogue.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "t3.h"
#include "t3_common.cuh"

namespace t3 {
namespace tc2 {

constexpr int BMP = 256;        // output rows per pair tile (128 per CTA)
constexpr int BN = 192;         // output columns per pair tile
constexpr int BNH = BN / 2;     // weight rows decoded by each CTA
constexpr int BK = 128;         // reduction elements per stage
constexpr int RAW_STAGES = 4;
constexpr int OP_STAGES = 2;
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = 512;
constexpr int kAccCol = 0;                     // 2 x 192 columns
constexpr int kActCol = ACC_BUFS * BN;         // 2 x 64 columns of f16 pairs
constexpr int kActWarps = 8;                  // two per TMEM lane quadrant
constexpr int kWWarps = 8;                    // weight decode
constexpr int kConvWarps = kActWarps + kWWarps;
constexpr int kWThreads = 32 * kWWarps;
constexpr int kProducerWarp = kConvWarps;
constexpr int kMmaWarp = kConvWarps + 1;      // MMA issuer (even CTA) / forwarder (odd CTA)
constexpr int kEpiWarp0 = kConvWarps + 2;
constexpr int kThreads = 32 * (kConvWarps + 2 + 4);
constexpr int kEpiBarrier = 1;
constexpr int64_t kChunkStages = 65536 / BK;  // exact f32 chunk for ternary products

constexpr int RAW_A = 128 * BK;                 // [128 rows][128 B], 128-byte swizzle
template <int OP> struct RawW;
template <> struct RawW<kOpFwd> { static constexpr int rows = BNH, cols = BK / 4; };  // [96 n][32 B]
template <> struct RawW<kOpDx> { static constexpr int rows = BK, cols = BN / 4; };     // [128 n][48 B]

// kActBytes: bytes per raw activation element (1 for int8; 2 for the bf16
// activations the fused quantizer reads, as two 64-element boxes per stage)
template <int OP, int kActBytes = 1> struct Layout {
  static constexpr int raw_a = RAW_A * kActBytes;
  static constexpr int raw_w = RawW<OP>::rows * RawW<OP>::cols;
  static constexpr int raw_stage = ((raw_a + raw_w) + 1023) / 1024 * 1024;
  static constexpr int opb_atom = BNH * 128;          // forward: [96 rows][64 f16]
  // forward: two 64-element k atoms, K-major; dX: MN-major, per 8 n rows two
  // 64-element k atoms (the CTA's 96 k fill one and a half)
  static constexpr int opb_stage = (OP == kOpDx) ? (BK / 8) * 2048 : 2 * opb_atom;
  static constexpr int stage_out = 128 * 32 * 4;
  static constexpr int off_opb = 0;
  static constexpr int off_raw = off_opb + OP_STAGES * opb_stage;
  static constexpr int off_out = off_raw + RAW_STAGES * raw_stage;
  static constexpr int off_cs = off_out + 2 * stage_out;  // a tile's column scales
  static constexpr int off_bar = off_cs + BN * 4;
  static constexpr int n_bars = 2 * RAW_STAGES + 3 * OP_STAGES + 2 * ACC_BUFS + 1;
  static constexpr int off_misc = off_bar + 8 * n_bars;
  static constexpr int smem_alloc = off_misc + 16 + 1024;
};
static_assert(4 * 33 * 32 * 4 <= 2 * Layout<kOpFwd>::stage_out,
              "the unaligned-output epilogue's row blocks fit the staging buffers");

// Output kind of the pair pipeline: the exact int32 product, or (one exact
// chunk only, bulk stores only) the scaled forms of t3_dequant_i32.
constexpr int kOutI32 = -1;

struct Params {
  int64_t M, N, K;        // the product's M, N, K
  int64_t out_rows, out_cols;
  int64_t num_stages;     // stages along the reduction
  int tiles_r, tiles_c;
  int32_t* out;           // used when the output cannot take bulk stores
  int use_tma_out;
  int out_kind;           // kOutI32, T3_OUT_F32, T3_OUT_BF16 or T3_OUT_F32_ADD
  const float* row_scale; // [out_rows] or null (ones)
  const float* col_scale; // [out_cols] or null (ones)
  // Wp rows a TMA map cannot describe (ceil(K/4) not a multiple of 16 bytes,
  // but of 4): the weight decoders then load their words from global memory
  const uint8_t* wp;
  int64_t kb_bytes;       // ceil(K/4), the row stride of Wp
  int w_tma;              // 1: weights come by TMA with the activations
  int w_vec4;             // Wp rows 4-byte aligned: word loads (else bytes)
  // activation rows a TMA map cannot describe (their stride is not a
  // multiple of 16 bytes): the activation converters load them themselves
  const int8_t* act;      // [act_rows][act_cols]
  int64_t act_rows, act_cols;
  int act_vec4;           // activation rows 4-byte aligned: word loads (else bytes)
  int a_tma;              // 1: activations come by TMA
  int mode;               // kernel instantiation: kModeTma, kModeWGlobal, kModeAGlobal
  // Schedule: tiles [0, dp_tiles) are taken whole, round-robin over the
  // pairs; the (tile, stage) iterations of the remaining tiles are split into
  // equal contiguous ranges, one per pair (stream-K), which each pair works
  // through before its whole tiles.  Those pieces add their int32 sums onto
  // output rows that a chained grid has zeroed; when dp_tiles < tiles_r *
  // tiles_c every output write waits for that grid.
  int dp_tiles;
  // kModeBf16: the inverse row scales 127 / amax of the bf16 activations
  const float* row_inv;
  int* err;
};

// One piece of a pair's work: a tile and the range [kb0, kb1) of its
// reduction stages.  Every role of both CTAs walks the same pieces in the same
// order, so their stage rings stay in step.
struct Piece {
  int tile, kb0, kb1;
};

// Piece i (0, 1, ...) of a pair: first the pair's equal share of the split
// tiles' (tile, stage) iterations, cut at tile boundaries (at most two
// pieces: a share is shorter than a tile), then the whole tiles pair,
// pair + npairs, ... below dp_tiles.  With the split pieces first, their
// adding flushes overlap the whole tiles' work and a pair's last flush is a
// plain store.  False past the last piece.  32-bit indices suffice: a
// reduction has at most 131072 stages and the split part fewer than npairs
// tiles.
__device__ __forceinline__ bool get_piece(const Params& p, int pair, int npairs, int i, Piece& w) {
  const int S = static_cast<int>(p.num_stages);
  // first the pair's share [b, e) of the split tiles' iterations, cut at tile
  // boundaries (their flushes add, and overlap the whole tiles after them)
  const int64_t total = static_cast<int64_t>(p.tiles_r * p.tiles_c - p.dp_tiles) * S;
  const int b = static_cast<int>(total * pair / npairs);
  const int e = static_cast<int>(total * (pair + 1) / npairs);
  const int n_sk = b < e ? (e - 1) / S - b / S + 1 : 0;
  if (i < n_sk) {
    const int t = b / S + i;  // split tile, counted from dp_tiles
    const int s0 = t * S > b ? t * S : b;
    w.tile = p.dp_tiles + t;
    w.kb0 = s0 - t * S;
    w.kb1 = (e - t * S < S) ? e - t * S : S;
    return true;
  }
  // then the whole tiles pair, pair + npairs, ... below dp_tiles
  const int tile = pair + (i - n_sk) * npairs;
  if (tile >= p.dp_tiles) return false;
  w.tile = tile;
  w.kb0 = 0;
  w.kb1 = S;
  return true;
}

// End of the exact accumulation group that starts at stage c0 of a piece
// ending at kb1: groups never cross a multiple of kChunkStages.
__device__ __forceinline__ int chunk_end(int c0, int kb1) {
  const int e = (c0 / static_cast<int>(kChunkStages) + 1) * static_cast<int>(kChunkStages);
  return e < kb1 ? e : kb1;
}

// Kernel instantiations: all operands by TMA; weights from global memory as
// whole words (activations by TMA); and the general one, where each operand
// comes by TMA or from global memory as p.a_tma / p.w_tma say.
constexpr int kModeTma = 0, kModeWGlobal = 1, kModeAGlobal = 2;
// The forward with bf16 activations quantized in the converters (both
// operands by TMA, whole tiles, int32 output).
constexpr int kModeBf16 = 3;

// Scaled epilogue: y = ((float)x * rs) * cs per element, each product rounded
// to nearest (no contraction); x is the accumulator, an exact integer in f32
// when the reduction is one chunk.  Stages float (128-byte-swizzled rows of
// 32 words, like the int32 path) or bf16 ([128][64 B], unswizzled).
// cs: this block's 32 column scales, staged in shared memory.
__device__ __forceinline__ void stage_scaled(uint8_t* buf, int srow, const uint32_t (&v)[32],
                                             float rs, const float* cs, int kind) {
  float y[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) y[e] = __fmul_rn(__fmul_rn(__uint_as_float(v[e]), rs), cs[e]);
  if (kind == T3_OUT_BF16) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(y[8 * g + 2 * j], y[8 * g + 2 * j + 1]);
        w[j] = *reinterpret_cast<const uint32_t*>(&b);
      }
      sts128(buf + srow * 64 + 16 * g, w[0], w[1], w[2], w[3]);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 8; ++c)
      sts128(buf + tc::sw128(srow, c), __float_as_uint(y[4 * c]), __float_as_uint(y[4 * c + 1]),
             __float_as_uint(y[4 * c + 2]), __float_as_uint(y[4 * c + 3]));
  }
}

// ---------------------------------------------------------------- cluster

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// A signal-only arrive on a barrier of the peer CTA.  Used where the data the
// signal announces never leaves the signalling CTA's SM: the peer half of a
// pair MMA reads the odd CTA's own shared memory and TMEM, whose writers have
// already fenced them (proxy fence, tcgen05.wait::st) before handing over.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D (both CTAs' TMEM) (+)= A (both CTAs' TMEM) * B (both CTAs' smem halves)^T.
__device__ __forceinline__ void umma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` in both CTAs of the pair once all prior MMAs are complete.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(static_cast<uint16_t>(0x3))
      : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------ converters

// Four int8 b0..b3 -> f16x2 words (b0, b2) and (b1, b3), exact (same bias
// trick as tc::s8x4_to_f16, other byte pairs).
__device__ __forceinline__ void s8x4_to_f16_evenodd(uint32_t x, uint32_t& even, uint32_t& odd) {
  const uint32_t y = x ^ 0x80808080u;
  even = hsub2(prmt(y, 0x64646464u, 0x4240u), 0x64806480u);
  odd = hsub2(prmt(y, 0x64646464u, 0x4341u), 0x64806480u);
}

// The converters work in two halves: *_load reads the raw bytes and converts
// them into 32 registers as soon as the raw stage has landed, *_store writes
// them once the operand slot is free, so that the conversion stays off the
// path from the MMA's release of a slot to the slot's next use.

// Activation row -> TMEM: thread (quadrant q, half h) owns lane q*32+lane and
// reduction elements [64h, 64h+64) of the stage.  The raw tile is [128][128 B]
// in the 128-byte swizzle.  kEvenOdd: within every 16 reduction elements the
// even ones come first, then the odd ones -- the order in which the forward's
// weight decode (w_fwd_load) emits its codes; both operands of the forward
// use it, so the products and their sum are unchanged.  Otherwise natural order.
template <bool kEvenOdd>
__device__ __forceinline__ void act_load(const uint8_t* raw_a, int row, int h, uint32_t (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 x = *reinterpret_cast<const uint4*>(raw_a + tc::sw128(row, 4 * h + c));
    if (kEvenOdd) {
      s8x4_to_f16_evenodd(x.x, v[8 * c + 0], v[8 * c + 4]);
      s8x4_to_f16_evenodd(x.y, v[8 * c + 1], v[8 * c + 5]);
      s8x4_to_f16_evenodd(x.z, v[8 * c + 2], v[8 * c + 6]);
      s8x4_to_f16_evenodd(x.w, v[8 * c + 3], v[8 * c + 7]);
    } else {
      tc::s8x4_to_f16(x.x, v[8 * c + 0], v[8 * c + 1]);
      tc::s8x4_to_f16(x.y, v[8 * c + 2], v[8 * c + 3]);
      tc::s8x4_to_f16(x.z, v[8 * c + 4], v[8 * c + 5]);
      tc::s8x4_to_f16(x.w, v[8 * c + 6], v[8 * c + 7]);
    }
  }
}

// Forward weights of this CTA: packed [96 n][32 B] -> f16 [96 n][128 k] as two
// 64-k atoms.  Unit = (row, 32-bit word w of 16 codes): 768 units, exactly
// three per weight thread, so that every weight warp (two per warp scheduler)
// does the same share -- the decode is issue-bound.  A word's 16 codes go out
// as two 16-byte chunks, even codes then odd codes (the order act_load<true>
// writes the activations in): masking the word with 0x33333333 leaves code 2j
// in nibble j, ready as a byte-permute selector into the f16 high-byte table,
// without spreading the codes first.
// Lanes: one warp instruction covers rows 4g .. 4g+3 x words 0..7, so its 32
// word loads (row stride 32 B) hit 32 distinct banks, and each 8-lane store
// phase (two rows of opposite parity x words 0..3 or 4..7) hits 8 distinct
// 16-byte bank groups of the swizzled rows.
constexpr int kFwdWordUnits = BNH * (BK / 16);
static_assert(kFwdWordUnits % kWThreads == 0 && BNH % 4 == 0, "equal forward weight share");
constexpr int kFwdWordsPerThread = kFwdWordUnits / kWThreads;

__device__ __forceinline__ void fwd_word_unit(int tid, int i, int& row, int& w) {
  const int wl = tid & 31;
  const int g = i * (kWThreads / 32) + (tid >> 5);  // group of four rows
  row = 4 * g + ((wl >> 2) & 1) + 2 * ((wl >> 3) & 1);
  w = (wl & 3) + 4 * (wl >> 4);
}

// One word of 16 codes -> 8 f16x2 words: its even codes (4 words), then its
// odd codes.
__device__ __forceinline__ void decode_word_f16(uint32_t x, uint32_t* v) {
  const uint32_t e = x & 0x33333333u, o = (x >> 2) & 0x33333333u;
  const uint32_t he0 = prmt(tc::kF16HiTable, 0u, e);
  const uint32_t he1 = prmt(tc::kF16HiTable, 0u, e >> 16);
  const uint32_t ho0 = prmt(tc::kF16HiTable, 0u, o);
  const uint32_t ho1 = prmt(tc::kF16HiTable, 0u, o >> 16);
  v[0] = prmt(he0, 0u, 0x1404u);
  v[1] = prmt(he0, 0u, 0x3424u);
  v[2] = prmt(he1, 0u, 0x1404u);
  v[3] = prmt(he1, 0u, 0x3424u);
  v[4] = prmt(ho0, 0u, 0x1404u);
  v[5] = prmt(ho0, 0u, 0x3424u);
  v[6] = prmt(ho1, 0u, 0x1404u);
  v[7] = prmt(ho1, 0u, 0x3424u);
}

__device__ __forceinline__ void w_fwd_load(const uint8_t* raw_w, int tid, uint32_t (&v)[32]) {
#pragma unroll
  for (int i = 0; i < kFwdWordsPerThread; ++i) {
    int row, w;
    fwd_word_unit(tid, i, row, w);
    const uint32_t x = *reinterpret_cast<const uint32_t*>(raw_w + row * 32 + 4 * w);
    decode_word_f16(x, v + 8 * i);
  }
}

__device__ __forceinline__ void w_fwd_store(uint8_t* opb, int tid, const uint32_t (&v)[32]) {
#pragma unroll
  for (int i = 0; i < kFwdWordsPerThread; ++i) {
    int row, w;
    fwd_word_unit(tid, i, row, w);
    uint8_t* atom = opb + (w >> 2) * Layout<kOpFwd>::opb_atom;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      sts128(atom + tc::sw128(row, 2 * (w & 3) + h), v[8 * i + 4 * h], v[8 * i + 4 * h + 1],
             v[8 * i + 4 * h + 2], v[8 * i + 4 * h + 3]);
  }
}

// dX weights of CTA `rank`, MN-major: packed [128 n][48 B = the pair's 192 k],
// of which this CTA's 96 k are bytes [24 rank, 24 rank + 24) of every row ->
// f16 [n / 8][atom a][8 rows][128 B], atom a holding k in [64 a, 64 a + 64) of
// the CTA's 96 (atom 1 half used), 16-B chunk q of row r at q ^ r.  No
// transpose: the tensor core reads the weights MN-major.  Unit = (row n, word j
// of 16 codes = k in [16 j, 16 j + 16)): 768 units, three per weight thread.
// A word goes out as chunk 2j (its even codes) and chunk 2j + 1 (its odd
// codes), like the forward's decode; here that permutes the MMA's N columns
// within every 16, and the epilogue puts them back (dx_column).
// Lanes: rows vary fastest (unit u = tid + 256 i is row u % 128, word
// u / 128), so each 8-lane store phase is 8 consecutive rows of one word, 8
// distinct 16-byte bank groups.  The 4-byte loads of 32 consecutive rows (48-B
// stride) are 4-way bank conflicted; a map with conflict-free loads (8 rows x
// 4 words per warp instruction) made dX 3% slower.
constexpr int kDxWordUnits = BK * (BN / 2 / 16);
static_assert(kDxWordUnits % kWThreads == 0, "equal dX weight share per thread");
constexpr int kDxWordsPerThread = kDxWordUnits / kWThreads;
static_assert(kDxWordsPerThread * 8 <= 32, "dX weight units fit the 32 staging registers");

__device__ __forceinline__ void dx_word_unit(int tid, int i, int& n, int& j) {
  const int u = tid + i * kWThreads;
  n = u % BK;
  j = u / BK;
}

// Accumulator column holding output column e of a 32-column block.
__host__ __device__ constexpr int dx_column(int e) {
  return (e & 16) | ((e & 1) << 3) | ((e & 15) >> 1);
}

// Its inverse: the output column held by accumulator column j.
__host__ __device__ constexpr int dx_slot(int j) {
  return (j & 16) | ((j & 7) << 1) | ((j >> 3) & 1);
}

__host__ __device__ constexpr bool dx_slot_inverts_dx_column() {
  for (int e = 0; e < 32; ++e)
    if (dx_slot(dx_column(e)) != e) return false;
  return true;
}
static_assert(dx_slot_inverts_dx_column(), "dx_slot must invert dx_column");

// 32 accumulator columns of a block into v[0..31] in output-column order:
// for dX each loaded column is bound straight to the register of the output
// column it holds (v[e] = accumulator column dx_column(e)), so undoing the
// weight decode's order costs no moves and no second array.
template <int OP>
__device__ __forceinline__ void tmem_ld_block(uint32_t taddr, uint32_t (&v)[32]) {
  if (OP == kOpFwd) {
    tmem_ld_32x32b_x32(taddr, v);
    return;
  }
#define T3_SLOT(j) "=r"(v[dx_slot(j)])
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : T3_SLOT(0), T3_SLOT(1), T3_SLOT(2), T3_SLOT(3), T3_SLOT(4), T3_SLOT(5), T3_SLOT(6),
        T3_SLOT(7), T3_SLOT(8), T3_SLOT(9), T3_SLOT(10), T3_SLOT(11), T3_SLOT(12), T3_SLOT(13),
        T3_SLOT(14), T3_SLOT(15), T3_SLOT(16), T3_SLOT(17), T3_SLOT(18), T3_SLOT(19), T3_SLOT(20),
        T3_SLOT(21), T3_SLOT(22), T3_SLOT(23), T3_SLOT(24), T3_SLOT(25), T3_SLOT(26), T3_SLOT(27),
        T3_SLOT(28), T3_SLOT(29), T3_SLOT(30), T3_SLOT(31)
      : "r"(taddr));
#undef T3_SLOT
}

__device__ __forceinline__ void w_dx_load(const uint8_t* raw_w, int tid, uint32_t rank,
                                          uint32_t (&v)[32]) {
#pragma unroll
  for (int i = 0; i < kDxWordsPerThread; ++i) {
    int n, j;
    dx_word_unit(tid, i, n, j);
    const uint32_t x = *reinterpret_cast<const uint32_t*>(
        raw_w + n * (BN / 4) + 24 * static_cast<int>(rank) + 4 * j);
    decode_word_f16(x, v + 8 * i);
  }
}

// The same words as w_fwd_load / w_dx_load read, from global memory (rows
// 4-byte aligned, words past N rows or past ceil(K/4) bytes are 0, i.e. code 0).
// kWords4: rows known to be 4-byte aligned (word loads only).
template <bool kWords4>
__device__ __forceinline__ void w_words_global(const Params& p, bool fwd, int tcol, int64_t kb,
                                               uint32_t rank, int tid, uint32_t* x) {
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    int64_t n, off;
    if (fwd) {
      int row, w;
      fwd_word_unit(tid, i, row, w);
      n = static_cast<int64_t>(tcol) * BN + static_cast<int64_t>(rank) * BNH + row;
      off = kb * (BK / 4) + 4 * w;
    } else {
      int nl, j;
      dx_word_unit(tid, i, nl, j);
      n = kb * BK + nl;
      off = static_cast<int64_t>(tcol) * (BN / 4) + 24 * static_cast<int64_t>(rank) + 4 * j;
    }
    uint32_t w = 0u;
    if (n < p.N && off < p.kb_bytes) {
      const uint8_t* src = p.wp + n * p.kb_bytes + off;
      if (kWords4 || p.w_vec4) {
        w = __ldg(reinterpret_cast<const uint32_t*>(src));
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (off + j < p.kb_bytes) w |= static_cast<uint32_t>(__ldg(src + j)) << (8 * j);
      }
    }
    x[i] = w;
  }
}

// The 64 activation bytes of thread half h (reduction elements
// [kb * BK + 64 h, +64)) of row m, from global memory; 0 past the rows or the
// reduction (as TMA's zero fill).
__device__ __forceinline__ void act_words_global(const Params& p, int64_t m, int64_t kb, int h,
                                                 uint32_t (&x)[16]) {
  const int64_t k0 = kb * BK + 64 * h;
  const int8_t* rowp = p.act + m * p.act_cols;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int64_t k = k0 + 4 * i;
    uint32_t w = 0u;
    if (m < p.act_rows && k < p.act_cols) {
      if (p.act_vec4 && k + 4 <= p.act_cols) {
        w = __ldg(reinterpret_cast<const uint32_t*>(rowp + k));
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (k + j < p.act_cols)
            w |= static_cast<uint32_t>(static_cast<uint8_t>(__ldg(rowp + k + j))) << (8 * j);
      }
    }
    x[i] = w;
  }
}

// act_load's conversion, from words already in registers (x[4 c + j] holds
// elements 64 h + 16 c + 4 j .. +3).
template <bool kEvenOdd>
__device__ __forceinline__ void act_conv(const uint32_t (&x)[16], uint32_t (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (kEvenOdd) {
      s8x4_to_f16_evenodd(x[4 * c], v[8 * c + 0], v[8 * c + 4]);
      s8x4_to_f16_evenodd(x[4 * c + 1], v[8 * c + 1], v[8 * c + 5]);
      s8x4_to_f16_evenodd(x[4 * c + 2], v[8 * c + 2], v[8 * c + 6]);
      s8x4_to_f16_evenodd(x[4 * c + 3], v[8 * c + 3], v[8 * c + 7]);
    } else {
      tc::s8x4_to_f16(x[4 * c], v[8 * c + 0], v[8 * c + 1]);
      tc::s8x4_to_f16(x[4 * c + 1], v[8 * c + 2], v[8 * c + 3]);
      tc::s8x4_to_f16(x[4 * c + 2], v[8 * c + 4], v[8 * c + 5]);
      tc::s8x4_to_f16(x[4 * c + 3], v[8 * c + 6], v[8 * c + 7]);
    }
  }
}

__device__ __forceinline__ void w_dx_store(uint8_t* opb, int tid, const uint32_t (&v)[32]) {
#pragma unroll
  for (int i = 0; i < kDxWordsPerThread; ++i) {
    int n, j;
    dx_word_unit(tid, i, n, j);
    const int r = n & 7;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = 2 * j + h;
      sts128(opb + (n >> 3) * 2048 + (q >> 3) * 1024 + r * 128 + (((q & 7) ^ r) << 4),
             v[8 * i + 4 * h], v[8 * i + 4 * h + 1], v[8 * i + 4 * h + 2], v[8 * i + 4 * h + 3]);
    }
  }
}

// Two bf16 activations (the high halves of fa and fb, low halves zero) ->
// their int8 codes of the row quantizer, q = rint(fl(x * inv)), as an exact
// f16 pair (q(a) low, q(b) high).  Adding 1.5 * 2^23 + 128 rounds a product
// p, |p| <= 127.00002 (|x| <= amax, inv = fl(127 / amax)), to the nearest
// integer with ties to even, and leaves q + 128 in the low 10 bits of the sum;
// f16 0x6400 | (q + 128) is 1024 + q + 128, and subtracting 1152 leaves q.
// No clamp is needed: |rint(p)| <= 127.
__device__ __forceinline__ uint32_t quant_pair_f16(uint32_t fa, uint32_t fb, float inv) {
  const float ta = __fadd_rn(__fmul_rn(__uint_as_float(fa), inv), 12583040.0f);
  const float tb = __fadd_rn(__fmul_rn(__uint_as_float(fb), inv), 12583040.0f);
  const uint32_t packed = (__float_as_uint(ta) & 0x3FFu) | ((__float_as_uint(tb) & 0x3FFu) << 16);
  return hsub2(packed | 0x64006400u, 0x64806480u);
}

// The same for a row whose inverse scale is infinite (amax so small that
// 127 / amax overflows): x * inf is +-inf, clamped to +-127, and 0 * inf counts
// as 0.
__device__ __forceinline__ uint32_t quant_pair_f16_inf(uint32_t fa, uint32_t fb) {
  const float a = __uint_as_float(fa), b = __uint_as_float(fb);
  const uint32_t ua = a > 0.0f ? 255u : (a < 0.0f ? 1u : 128u);
  const uint32_t ub = b > 0.0f ? 255u : (b < 0.0f ? 1u : 128u);
  return hsub2((ua | (ub << 16)) | 0x64006400u, 0x64806480u);
}

// bf16 activation row -> quantized f16 pairs for TMEM: thread (quadrant q,
// half h) owns row `row` and reduction elements [64h, 64h+64) of the stage,
// which are box h of the raw stage ([128 rows][128 B] in the 128-byte
// swizzle).  Same order as act_load<true>: within every 16 elements the even
// ones first, then the odd ones.
__device__ __forceinline__ void act_load_bf16(const uint8_t* raw_a, int row, int h, float inv,
                                              bool inv_finite, uint32_t (&v)[32]) {
  const uint8_t* box = raw_a + h * RAW_A;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    // 16 elements: words w[2j], w[2j+1] hold elements (4j, 4j+1), (4j+2, 4j+3)
    const uint4 x0 = *reinterpret_cast<const uint4*>(box + tc::sw128(row, 2 * c));
    const uint4 x1 = *reinterpret_cast<const uint4*>(box + tc::sw128(row, 2 * c + 1));
    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t ea = w[2 * j] << 16, eb = w[2 * j + 1] << 16;                 // 4j, 4j+2
      const uint32_t oa = w[2 * j] & 0xFFFF0000u, ob = w[2 * j + 1] & 0xFFFF0000u;  // 4j+1, 4j+3
      if (inv_finite) {
        v[8 * c + j] = quant_pair_f16(ea, eb, inv);
        v[8 * c + 4 + j] = quant_pair_f16(oa, ob, inv);
      } else {
        v[8 * c + j] = quant_pair_f16_inf(ea, eb);
        v[8 * c + 4 + j] = quant_pair_f16_inf(oa, ob);
      }
    }
  }
}

// How many stages one pair runs in all (whole tiles and stream-K pieces).
__device__ __forceinline__ int64_t pair_stage_count(const Params& p, int pair, int npairs) {
  const int64_t whole = pair < p.dp_tiles ? (p.dp_tiles - 1 - pair) / npairs + 1 : 0;
  const int64_t total = static_cast<int64_t>(p.tiles_r * p.tiles_c - p.dp_tiles) * p.num_stages;
  return whole * p.num_stages + total * (pair + 1) / npairs - total * pair / npairs;
}

// ------------------------------------------------------------------ kernel

// kSplit: the split schedule (operands by TMA only); without it every pair
// takes whole tiles and the loops below reduce to plain tile loops.
template <int OP, int kMode, bool kSplit>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc2_kernel(const Params p, const __grid_constant__ CUtensorMap map_a,
               const __grid_constant__ CUtensorMap map_w,
               const __grid_constant__ CUtensorMap map_out) {
  static_assert(!kSplit || kMode == kModeTma, "the split schedule takes TMA operands");
  static_assert(kMode != kModeBf16 || (OP == kOpFwd && !kSplit), "bf16 activations: forward, whole tiles");
  using L = Layout<OP, kMode == kModeBf16 ? 2 : 1>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((base_addr + 1023u) & ~1023u) - base_addr);
  uint8_t* opb = smem + L::off_opb;
  uint8_t* raw = smem + L::off_raw;
  uint8_t* stage_out = smem + L::off_out;
  float* cs_tile = reinterpret_cast<float*>(smem + L::off_cs);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::off_bar);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + RAW_STAGES;
  uint64_t* op_full = raw_empty + RAW_STAGES;   // leader: 16 arrivals (8 warps x 2 CTAs)
  uint64_t* op_empty = op_full + OP_STAGES;     // both: MMA commit (multicast)
  uint64_t* acc_full = op_empty + OP_STAGES;    // both: MMA commit (multicast)
  uint64_t* acc_empty = acc_full + ACC_BUFS;    // leader: 8 arrivals (4 warps x 2 CTAs)
  uint64_t* op_ready = acc_empty + ACC_BUFS;    // odd CTA: its converters, before forwarding
  uint64_t* drain_bar = op_ready + OP_STAGES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::off_misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int num_tiles = p.tiles_r * p.tiles_c;
  const int code_base = (OP + 4) << 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW_STAGES; ++s) {
      mbar_init(&raw_full[s], 1);
      // without weight TMA only the activation warps read the raw stages
      // the warps that read the raw stages release them
      const int readers = (p.a_tma ? kActWarps : 0) + (p.w_tma ? kWWarps : 0);
      mbar_init(&raw_empty[s], (kMode == kModeTma || kMode == kModeBf16) ? kConvWarps
                               : kMode == kModeWGlobal ? kActWarps
                               : (readers > 0 ? readers : 1));
    }
    for (int s = 0; s < OP_STAGES; ++s) {
      mbar_init(&op_full[s], kConvWarps + 1);  // own converters + the odd CTA's forwarder
      mbar_init(&op_empty[s], 1);
      mbar_init(&op_ready[s], kConvWarps);
    }
    for (int s = 0; s < ACC_BUFS; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 8);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp < kConvWarps) {
    // ---------------------------------------------------------- converters
    const bool act_warp = warp < kActWarps;
    const int q = warp & 3, h = (warp >> 2) & 1;
    const int row = q * 32 + lane;
    const int wtid = threadIdx.x - kActWarps * 32;
    uint64_t* signal = (rank == 0) ? op_full : op_ready;  // local, CTA scope
    uint32_t rs = 0, rph = 0, os = 0, oph = 0;
    bool ok = true;
    static_assert(kFwdWordsPerThread == 3 && kDxWordsPerThread == 3, "three words per thread");
    // weights from global memory: this stage's words, loaded during the
    // previous stage (while that one waited for its operand slot)
    const bool wg = kMode == kModeWGlobal || (kMode == kModeAGlobal && !p.w_tma);
    const bool w_global = wg && !act_warp;
    const bool a_global = kMode == kModeAGlobal && act_warp && !p.a_tma;
    uint32_t ax[16];  // a_global: this stage's activation words, loaded a stage ahead
    if (a_global && pair < num_tiles)
      act_words_global(p, static_cast<int64_t>(pair / p.tiles_c) * BMP + rank * 128 + row, 0, h, ax);
    uint32_t wx[3] = {0u, 0u, 0u};
    if (w_global && pair < num_tiles)
      w_words_global<kMode == kModeWGlobal>(p, OP == kOpFwd, pair % p.tiles_c, 0, rank, wtid, wx);
    // the split schedule only needs the count of the pair's stages here
    int64_t left = kSplit ? pair_stage_count(p, pair, npairs) : 0;
    for (int tile = pair; ok && tile < (kSplit ? pair + 1 : num_tiles); tile += npairs) {
      // bf16 activations: this thread's row's inverse scale
      float row_inv = 0.0f;
      bool inv_finite = true;
      if constexpr (kMode == kModeBf16) {
        const int64_t m = static_cast<int64_t>(tile / p.tiles_c) * BMP + rank * 128 + row;
        row_inv = (act_warp && m < p.M) ? __ldg(p.row_inv + m) : 0.0f;
        inv_finite = row_inv <= 3.402823466e38f;  // false for +inf
      }
      for (int64_t kb = 0; kSplit ? left-- > 0 : kb < p.num_stages; ++kb) {
        const uint8_t* ra = raw + rs * L::raw_stage;
        const uint32_t act_taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kActCol +
                                   os * (BK / 2) + 32 * h;
        if (kMode == kModeAGlobal && a_global) {
          uint32_t v[32];
          act_conv<OP == kOpFwd>(ax, v);
          // the next stage's words go in flight now
          const bool last_kb = kb + 1 == p.num_stages;
          const int ntile = last_kb ? tile + npairs : tile;
          if (ntile < num_tiles)
            act_words_global(p, static_cast<int64_t>(ntile / p.tiles_c) * BMP + rank * 128 + row,
                             last_kb ? 0 : kb + 1, h, ax);
          ok = mbar_wait(&op_empty[os], oph ^ 1u, abort_flag, p.err, code_base | 2);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tmem_st_32x32b_x32(act_taddr, v);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&signal[os]);
          if (++rs == RAW_STAGES) { rs = 0; rph ^= 1u; }
          if (++os == OP_STAGES) { os = 0; oph ^= 1u; }
          continue;
        }
        if (kMode != kModeTma && w_global) {
          uint32_t v[32];
#pragma unroll
          for (int i = 0; i < 3; ++i) decode_word_f16(wx[i], v + 8 * i);
          // the next stage's words go in flight now
          const bool last_kb = kb + 1 == p.num_stages;
          const int ntile = last_kb ? tile + npairs : tile;
          if (ntile < num_tiles)
            w_words_global<kMode == kModeWGlobal>(p, OP == kOpFwd, ntile % p.tiles_c, last_kb ? 0 : kb + 1, rank, wtid, wx);
          ok = mbar_wait(&op_empty[os], oph ^ 1u, abort_flag, p.err, code_base | 2);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          if (OP == kOpFwd)
            w_fwd_store(opb + os * L::opb_stage, wtid, v);
          else
            w_dx_store(opb + os * L::opb_stage, wtid, v);
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&signal[os]);
          if (++rs == RAW_STAGES) { rs = 0; rph ^= 1u; }
          if (++os == OP_STAGES) { os = 0; oph ^= 1u; }
          continue;
        }
        // convert as soon as the raw stage is in, release it, and wait for the
        // operand slot only before storing: the two-slot ring runs latency-bound
        // on the slot hand-off, which the conversion then stays off
        ok = mbar_wait(&raw_full[rs], rph, abort_flag, p.err, code_base | 2);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        uint32_t v[32];
        if (act_warp) {
          if constexpr (kMode == kModeBf16)
            act_load_bf16(ra, row, h, row_inv, inv_finite, v);
          else
            act_load<OP == kOpFwd>(ra, row, h, v);
        } else if (OP == kOpFwd) {
          w_fwd_load(ra + L::raw_a, wtid, v);
        } else {
          w_dx_load(ra + L::raw_a, wtid, rank, v);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rs]);
        ok = mbar_wait(&op_empty[os], oph ^ 1u, abort_flag, p.err, code_base | 2);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        if (act_warp) {
          tmem_st_32x32b_x32(act_taddr, v);
          tmem_wait_st();
        } else {
          if (OP == kOpFwd)
            w_fwd_store(opb + os * L::opb_stage, wtid, v);
          else
            w_dx_store(opb + os * L::opb_stage, wtid, v);
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&signal[os]);
        if (++rs == RAW_STAGES) { rs = 0; rph ^= 1u; }
        if (++os == OP_STAGES) { os = 0; oph ^= 1u; }
      }
    }
  } else if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    const bool wg_p = kMode == kModeWGlobal || (kMode == kModeAGlobal && !p.w_tma);
    // with both operands from global memory there is nothing to copy
    const bool ag_p = kMode == kModeAGlobal && !p.a_tma;
    const bool idle = ag_p && wg_p;
    if (lane == 0 && !idle) {
      if (!ag_p) prefetch_tensormap(&map_a);
      if (!wg_p) prefetch_tensormap(&map_w);
    }
    uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
    bool ok = true;
    Piece w{pair, 0, 0};
    for (int i = 0, tile = pair; ok && !idle; ++i, tile += npairs) {
      int64_t kb0 = 0, kb1 = p.num_stages;
      if constexpr (kSplit) {
        if (!get_piece(p, pair, npairs, i, w)) break;
        tile = w.tile;
        kb0 = w.kb0;
        kb1 = w.kb1;
      } else {
        if (tile >= num_tiles) break;
      }
      const int tr = tile / p.tiles_c, tcol = tile % p.tiles_c;
      const int ay = tr * BMP + static_cast<int>(rank) * 128;
      int wx, wy;  // weight box origin and its per-stage step
      if (OP == kOpFwd) {
        wx = 0;
        wy = tcol * BN + static_cast<int>(rank) * BNH;
      } else {
        wx = tcol * (BN / 4);
        wy = 0;
      }
      for (int64_t kb = kb0; kb < kb1; ++kb) {
        if (lane == 0)
          ok = mbar_wait(&raw_empty[stage], phase ^ 1u, abort_flag, p.err, code_base | 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* dst = raw + stage * L::raw_stage;
          mbar_arrive_expect_tx(&raw_full[stage], (ag_p ? 0 : L::raw_a) + (wg_p ? 0 : L::raw_w));
          if (kMode == kModeBf16) {
            // two boxes of 64 bf16 (128 B) x 128 rows
            tma_load_2d(dst, &map_a, &raw_full[stage], static_cast<int>(kb * BK), ay);
            tma_load_2d(dst + RAW_A, &map_a, &raw_full[stage], static_cast<int>(kb * BK + BK / 2), ay);
          } else if (!ag_p) {
            tma_load_2d(dst, &map_a, &raw_full[stage], static_cast<int>(kb * BK), ay);
          }
          if (!wg_p) {
            if (OP == kOpFwd)
              tma_load_2d(dst + L::raw_a, &map_w, &raw_full[stage], static_cast<int>(kb * (BK / 4)), wy);
            else
              tma_load_2d(dst + L::raw_a, &map_w, &raw_full[stage], wx, static_cast<int>(kb * BK));
          }
        }
        issued_mask |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == RAW_STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      for (int s = 0; s < RAW_STAGES; ++s) {
        if (!(issued_mask & (1u << s))) continue;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&raw_full[s], (issued_phase >> s) & 1u) &&
               global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------- MMA (even CTA)
    if (rank == 0 && lane == 0) {
      // the dX weights are MN-major (instruction-descriptor bit 16)
      constexpr uint32_t idesc = idesc_f16_f32(BMP, BN) | (OP == kOpDx ? (1u << 16) : 0u);
      uint32_t os = 0, oph = 0, ab = 0, aph = 0;
      bool ok = true, issued_any = false;
      Piece w{pair, 0, 0};
      for (int i = 0, tile = pair; ok; ++i, tile += npairs) {
        int64_t kb0 = 0, kb1 = p.num_stages;
        if constexpr (kSplit) {
          if (!get_piece(p, pair, npairs, i, w)) break;
          kb0 = w.kb0;
          kb1 = w.kb1;
        } else {
          if (tile >= num_tiles) break;
        }
        for (int64_t c0 = kb0, c1; ok && c0 < kb1; c0 = c1) {
          c1 = kSplit ? chunk_end(static_cast<int>(c0), static_cast<int>(kb1))
                      : ((kb1 < c0 + kChunkStages) ? kb1 : c0 + kChunkStages);
          ok = mbar_wait(&acc_empty[ab], aph ^ 1u, abort_flag, p.err, code_base | 3);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + kAccCol + ab * BN;
          for (int64_t kb = c0; kb < c1; ++kb) {
            ok = mbar_wait(&op_full[os], oph, abort_flag, p.err, code_base | 3);
            if (!ok) break;
            tc_fence_after();
            const uint32_t b0 = smem_addr(opb + os * L::opb_stage);
            const uint32_t a0 = tmem_base + kActCol + os * (BK / 2);
#pragma unroll
            for (int j = 0; j < BK / 16; ++j) {
              // K-step j: forward weights K-major (atom j/4, 32 B further per
              // step); dX weights MN-major (two 8-row n groups further per step)
              const uint64_t bdesc =
                  (OP == kOpDx)
                      ? smem_desc_mn_sw128(b0 + j * 4096, 1024, 2048)
                      : smem_desc_k_sw128(b0 + (j >> 2) * L::opb_atom + 32 * (j & 3));
              umma_pair_ts(d_tmem, a0 + 8 * j, bdesc, idesc, (kb > c0 || j > 0) ? 1u : 0u);
            }
            issued_any = true;
            umma_commit_pair(&op_empty[os]);
            if (++os == OP_STAGES) { os = 0; oph ^= 1u; }
          }
          if (!ok) break;
          umma_commit_pair(&acc_full[ab]);
          if (++ab == ACC_BUFS) { ab = 0; aph ^= 1u; }
        }
      }
      if (!ok && issued_any) {
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(drain_bar))
            : "memory");
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    if (rank == 1 && lane == 0) {
      // forward each stage's readiness to the even CTA's MMA issuer
      const uint32_t op_full_leader0 = peer_addr(&op_full[0], 0);
      uint32_t os = 0, oph = 0;
      bool ok = true;
      Piece w{pair, 0, 0};
      for (int i = 0, tile = pair; ok; ++i, tile += npairs) {
        int64_t kb0 = 0, kb1 = p.num_stages;
        if constexpr (kSplit) {
          if (!get_piece(p, pair, npairs, i, w)) break;
          kb0 = w.kb0;
          kb1 = w.kb1;
        } else {
          if (tile >= num_tiles) break;
        }
        for (int64_t kb = kb0; kb < kb1; ++kb) {
          ok = mbar_wait(&op_ready[os], oph, abort_flag, p.err, code_base | 5);
          if (!ok) break;
          mbar_arrive_cluster_relaxed(op_full_leader0 + 8u * os);
          if (++os == OP_STAGES) { os = 0; oph ^= 1u; }
        }
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int epi_tid = threadIdx.x - kEpiWarp0 * 32;
    const int srow = q * 32 + lane;
    const uint32_t acc_empty_leader0 = peer_addr(&acc_empty[0], 0);
    uint32_t ab = 0, aph = 0, slab = 0;
    bool ok = true;
    if (p.use_tma_out && epi_tid == 0) prefetch_tensormap(&map_out);
    // split schedule: the zeroing grid launched just before has finished
    // before the first output write
    if (kSplit) grid_dependency_wait();
    Piece w{pair, 0, 0};
    for (int i = 0, tile = pair; ok; ++i, tile += npairs) {
      int64_t kb0 = 0, kb1 = p.num_stages;
      if constexpr (kSplit) {
        if (!get_piece(p, pair, npairs, i, w)) break;
        tile = w.tile;
        kb0 = w.kb0;
        kb1 = w.kb1;
      } else {
        if (tile >= num_tiles) break;
      }
      const int tr = tile / p.tiles_c, tcol = tile % p.tiles_c;
      const int row0 = tr * BMP + static_cast<int>(rank) * 128;
      const int64_t row = static_cast<int64_t>(row0) + srow;
      const float rs =
          (p.out_kind != kOutI32 && p.row_scale && row < p.out_rows) ? __ldg(p.row_scale + row) : 1.0f;
      for (int64_t c0 = kb0, c1; c0 < kb1; c0 = c1) {
        c1 = kSplit ? chunk_end(static_cast<int>(c0), static_cast<int>(kb1))
                    : ((kb1 < c0 + kChunkStages) ? kb1 : c0 + kChunkStages);
        ok = mbar_wait(&acc_full[ab], aph, abort_flag, p.err, code_base | 4);
        ok = named_bar_and(kEpiBarrier, 128, __all_sync(0xffffffffu, ok));
        if (!ok) break;
        tc_fence_after();
        // a whole tile's first chunk is stored; its later chunks, and every
        // stream-K piece, are added
        const bool sk = kSplit && tile >= p.dp_tiles;
        const bool first = !sk && c0 == 0;
        if (p.use_tma_out && !sk && c0 == kChunkStages && epi_tid == 0) bulk_wait_group<0>();
        if (p.out_kind != kOutI32) {
          // the tile's column scales, once (the barrier above ends the previous
          // tile's reads of them)
          for (int j = epi_tid; j < BN; j += 128) {
            const int64_t col = static_cast<int64_t>(tcol) * BN + j;
            cs_tile[j] = p.col_scale ? (col < p.out_cols ? __ldg(p.col_scale + col) : 0.0f) : 1.0f;
          }
          named_bar_sync(kEpiBarrier, 128);
        }
        for (int cb = 0; cb < BN / 32; ++cb) {
          const int64_t col0 = static_cast<int64_t>(tcol) * BN + cb * 32;
          if (col0 >= p.out_cols) break;
          uint32_t v[32];
          tmem_ld_block<OP>(
              tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kAccCol + ab * BN + cb * 32, v);
          tmem_wait_ld();
          if (p.use_tma_out) {
            uint8_t* buf = stage_out + (slab & 1) * L::stage_out;
            if (epi_tid == 0) bulk_wait_group_read<1>();
            named_bar_sync(kEpiBarrier, 128);
            if (p.out_kind == kOutI32) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const int4 val =
                    make_int4(tc::f32_bits_to_i32(v[4 * c]), tc::f32_bits_to_i32(v[4 * c + 1]),
                              tc::f32_bits_to_i32(v[4 * c + 2]), tc::f32_bits_to_i32(v[4 * c + 3]));
                sts128(buf + tc::sw128(srow, c), val);
              }
            } else {
              stage_scaled(buf, srow, v, rs, cs_tile + cb * 32, p.out_kind);
            }
            fence_proxy_async_smem();
            named_bar_sync(kEpiBarrier, 128);
            if (epi_tid == 0) {
              // the tensor map carries the element type: int32, f32 or bf16
              if ((p.out_kind == kOutI32 && !first) || p.out_kind == T3_OUT_F32_ADD)
                tma_reduce_add_2d(&map_out, buf, static_cast<int>(col0), row0);
              else
                tma_store_2d(&map_out, buf, static_cast<int>(col0), row0);
              bulk_commit_group();
            }
            ++slab;
          } else {
            // rows TMA cannot address (int32 only): row by row through this
            // warp's part of the idle staging buffers; stream-K pieces add
            // atomically (other pairs add into the same elements)
            uint32_t* scratch = reinterpret_cast<uint32_t*>(stage_out) + q * (33 * 32);
            tc::out_block32(scratch, v, lane, p.out, p.out_cols, row0 + q * 32, p.out_rows, col0,
                            p.out_cols, sk ? tc::kOutAtomicAdd : (first ? tc::kOutStore : tc::kOutAdd));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_leader0 + 8u * ab);
        if (++ab == ACC_BUFS) { ab = 0; aph ^= 1u; }
      }
    }
    if (p.use_tma_out && epi_tid == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's TMEM and barriers stay alive until both CTAs are done
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace tc2
}  // namespace t3
