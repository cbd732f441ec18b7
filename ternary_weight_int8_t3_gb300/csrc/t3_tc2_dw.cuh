// t3_tc2_dw.cuh -- CTA-pair tensor-core pipeline for the dW product
// (sm_103a: tcgen05 cta_group::2 with both operands MN-major in shared memory,
// TMA, mbarrier).
//
// What it computes: kernel 2 of "spec(igla): hslm_bwd_ptx -- HSLM backward dX
// and dW as int8 tensor-core PTX written by t27": dW[k][n] = sum_m A[m][k] dY[m][n],
// int8 x int8 -> int32.
//
// Why this shape.  Both operands arrive with the reduction index m as their
// row: A [M][K] and dY [M][N] are MN-major for the tensor core.  tcgen05
// reads MN-major operands from shared memory directly (instruction-descriptor
// bits 15/16), so the converters only widen int8 to f16 in place and never
// transpose.  Shared-memory bytes, not the tensor core, bound these kernels, so:
//   * two CTAs on two SMs issue one M=256 N=256 MMA (cta_group::2); each CTA
//     holds 128 dW rows (k) of A and 128 dW columns (n) of dY, half of what a
//     single CTA would have to write and read for the same product tile;
//   * a 256 x 256 tile per pair covers the 1280 x 3456 output of the layer in
//     one wave of pairs.
// MN-major 128-byte-swizzle layout (measured on the GPU): an atom is 8 rows of
// the reduction (m) x 64 f16 along MN (128 B per row, 16-B chunk c of row r at
// c ^ r); the descriptor's leading offset is the stride between atoms along MN
// (1 KB here), its stride offset the stride between 8-row groups along m (2 KB).
// Exactness: each product is at most 2^14 in magnitude, so a chunk of 1024
// reduction elements sums to at most 2^24 in f32, exactly; chunks are added in
// int32 by TMA bulk reduce-add onto an output that a zeroing grid cleared.
// Work units are (tile, chunk) pairs, numbered tile-major and dealt to the CTA
// pairs in equal contiguous ranges: 70 tiles x 16 chunks of the layer above
// give every pair 14 or 15 units instead of one whole tile to 70 of 76 pairs.
// A pair takes its units chunk-first, so that all pairs sweep the reduction
// together and the inputs they read at one time stay few.
//
// Roles per CTA (704 threads): warps 0-7 convert A, warps 8-15 convert dY,
// warp 16 is the TMA producer, warp 17 issues the MMAs (even CTA) or forwards
// the odd CTA's "stage ready" to the even CTA with one cluster arrive per
// stage, warps 18-21 are the epilogue.
#pragma once
#include <cstdint>
#include "t3_tc2.cuh"

namespace t3 {
namespace dw2 {

constexpr int BMP = 256;        // dW rows (k) per pair tile, 128 per CTA
constexpr int BN = 256;         // dW columns (n) per pair tile, 128 per CTA
constexpr int BNH = BN / 2;
constexpr int BK = 128;         // reduction elements (m) per stage
constexpr int RAW_STAGES = 2;
constexpr int OP_STAGES = 2;    // converted stages (64 KB each)
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = ACC_BUFS * BN;  // 512
constexpr int kConvWarps = 16;            // 8 for A, 8 for dY
constexpr int kHalfThreads = 32 * kConvWarps / 2;
constexpr int kProducerWarp = kConvWarps;
constexpr int kMmaWarp = kConvWarps + 1;
constexpr int kEpiWarp0 = kConvWarps + 2;
constexpr int kThreads = 32 * (kConvWarps + 2 + 4);
constexpr int kEpiBarrier = 1;
constexpr int kChunkElems = 1024;  // exact f32 chunk for int8 x int8 (|sum| <= 2^24)

constexpr int RAW_OP = BK * 128;            // one operand's raw box [128 m][128 B]
constexpr int RAW_STAGE = 2 * RAW_OP;       // A then dY
constexpr int MN_ATOM = 1024;               // 8 m rows x 128 B
constexpr int K_GROUP = 2 * MN_ATOM;        // two MN atoms (128 f16) per 8 m rows
constexpr int OP_OPERAND = (BK / 8) * K_GROUP;  // 32 KB of f16 per operand
constexpr int OP_STAGE = 2 * OP_OPERAND;
constexpr int STAGE_OUT = 128 * 32 * 4;
constexpr int OFF_OP = 0;
constexpr int OFF_RAW = OFF_OP + OP_STAGES * OP_STAGE;
constexpr int OFF_OUT = OFF_RAW + RAW_STAGES * RAW_STAGE;
constexpr int OFF_BAR = OFF_OUT + 2 * STAGE_OUT;
constexpr int N_BARS = 2 * RAW_STAGES + 3 * OP_STAGES + 2 * ACC_BUFS + 1;
constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
static_assert(4 * 33 * 32 * 4 <= 2 * STAGE_OUT, "unaligned-output row blocks fit the staging buffers");

struct Params {
  int64_t M, N, K;       // the product's sizes: reduction M, dW [K][N]
  int64_t num_stages;    // stages along the reduction
  int tiles_r, tiles_c;  // tiles along k, along n
  int num_chunks;        // exact chunks along the reduction
  // operands a TMA map cannot describe (row stride or base not 16-byte
  // aligned): the converters load them from global memory (kGlobal)
  const int8_t* a;       // [M][K]
  const int8_t* dy;      // [M][N]
  int a_vec4, dy_vec4;   // rows 4-byte aligned: word loads (else bytes)
  int32_t* out;          // dW, for per-element adds when it cannot take bulk adds
  int use_tma_out;
  int global_ops;        // 1: the kGlobal instantiation
  int* err;
};

// 16 bytes of row m, columns [col, col + 16), from global memory; 0 past the
// rows or columns (as TMA's zero fill).
__device__ __forceinline__ uint4 row16_global(const int8_t* base, int64_t rows, int64_t cols,
                                              int vec4, int64_t m, int64_t col) {
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if (m < rows) {
    const int8_t* rowp = base + m * cols;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t k = col + 4 * i;
      if (vec4 && k + 4 <= cols) {
        w[i] = __ldg(reinterpret_cast<const uint32_t*>(rowp + k));
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (k + j < cols)
            w[i] |= static_cast<uint32_t>(static_cast<uint8_t>(__ldg(rowp + k + j))) << (8 * j);
      }
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The (tile, chunk) units of one CTA pair: tile-major numbers [u0, u1).
struct Units {
  int64_t u0, u1;
  int nc, t0, t1;
  __device__ __forceinline__ Units(const Params& p, int pair, int npairs) {
    nc = p.num_chunks;
    const int64_t total = static_cast<int64_t>(p.tiles_r) * p.tiles_c * nc;
    u0 = total * pair / npairs;
    u1 = total * (pair + 1) / npairs;
    t0 = static_cast<int>(u0 / nc);
    t1 = static_cast<int>((u1 - 1) / nc);
  }
  __device__ __forceinline__ bool has(int t, int c) const {
    const int64_t u = static_cast<int64_t>(t) * nc + c;
    return u >= u0 && u < u1;
  }
};

// D (both CTAs' TMEM) (+)= A (both CTAs' shared memory) x B (both CTAs' shared
// memory), both descriptors MN-major.
__device__ __forceinline__ void umma_pair_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor: f16 x f16 -> f32, A and B MN-major.
__host__ __device__ constexpr uint32_t idesc_f16_mn(int m, int n) {
  return (1u << 4) | (1u << 15) | (1u << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// One unit of one operand's stage: raw int8 row m (of 128), 16-byte chunk c
// (16 MN values) -> two 8-value f16 chunks 2c, 2c+1 of MN-major atom c/4
// (widen_store: the stores of the widened chunks lo, hi).
// Threads c >= 4 write their odd chunk first so that each 8-thread store
// phase hits 8 distinct bank groups.
__device__ __forceinline__ void widen_store(const uint4 lo, const uint4 hi, int m, int c,
                                            uint8_t* op) {
  const int r = m & 7;
  uint8_t* row = op + (m >> 3) * K_GROUP + (c >> 2) * MN_ATOM + r * 128;
  // selects, not a branch: a branch on c would split every warp and issue
  // each store twice with half of the threads
  const bool odd_first = c >= 4;
  const int c0 = (2 * c) & 7, c1 = (2 * c + 1) & 7;
  const int f = odd_first ? c1 : c0, g = odd_first ? c0 : c1;
  const uint4 first = odd_first ? hi : lo, second = odd_first ? lo : hi;
  sts128(row + ((f ^ r) << 4), first);
  sts128(row + ((g ^ r) << 4), second);
}

__device__ __forceinline__ void widen_regs(uint4 x, uint4& lo, uint4& hi) {
  tc::s8x4_to_f16(x.x, lo.x, lo.y);
  tc::s8x4_to_f16(x.y, lo.z, lo.w);
  tc::s8x4_to_f16(x.z, hi.x, hi.y);
  tc::s8x4_to_f16(x.w, hi.z, hi.w);
}

__device__ __forceinline__ void widen_unit(uint4 x, int m, int c, uint8_t* op) {
  uint4 lo, hi;
  widen_regs(x, lo, hi);
  widen_store(lo, hi, m, c, op);
}

// Unit (row m, chunk c) of a raw stage [128 m][128 MN], widened in registers.
__device__ __forceinline__ void widen_load(const uint8_t* raw, int m, int c, uint4& lo, uint4& hi) {
  widen_regs(*reinterpret_cast<const uint4*>(raw + m * 128 + 16 * c), lo, hi);
}

// (row m, 16-byte chunk c) units of one operand's stage, four per converter thread
constexpr int kUnitsPerThread = BK * 8 / kHalfThreads;
static_assert(kUnitsPerThread == 4, "four units per converter thread");

// kGlobal: the instantiation whose converters load the operands from global
// memory (no raw stages, an idle producer).
template <int CHUNK, bool kGlobal>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    dw2_kernel(const Params p, const __grid_constant__ CUtensorMap map_a,
               const __grid_constant__ CUtensorMap map_dy,
               const __grid_constant__ CUtensorMap map_out) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((base_addr + 1023u) & ~1023u) - base_addr);
  uint8_t* op = smem + OFF_OP;
  uint8_t* raw = smem + OFF_RAW;
  uint8_t* stage_out = smem + OFF_OUT;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + RAW_STAGES;
  uint64_t* op_full = raw_empty + RAW_STAGES;   // even CTA: both CTAs' converters
  uint64_t* op_empty = op_full + OP_STAGES;     // both: MMA commit (multicast)
  uint64_t* acc_full = op_empty + OP_STAGES;    // both: MMA commit (multicast)
  uint64_t* acc_empty = acc_full + ACC_BUFS;    // even CTA: 4 epilogue warps x 2 CTAs
  uint64_t* op_ready = acc_empty + ACC_BUFS;    // odd CTA: its converters, before forwarding
  uint64_t* drain_bar = op_ready + OP_STAGES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc2::cluster_rank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const Units units(p, pair, npairs);
  constexpr int64_t kChunkStages = CHUNK / BK;
  constexpr int code_base = 7 << 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW_STAGES; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kConvWarps);
    }
    for (int s = 0; s < OP_STAGES; ++s) {
      mbar_init(&op_full[s], kConvWarps + 1);  // own converters + the odd CTA's forwarder
      mbar_init(&op_ready[s], kConvWarps);
      mbar_init(&op_empty[s], 1);
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
    tc2::tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tc2::tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc2::cluster_sync();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp < kConvWarps) {
    // ---------------------------------------------------------- converters
    const bool a_warp = warp < kConvWarps / 2;
    const int htid = a_warp ? threadIdx.x : threadIdx.x - kHalfThreads;
    uint64_t* signal = (rank == 0) ? op_full : op_ready;  // local, CTA scope
    uint32_t rs = 0, rph = 0, os = 0, oph = 0;
    bool ok = true;
    for (int c = 0; ok && c < units.nc; ++c)
    for (int tile = units.t0; ok && tile <= units.t1; ++tile) {
      if (!units.has(tile, c)) continue;
      const int64_t k1 = min(p.num_stages, (c + 1) * kChunkStages);
      for (int64_t kb = c * kChunkStages; kb < k1; ++kb) {
        if (kGlobal) {
          // this stage's units go in flight before the wait for the slot
          const int tr = tile / p.tiles_c, tcol = tile % p.tiles_c;
          uint4 x[kUnitsPerThread];
#pragma unroll
          for (int i = 0; i < kUnitsPerThread; ++i) {
            const int u = htid + i * kHalfThreads, m = u >> 3, cc = u & 7;
            const int64_t mg = kb * BK + m;
            x[i] = a_warp ? row16_global(p.a, p.M, p.K, p.a_vec4, mg,
                                         static_cast<int64_t>(tr) * BMP + rank * 128 + 16 * cc)
                          : row16_global(p.dy, p.M, p.N, p.dy_vec4, mg,
                                         static_cast<int64_t>(tcol) * BN + rank * BNH + 16 * cc);
          }
          ok = mbar_wait(&op_empty[os], oph ^ 1u, abort_flag, p.err, code_base | 2);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          uint8_t* o = op + os * OP_STAGE + (a_warp ? 0 : OP_OPERAND);
#pragma unroll
          for (int i = 0; i < kUnitsPerThread; ++i) {
            const int u = htid + i * kHalfThreads;
            widen_unit(x[i], u >> 3, u & 7, o);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&signal[os]);
          if (++os == OP_STAGES) { os = 0; oph ^= 1u; }
          continue;
        }
        // widen as soon as the raw stage is in and release it; wait for the
        // operand slot (freed when the MMAs two stages back complete) only
        // before storing, so that the widening stays off the slot hand-off
        ok = mbar_wait(&raw_full[rs], rph, abort_flag, p.err, code_base | 2);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const uint8_t* r = raw + rs * RAW_STAGE + (a_warp ? 0 : RAW_OP);
        uint4 lo[kUnitsPerThread], hi[kUnitsPerThread];
#pragma unroll
        for (int i = 0; i < kUnitsPerThread; ++i) {
          const int u = htid + i * kHalfThreads;
          widen_load(r, u >> 3, u & 7, lo[i], hi[i]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rs]);
        ok = mbar_wait(&op_empty[os], oph ^ 1u, abort_flag, p.err, code_base | 2);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        uint8_t* o = op + os * OP_STAGE + (a_warp ? 0 : OP_OPERAND);
#pragma unroll
        for (int i = 0; i < kUnitsPerThread; ++i) {
          const int u = htid + i * kHalfThreads;
          widen_store(lo[i], hi[i], u >> 3, u & 7, o);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&signal[os]);
        if (++rs == RAW_STAGES) { rs = 0; rph ^= 1u; }
        if (++os == OP_STAGES) { os = 0; oph ^= 1u; }
      }
    }
  } else if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !kGlobal) {
      prefetch_tensormap(&map_a);
      prefetch_tensormap(&map_dy);
    }
    uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
    bool ok = true;
    for (int c = 0; ok && !kGlobal && c < units.nc; ++c)
    for (int tile = units.t0; ok && tile <= units.t1; ++tile) {
      if (!units.has(tile, c)) continue;
      const int tr = tile / p.tiles_c, tcol = tile % p.tiles_c;
      const int ax = tr * BMP + static_cast<int>(rank) * 128;    // k of this CTA's A rows
      const int bx = tcol * BN + static_cast<int>(rank) * BNH;   // n of this CTA's dY rows
      const int64_t k1 = min(p.num_stages, (c + 1) * kChunkStages);
      for (int64_t kb = c * kChunkStages; kb < k1; ++kb) {
        if (lane == 0)
          ok = mbar_wait(&raw_empty[stage], phase ^ 1u, abort_flag, p.err, code_base | 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* dst = raw + stage * RAW_STAGE;
          const int y = static_cast<int>(kb * BK);
          mbar_arrive_expect_tx(&raw_full[stage], RAW_STAGE);
          tma_load_2d(dst, &map_a, &raw_full[stage], ax, y);
          tma_load_2d(dst + RAW_OP, &map_dy, &raw_full[stage], bx, y);
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
      constexpr uint32_t idesc = idesc_f16_mn(BMP, BN);
      uint32_t os = 0, oph = 0, ab = 0, aph = 0;
      bool ok = true, issued_any = false;
      const uint64_t adesc0 = smem_desc_mn_sw128(smem_addr(op), MN_ATOM, K_GROUP);
      for (int c = 0; ok && c < units.nc; ++c)
      for (int tile = units.t0; ok && tile <= units.t1; ++tile) {
        if (!units.has(tile, c)) continue;
        {
          const int64_t c0 = c * kChunkStages;
          const int64_t c1 = min(p.num_stages, c0 + kChunkStages);
          ok = mbar_wait(&acc_empty[ab], aph ^ 1u, abort_flag, p.err, code_base | 3);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + ab * BN;
          // 32-bit stage count and descriptors from slot 0's: the issuer's own
          // work between its MMAs stays short
          const int n_st = static_cast<int>(c1 - c0);
          for (int st = 0; st < n_st; ++st) {
            ok = mbar_wait(&op_full[os], oph, abort_flag, p.err, code_base | 3);
            if (!ok) break;
            tc_fence_after();
            const uint64_t adesc = adesc0 + static_cast<uint64_t>((os * OP_STAGE) >> 4);
            const uint64_t bdesc = adesc + static_cast<uint64_t>(OP_OPERAND >> 4);
            // K-step j covers m rows [16j, 16j + 16): two 8-row groups further on
#pragma unroll
            for (int j = 0; j < BK / 16; ++j)
              umma_pair_ss(d_tmem, adesc + static_cast<uint64_t>((2 * j * K_GROUP) >> 4),
                           bdesc + static_cast<uint64_t>((2 * j * K_GROUP) >> 4), idesc,
                           (st > 0 || j > 0) ? 1u : 0u);
            issued_any = true;
            tc2::umma_commit_pair(&op_empty[os]);
            if (++os == OP_STAGES) { os = 0; oph ^= 1u; }
          }
          if (!ok) break;
          tc2::umma_commit_pair(&acc_full[ab]);
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
      // forward each stage's readiness to the even CTA's MMA issuer: one
      // signal-only cluster arrive per stage (the operands stay in this SM's
      // shared memory, fenced for the tensor core by the converters)
      const uint32_t op_full_leader0 = tc2::peer_addr(&op_full[0], 0);
      uint32_t os = 0, oph = 0;
      bool ok = true;
      for (int c = 0; ok && c < units.nc; ++c)
      for (int tile = units.t0; ok && tile <= units.t1; ++tile) {
        if (!units.has(tile, c)) continue;
        const int64_t k1 = min(p.num_stages, (c + 1) * kChunkStages);
        for (int64_t kb = c * kChunkStages; kb < k1; ++kb) {
          ok = mbar_wait(&op_ready[os], oph, abort_flag, p.err, code_base | 5);
          if (!ok) break;
          tc2::mbar_arrive_cluster_relaxed(op_full_leader0 + 8u * os);
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
    const uint32_t acc_empty_leader0 = tc2::peer_addr(&acc_empty[0], 0);
    uint32_t ab = 0, aph = 0, slab = 0;
    bool ok = true;
    if (epi_tid == 0 && p.use_tma_out) prefetch_tensormap(&map_out);
    // every unit adds onto the output: the zeroing grid must have completed
    grid_dependency_wait();
    for (int c = 0; ok && c < units.nc; ++c)
    for (int tile = units.t0; ok && tile <= units.t1; ++tile) {
      if (!units.has(tile, c)) continue;
      const int tr = tile / p.tiles_c, tcol = tile % p.tiles_c;
      const int row0 = tr * BMP + static_cast<int>(rank) * 128;
      {
        ok = mbar_wait(&acc_full[ab], aph, abort_flag, p.err, code_base | 4);
        ok = named_bar_and(kEpiBarrier, 128, __all_sync(0xffffffffu, ok));
        if (!ok) break;
        tc_fence_after();
        for (int cb = 0; cb < BN / 32; ++cb) {
          const int64_t col0 = static_cast<int64_t>(tcol) * BN + cb * 32;
          if (col0 >= p.N) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * BN + cb * 32,
                             v);
          tmem_wait_ld();
          if (!p.use_tma_out) {
            // rows of dW not 16-byte aligned: atomic adds row by row, through
            // this warp's part of the idle staging buffers
            uint32_t* scratch = reinterpret_cast<uint32_t*>(stage_out) + q * (33 * 32);
            tc::out_block32(scratch, v, lane, p.out, p.N, row0 + q * 32, p.K, col0, p.N,
                            tc::kOutAtomicAdd);
            continue;
          }
          uint8_t* buf = stage_out + (slab & 1) * STAGE_OUT;
          if (epi_tid == 0) bulk_wait_group_read<1>();
          named_bar_sync(kEpiBarrier, 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int4 val =
                make_int4(tc::f32_bits_to_i32(v[4 * c]), tc::f32_bits_to_i32(v[4 * c + 1]),
                          tc::f32_bits_to_i32(v[4 * c + 2]), tc::f32_bits_to_i32(v[4 * c + 3]));
            sts128(buf + tc::sw128(srow, c), val);
          }
          fence_proxy_async_smem();
          named_bar_sync(kEpiBarrier, 128);
          if (epi_tid == 0 && row0 < p.K) {  // a tile half wholly past K writes nothing
            tma_reduce_add_2d(&map_out, buf, static_cast<int>(col0), row0);
            bulk_commit_group();
          }
          ++slab;
        }
        tc_fence_before();
        __syncwarp();
        // the accumulator reads are complete (tcgen05.wait::ld): signal only
        if (lane == 0) tc2::mbar_arrive_cluster_relaxed(acc_empty_leader0 + 8u * ab);
        if (++ab == ACC_BUFS) { ab = 0; aph ^= 1u; }
      }
    }
    if (epi_tid == 0 && p.use_tma_out) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  tc2::cluster_sync();  // the peer's TMEM and barriers stay alive until both CTAs are done
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc2::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace dw2
}  // namespace t3
