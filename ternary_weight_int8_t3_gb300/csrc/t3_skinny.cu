// t3_skinny.cu -- the small-M forward (M <= 32): C = A . W at the rate of
// reading the packed weights.
//
// What it computes: the forward product of "t27c PTX backend: ternary x int8
// GEMM kernel emitted by a .t27 spec (int8 mma.sync), ptx-run glue", section
// "What this adds": C[m][n] = sum_k A[m][k] W[k][n], W from 2-bit codes.
//
// With M <= 32 there is little work per packed weight byte and the product is
// bound by streaming Wp (N * ceil(K/4) bytes) from HBM once.  The pages have no
// such path; this one is built for sm_103a:
//   * swap-AB on the tensor core with 8-bit floats: D[n][r] = W^T[n][k] . B[r][k]
//     with tcgen05.mma kind::f8f6f4 (e4m3 x e4m3 -> f32), K = 32 per
//     instruction, issued for a CTA pair (cta_group::2, M = 256 weight rows,
//     128 per SM): one pair instruction costs its issuing thread about as much
//     as a single-CTA one, so the pair halves the issue time per weight byte;
//   * several threads issue, each into its own accumulator, for equal parts
//     of every unit's reduction: an issuing thread waits about 55 cycles per
//     instruction whatever N is, while the tensor pipe needs N/2 cycles, so
//     at N <= 32 four issuers keep it busy and at N = 48 or 64 two do;
//   * every weight is exact in e4m3 (+1 = 0x38, -1 = 0xB8).  An activation
//     is split into two 4-bit digits, each stored as an e4m3 byte whose value
//     is exactly byte * 2^-9 (bytes 0..15 are the subnormals and the first
//     normal binade), so the conversion is bit arithmetic and every f32 sum is
//     an integer multiple of 2^-9 far inside 2^24 units.  For M < 32 the
//     digits are those of u = a + 128 (hi = u >> 4, lo = u & 15, both in
//     [0, 15]) and one extra B row of ones yields sum_k w, so that
//     C = 16 * D_hi + D_lo - 128 * D_ones.  For M = 32, where no spare row is
//     left, hi = a >> 4 in [-8, 7] is stored as sign | magnitude, lo = a & 15;
//   * the B operand has NB rows (NB = 2M + 1 rounded up to 16, or 64 for
//     M = 32): row 2m holds the hi digits of activation row m, row 2m+1 its lo
//     digits, row 2M the ones.  Each CTA of the pair holds NB/2 of them and
//     converts its activation rows per unit from a TMA-loaded raw slice that
//     travels with the unit's weights; rows without an activation row are set
//     once, before the first unit;
//   * the weights are decoded in registers straight into TMEM (the MMA's A
//     operand), one byte permute per four weights, in a permuted order within
//     each 16-code word (even codes, then odd codes) that the activations copy;
//   * units are 128 weight rows x 512 k per CTA, ordered (tile, k) and split
//     evenly over the pairs; each run of units of one tile ends with a TMA
//     reduce-add of its int32 partial into C.  A small kernel zeroes C first.
//     Both are launched as programmatic dependents: the zeroing kernel waits
//     (griddepcontrol.wait) for the preceding grid to complete and then lets
//     this kernel launch, whose prologue and weight stream overlap the
//     zeroing; it waits for the zeroing only before its first reduce-add.
#include <atomic>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {
namespace sk {

constexpr int TN = 128;          // weight rows per CTA (TMEM lanes)
constexpr int TP = 2 * TN;       // weight rows per pair tile (MMA M)
constexpr int UK = 512;          // reduction elements per unit
constexpr int UB = UK / 4;       // packed bytes per row per unit (128)
constexpr int RUN_MAX = 2048;    // units per accumulation run: f32 sums stay exact
constexpr int RAW_STAGES = 6;
constexpr int A_BUFS = 3;        // TMEM weight buffers and B buffers
constexpr int NB_MAX = 64;       // B rows (MMA N)
constexpr int HALF_MAX = NB_MAX / 4;  // activation rows each CTA converts
constexpr int TMEM_COLS = 512;
constexpr int kMaxIssuers = 4;
constexpr int ACC_REGION = 128;                  // kIss accumulators of 128 / kIss columns
constexpr int kACol = ACC_REGION;                // then three weight buffers of 128 columns
constexpr int kStepsPerUnit = UK / 32;           // MMA K-steps per unit
constexpr int kDecWarps = 16;  // four per lane quadrant, each a quarter of every unit
constexpr int kProducerWarp = kDecWarps;
constexpr int kMmaWarp0 = kDecWarps + 1;  // MMA issuers (even CTA)
constexpr int kEpiWarp0 = kMmaWarp0 + kMaxIssuers;
constexpr int kThreads = 32 * (kEpiWarp0 + 4);
constexpr int kEpiBarrier = 1;
constexpr int kDecBarrier = 2;

constexpr int RAW_W = TN * UB;                    // 16 KB of codes, 128-byte swizzle
constexpr int ACT_BOX = 256;                      // activation bytes per TMA box row
constexpr int ACT_BOX_BYTES = HALF_MAX * ACT_BOX;
constexpr int RAW_ACT = (UK / ACT_BOX) * ACT_BOX_BYTES;  // [box][row][256 B]
constexpr int RAW_STAGE = RAW_W + RAW_ACT;        // 24 KB
constexpr int kActIters = HALF_MAX * (UK / 16) / (kDecWarps * 32);  // chunks per thread
constexpr int B_ATOM = (NB_MAX / 2) * 128;   // one 128-k atom of up to NB/2 rows x 128 B
constexpr int B_BUF = (UK / 128) * B_ATOM;   // 16 KB
constexpr int STAGE_OUT = (NB_MAX / 2) * TN * 4;         // [NB/2 rows m][128 int32]
constexpr int OFF_RAW = 0;
constexpr int OFF_B = OFF_RAW + RAW_STAGES * RAW_STAGE;
constexpr int OFF_OUT = OFF_B + A_BUFS * B_BUF;
constexpr int OFF_BAR = OFF_OUT + 2 * STAGE_OUT;
constexpr int N_BARS = 2 * RAW_STAGES + 2 * A_BUFS + 2 + kMaxIssuers;
constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
static_assert(RAW_STAGE % 1024 == 0, "swizzled TMA destinations need 1024-byte alignment");
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
static_assert(kACol + A_BUFS * (UK / 4) <= TMEM_COLS, "TMEM budget");
static_assert(kStepsPerUnit % (4 * kMaxIssuers) == 0, "issuers split every unit in whole atoms");

struct Params {
  const int8_t* A;     // [M][K]
  const uint8_t* Wp;   // [N][ceil(K/4)]
  int32_t* C;          // [M][N], zeroed by the preceding kernel
  int M, N, K;
  int NB;              // B rows = MMA N; NB/4 activation rows per CTA, NB/2 output rows m
  int ones_row;        // B row of ones (unsigned digits), or -1 (signed digits)
  int units_total, units_k;  // units in (tile, k) order; units along k per tile
  int use_tma_w, use_tma_out, use_tma_act;
  int* err;
};

// Walks units in (tile, k-unit) order.
struct UnitIter {
  int t, uk, units_k;
  __device__ void init(const Params& p, int u) {
    units_k = p.units_k;
    t = u / units_k;
    uk = u - t * units_k;
  }
  __device__ void next() {
    if (++uk == units_k) {
      uk = 0;
      ++t;
    }
  }
};

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

// e4m3 weight of code c = byte c of this word: 0 -> 0x00, 1 -> 0x38 (+1.0),
// 2 -> 0xB8 (-1.0), 3 -> 0x00.
constexpr uint32_t kE4m3Table = 0x00B83800u;

// 16 codes (one word, code i at bits 2i) -> 4 words of e4m3 weights in the
// permuted reduction order 0,2,4,6 | 8,10,12,14 | 1,3,5,7 | 9,11,13,15.
__device__ __forceinline__ void decode16_e4m3(uint32_t x, uint32_t* o) {
  const uint32_t ev = x & 0x33333333u;         // nibble t = code 2t
  const uint32_t od = (x >> 2) & 0x33333333u;  // nibble t = code 2t+1
  o[0] = prmt(kE4m3Table, 0u, ev);
  o[1] = prmt(kE4m3Table, 0u, ev >> 16);
  o[2] = prmt(kE4m3Table, 0u, od);
  o[3] = prmt(kE4m3Table, 0u, od >> 16);
}

// D (both CTAs' TMEM) (+)= A (both CTAs' TMEM, e4m3) x B (both CTAs' shared
// memory halves, e4m3), f32 accumulation.
__device__ __forceinline__ void umma_f8_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor: e4m3 x e4m3 -> f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// Four int8 (a word) -> the e4m3 bytes of their two digits, in the same byte
// order.  Unsigned: u = a + 128, hi = u >> 4, lo = u & 15.  Signed:
// hi = a >> 4 stored as sign | magnitude, lo = a & 15.
template <bool kSigned>
__device__ __forceinline__ void s8x4_to_digits(uint32_t y, uint32_t& hi, uint32_t& lo) {
  if (kSigned) {
    lo = y & 0x0F0F0F0Fu;
    const uint32_t h4 = (y >> 4) & 0x0F0F0F0Fu;       // hi as a 4-bit two's complement
    const uint32_t neg = (y >> 7) & 0x01010101u;      // 1 where hi < 0
    const uint32_t mag = (h4 ^ (neg * 0x0Fu)) + neg;  // |hi| = 16 - h4 where negative
    hi = mag | (neg << 7);
  } else {
    const uint32_t u = y ^ 0x80808080u;
    hi = (u >> 4) & 0x0F0F0F0Fu;
    lo = u & 0x0F0F0F0Fu;
  }
}

// 16 activations -> the hi and lo digit words of one 16-element group, in the
// decode's permuted order (even bytes, then odd bytes).
template <bool kSigned>
__device__ __forceinline__ void act16_to_digits(const uint4 x, uint4& hi, uint4& lo) {
  s8x4_to_digits<kSigned>(prmt(x.x, x.y, 0x6420u), hi.x, lo.x);
  s8x4_to_digits<kSigned>(prmt(x.z, x.w, 0x6420u), hi.y, lo.y);
  s8x4_to_digits<kSigned>(prmt(x.x, x.y, 0x7531u), hi.z, lo.z);
  s8x4_to_digits<kSigned>(prmt(x.z, x.w, 0x7531u), hi.w, lo.w);
}

// Cluster barrier in two halves: arrive (no ordering of earlier memory
// accesses) and wait.  Every thread arrives once and waits once per phase.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

template <bool kSigned, int kIss>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    skinny_fwd_kernel(const Params p, const __grid_constant__ CUtensorMap map_w,
                      const __grid_constant__ CUtensorMap map_out,
                      const __grid_constant__ CUtensorMap map_act) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((base_addr + 1023u) & ~1023u) - base_addr);
  uint8_t* raw = smem + OFF_RAW;
  uint8_t* bop = smem + OFF_B;
  uint8_t* stage_out = smem + OFF_OUT;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* raw_full = bars;                    // TMA bytes landed
  uint64_t* raw_empty = raw_full + RAW_STAGES;  // decoders done with the stage
  uint64_t* a_full = raw_empty + RAW_STAGES;    // even CTA: both CTAs' operands ready
  uint64_t* a_empty = a_full + A_BUFS;          // both: MMAs of the buffer done (multicast)
  uint64_t* acc_full = a_empty + A_BUFS;        // both: run complete (multicast)
  uint64_t* acc_empty = acc_full + 1;           // even CTA: both epilogues drained
  uint64_t* drain_bar = acc_empty + 1;          // one per issuer, error path only
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  constexpr int kAccStride = ACC_REGION / kIss;  // columns per accumulator (>= NB)
  constexpr int kStepsPerIssuer = kStepsPerUnit / kIss;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc2::cluster_rank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int u0 = static_cast<int>(static_cast<int64_t>(p.units_total) * pair / npairs);
  const int u1 = static_cast<int>(static_cast<int64_t>(p.units_total) * (pair + 1) / npairs);
  const int n_units = u1 - u0;
  const int half_rows = p.NB >> 2;  // activation row slots of this CTA
  const int m_lo = static_cast<int>(rank) * half_rows;
  const int real_rows = max(0, min(p.M - m_lo, half_rows));  // activation rows present
  constexpr int code_base = 4 << 8;
  launch_dependents();  // a dependent grid still waits for this one before touching its data

  if (warp == kProducerWarp && lane == 0) {
    if (p.use_tma_w) prefetch_tensormap(&map_w);
    if (p.use_tma_act) prefetch_tensormap(&map_act);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW_STAGES; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kDecWarps);
    }
    for (int s = 0; s < A_BUFS; ++s) {
      mbar_init(&a_full[s], 2 * kDecWarps);  // the decoders of both CTAs
      mbar_init(&a_empty[s], kIss);
    }
    mbar_init(acc_full, kIss);
    mbar_init(acc_empty, 8);  // 4 epilogue warps x 2 CTAs
    for (int j = 0; j < kMaxIssuers; ++j) mbar_init(&drain_bar[j], 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp0) {
    tc2::tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tc2::tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // Both CTAs' barriers and TMEM must exist before any remote arrive or pair
  // MMA: every role waits on this cluster phase before its first such step;
  // the producer, whose barriers are local, starts loading at once.
  cluster_arrive_relaxed();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp < kDecWarps) {
    // ------------------------------- weight decode -> TMEM, activations -> B
    const int q = warp & 3, h = warp >> 2;  // lane quadrant, quarter of the unit
    const int gtid = threadIdx.x;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    // the even CTA's decoders arrive locally; the odd CTA's arrive on the even
    // CTA's barrier.  A signal-only arrive: the operands it announces stay in
    // this SM's TMEM and shared memory, already completed (tcgen05.wait::st)
    // and fenced for the tensor core (fence.proxy.async).
    const uint32_t a_full_leader0 = tc2::peer_addr(&a_full[0], 0);
    // B rows that no activation row of this CTA rewrites: zero digits, and
    // the row of ones where it falls in this CTA
    const int dtid = threadIdx.x;  // 0 .. 32 * kDecWarps - 1
    for (int idx = dtid; idx < A_BUFS * B_BUF / 16; idx += 32 * kDecWarps)
      reinterpret_cast<uint4*>(bop)[idx] = make_uint4(0u, 0u, 0u, 0u);
    named_bar_sync(kDecBarrier, 32 * kDecWarps);
    const int local_ones = p.ones_row - static_cast<int>(rank) * (p.NB >> 1);
    if (local_ones >= 0 && local_ones < (p.NB >> 1)) {
      for (int idx = dtid; idx < A_BUFS * (UK / 16); idx += 32 * kDecWarps) {
        const int b = idx / (UK / 16), c = idx % (UK / 16);
        *reinterpret_cast<uint4*>(bop + b * B_BUF + (c >> 3) * B_ATOM +
                                  tc::sw128(local_ones, c & 7)) =
            make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(kDecBarrier, 32 * kDecWarps);
    cluster_wait();
    UnitIter it;
    it.init(p, u0);
    for (int i = 0; i < n_units; ++i, it.next()) {
      const int rs = i % RAW_STAGES, ab = i % A_BUFS;  // compile-time divisors
      const uint32_t rph = (i / RAW_STAGES) & 1, aph = (i / A_BUFS) & 1;
      bool ok = mbar_wait(&raw_full[rs], rph, abort_flag, p.err, code_base | 2) &&
                mbar_wait(&a_empty[ab], aph ^ 1u, abort_flag, p.err, code_base | 2);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint8_t* stage = raw + rs * RAW_STAGE;
      // This CTA's activation rows of the unit, loaded first so that their
      // latency passes under the weight decode: chunk ci is 16 elements c of
      // row ml (activation row m_lo + ml).
      const int chunks = real_rows * (UK / 16);
      uint4 xa[kActIters];
#pragma unroll
      for (int r = 0; r < kActIters; ++r) {
        const int ci = gtid + r * kDecWarps * 32;
        const int ml = ci / (UK / 16), c = ci % (UK / 16);
        xa[r] = make_uint4(0u, 0u, 0u, 0u);
        if (ci >= chunks) continue;
        if (p.use_tma_act) {
          xa[r] = *reinterpret_cast<const uint4*>(stage + RAW_W + (c >> 4) * ACT_BOX_BYTES +
                                                  ml * ACT_BOX + ((c & 15) << 4));
        } else {
          const int64_t m = m_lo + ml;
          const int64_t k0 = static_cast<int64_t>(it.uk) * UK + 16 * c;
          const int8_t* a = p.A + m * p.K + k0;
          uint32_t w[4] = {0u, 0u, 0u, 0u};
          for (int j = 0; j < 16; ++j)
            if (k0 + j < p.K)
              w[j >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(__ldg(a + j))) << (8 * (j & 3));
          xa[r] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      // 32 bytes = 128 codes of this row's quarter of the unit: 16-byte
      // chunks 2h, 2h+1 of the row, in the 128-byte swizzle when TMA loaded them
      const uint8_t* src = stage + row * UB;
      const int swz = p.use_tma_w ? (row & 7) : 0;
      const uint32_t col0 = kACol + ab * (UK / 4) + 32 * h;
      {
        const int c0 = 2 * h;
        const uint4 x0 = *reinterpret_cast<const uint4*>(src + ((c0 ^ swz) << 4));
        const uint4 x1 = *reinterpret_cast<const uint4*>(src + (((c0 + 1) ^ swz) << 4));
        uint32_t v[32];
        decode16_e4m3(x0.x, v);
        decode16_e4m3(x0.y, v + 4);
        decode16_e4m3(x0.z, v + 8);
        decode16_e4m3(x0.w, v + 12);
        decode16_e4m3(x1.x, v + 16);
        decode16_e4m3(x1.y, v + 20);
        decode16_e4m3(x1.z, v + 24);
        decode16_e4m3(x1.w, v + 28);
        tc2::tmem_st_32x32b_x32(lane_addr + col0, v);
      }
      // activations -> this CTA's half of the B operand: row 2 ml = hi
      // digits, row 2 ml + 1 = lo digits, atoms of 128 k in the 128-byte swizzle
      uint8_t* bbuf = bop + ab * B_BUF;
#pragma unroll
      for (int r = 0; r < kActIters; ++r) {
        const int ci = gtid + r * kDecWarps * 32;
        if (ci >= chunks) continue;
        const int ml = ci / (UK / 16), c = ci % (UK / 16);
        uint4 hi, lo;
        act16_to_digits<kSigned>(xa[r], hi, lo);
        uint8_t* atom = bbuf + (c >> 3) * B_ATOM;
        sts128(atom + tc::sw128(2 * ml, c & 7), hi);
        sts128(atom + tc::sw128(2 * ml + 1, c & 7), lo);
      }
      fence_proxy_async_smem();
      tc2::tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&raw_empty[rs]);
        if (rank == 0)
          mbar_arrive(&a_full[ab]);
        else
          tc2::mbar_arrive_cluster_relaxed(a_full_leader0 + 8u * ab);
      }
    }
  } else if (warp == kProducerWarp) {
    // ------------------------------------- packed weights and activations in
    uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
    bool ok = true;
    const int64_t kbytes = (static_cast<int64_t>(p.K) + 3) / 4;
    const uint32_t tx = (p.use_tma_w ? RAW_W : 0) +
                        (p.use_tma_act ? (UK / ACT_BOX) * half_rows * ACT_BOX : 0);
    UnitIter it;
    it.init(p, u0);
    for (int i = 0; i < n_units; ++i, it.next()) {
      if (lane == 0)
        ok = mbar_wait(&raw_empty[stage], phase ^ 1u, abort_flag, p.err, code_base | 1);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      uint8_t* dst = raw + stage * RAW_STAGE;
      const int wx = it.uk * UB, wy = it.t * TP + static_cast<int>(rank) * TN;
      if (!p.use_tma_w) {
        tc::manual_box(dst, p.Wp, kbytes, p.N, kbytes, wy, wx, TN, UB, lane);
        __threadfence_block();
        __syncwarp();
      }
      if (lane == 0) {
        if (tx > 0) {
          mbar_arrive_expect_tx(&raw_full[stage], tx);
          if (p.use_tma_w) tma_load_2d(dst, &map_w, &raw_full[stage], wx, wy);
          if (p.use_tma_act)
            for (int b = 0; b < UK / ACT_BOX; ++b)
              tma_load_2d(dst + RAW_W + b * ACT_BOX_BYTES, &map_act, &raw_full[stage],
                          it.uk * UK + b * ACT_BOX, m_lo);
        } else {
          mbar_arrive(&raw_full[stage]);
        }
      }
      issued_mask |= 1u << stage;
      issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
      if (++stage == RAW_STAGES) { stage = 0; phase ^= 1u; }
    }
    cluster_wait();
    if (!ok && lane == 0) {
      for (int s = 0; s < RAW_STAGES; ++s) {
        if (!(issued_mask & (1u << s))) continue;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&raw_full[s], (issued_phase >> s) & 1u) &&
               global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp < kEpiWarp0) {
    const int j = warp - kMmaWarp0;  // issuer j: K-steps [j S, j S + S) of every unit
    cluster_wait();
    if (rank == 0 && lane == 0 && j < kIss) {
      // ------------------------------------------------------ MMA issuers
      const uint32_t idesc = idesc_e4m3_f32(TP, p.NB);
      uint32_t acc_ph = 0;
      bool ok = true, issued_any = false, seg_first = true;
      int run_len = 0;
      UnitIter it;
      it.init(p, u0);
      for (int i = 0; i < n_units; ++i, it.next()) {
        const int ab = i % A_BUFS;
        const uint32_t aph = (i / A_BUFS) & 1;
        ++run_len;
        const bool seg_last =
            (i + 1 == n_units) || (it.uk + 1 == it.units_k) || (run_len == RUN_MAX);
        if (seg_first) ok = mbar_wait(acc_empty, acc_ph ^ 1u, abort_flag, p.err, code_base | 3);
        if (ok) ok = mbar_wait(&a_full[ab], aph, abort_flag, p.err, code_base | 3);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + j * kAccStride;
        // K-step k reads A columns [8k, 8k + 8) and B atom k/4 at byte 32 (k%4);
        // only the descriptor's start-address field changes, by (offset >> 4)
        const uint32_t a_tmem =
            tmem_base + kACol + ab * (UK / 4) + 8 * kStepsPerIssuer * j;
        const uint64_t bdesc0 = smem_desc_k_sw128(
            smem_addr(bop + ab * B_BUF + (kStepsPerIssuer / 4) * j * B_ATOM));
#pragma unroll
        for (int s = 0; s < kStepsPerIssuer; ++s)
          umma_f8_pair_ts(d_tmem, a_tmem + 8 * s,
                          bdesc0 + static_cast<uint64_t>(((s >> 2) * B_ATOM + 32 * (s & 3)) >> 4),
                          idesc, (seg_first && s == 0) ? 0u : 1u);
        issued_any = true;
        tc2::umma_commit_pair(&a_empty[ab]);
        seg_first = seg_last;
        if (seg_last) {
          tc2::umma_commit_pair(acc_full);
          run_len = 0;
          acc_ph ^= 1u;
        }
      }
      // the odd CTA's last remote arrive has landed before this CTA may exit
      if (ok && j == 0) mbar_wait(acc_empty, acc_ph ^ 1u, abort_flag, p.err, code_base | 3);
      if (!ok && issued_any) {
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&drain_bar[j]))
            : "memory");
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&drain_bar[j], 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int etid = threadIdx.x - kEpiWarp0 * 32;
    const int nloc = q * 32 + lane;
    const uint32_t acc_empty_leader0 = tc2::peer_addr(acc_empty, 0);
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t acc_ph = 0, slab = 0;
    if (p.use_tma_out && etid == 0) prefetch_tensormap(&map_out);
    cluster_wait();
    grid_dependency_wait();  // C has been zeroed (long before the first run ends)
    UnitIter it;
    it.init(p, u0);
    int i = 0;
    while (i < n_units) {
      // the run of units of one tile that starts at unit i
      const int t = it.t;
      int len = 1;
      while (i + len < n_units && it.uk + 1 < it.units_k && len < RUN_MAX) {
        it.next();
        ++len;
      }
      bool ok = mbar_wait(acc_full, acc_ph, abort_flag, p.err, code_base | 4);
      ok = named_bar_and(kEpiBarrier, 128, __all_sync(0xffffffffu, ok));
      if (!ok) break;
      tc_fence_after();
      const int n0 = t * TP + static_cast<int>(rank) * TN;
      const int64_t n = static_cast<int64_t>(n0) + nloc;
      uint8_t* buf = stage_out + (slab & 1) * STAGE_OUT;
      int32_t* sb = reinterpret_cast<int32_t*>(buf);
      // Summed over the issuers' accumulators, in units of 2^-9 (scaling by
      // 512 is exact): column 2m holds the hi digits' sum of row m, column
      // 2m + 1 the lo digits' sum, column ones_row the sum of the weights.
      int32_t bias = 0;  // 128 * sum_k w for unsigned digits
      uint32_t o[kIss];
      if (!kSigned) {
#pragma unroll
        for (int a = 0; a < kIss; ++a)
          asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                       : "=r"(o[a]) : "r"(lane_base + a * kAccStride + p.ones_row));
      }
      // BW columns (BW/2 rows m) of every accumulator per TMEM round trip
      constexpr int BW = 64 / kIss;
      for (int cb = 0; cb < p.NB; cb += BW) {
        uint32_t d[kIss][BW];
        const bool full = cb + BW <= p.NB;
#pragma unroll
        for (int a = 0; a < kIss; ++a) {
          if constexpr (BW == 32) {
            if (full)
              tmem_ld_32x32b_x32(lane_base + a * kAccStride + cb, d[a]);
            else
              tmem_ld_32x32b_x16(lane_base + a * kAccStride + cb,
                                 *reinterpret_cast<uint32_t(*)[16]>(d[a]));
          } else {
            tmem_ld_32x32b_x16(lane_base + a * kAccStride + cb, d[a]);
          }
        }
        tmem_wait_ld();
        if (cb == 0 && p.use_tma_out) {
          // the staging buffer's previous bulk add has read it
          if (etid == 0) bulk_wait_group_read<1>();
          named_bar_sync(kEpiBarrier, 128);
        }
        if (!kSigned && cb == 0) {
          int32_t ones = 0;
#pragma unroll
          for (int a = 0; a < kIss; ++a) ones += __float2int_rn(__uint_as_float(o[a]) * 512.0f);
          bias = 128 * ones;
        }
#pragma unroll
        for (int e = 0; e < BW / 2; ++e) {
          if (!full && e >= 8) break;
          const int m = (cb >> 1) + e;
          int32_t hi = 0, lo = 0;
#pragma unroll
          for (int a = 0; a < kIss; ++a) {
            hi += __float2int_rn(__uint_as_float(d[a][2 * e]) * 512.0f);
            lo += __float2int_rn(__uint_as_float(d[a][2 * e + 1]) * 512.0f);
          }
          const int32_t v = 16 * hi + lo - bias;
          if (p.use_tma_out) {
            sb[m * TN + nloc] = v;
          } else if (n < p.N && m < p.M) {
            atomicAdd(p.C + static_cast<int64_t>(m) * p.N + n, v);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      // the accumulator reads are complete (tcgen05.wait::ld): signal only
      if (lane == 0) tc2::mbar_arrive_cluster_relaxed(acc_empty_leader0);
      acc_ph ^= 1u;
      if (p.use_tma_out) {
        fence_proxy_async_smem();
        named_bar_sync(kEpiBarrier, 128);
        if (etid == 0 && n0 < p.N) {  // a tile half wholly past N adds nothing
          tma_reduce_add_2d(&map_out, buf, n0, 0);
          bulk_commit_group();
        }
        ++slab;
      }
      i += len;
      if (i < n_units) it.next();
    }
    if (p.use_tma_out && etid == 0) bulk_wait_group_read<0>();  // the stores finish by themselves
  }

  tc_fence_before();
  __syncthreads();
  // No cross-CTA operation is in flight any more (the even CTA has seen the
  // odd CTA's last arrive, the odd CTA the last commit); the barrier keeps
  // the pair's TMEM allocated until both CTAs are done with it.
  cluster_arrive_relaxed();
  cluster_wait();
  tc_fence_after();
  if (warp == kMmaWarp0) {
    __syncwarp();
    tc2::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// Zeroes C ([n] int32).  Launched as a programmatic dependent of whatever
// precedes it, so that its launch overlaps that grid's tail: it waits for that
// grid to complete before anything else, then lets the product kernel launch.
__global__ void __launch_bounds__(256) zero_kernel_pdl(int32_t* C, int64_t n) {
  grid_dependency_wait();
  launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (reinterpret_cast<uintptr_t>(C) % 16 == 0) {
    const int64_t n4 = n / 4;
    int4* c4 = reinterpret_cast<int4*>(C);
    for (int64_t i = tid; i < n4; i += stride) c4[i] = make_int4(0, 0, 0, 0);
    for (int64_t i = 4 * n4 + tid; i < n; i += stride) C[i] = 0;
  } else {
    for (int64_t i = tid; i < n; i += stride) C[i] = 0;
  }
}

}  // namespace sk

int launch_zero_pdl(int32_t* out, int64_t n, int sms, cudaStream_t s) {
  int64_t zgrid = (n / 4 + 255) / 256;
  if (zgrid < 1) zgrid = 1;
  if (zgrid > 2 * sms) zgrid = 2 * sms;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t zcfg = {};
  zcfg.gridDim = dim3(static_cast<unsigned>(zgrid), 1, 1);
  zcfg.blockDim = dim3(256, 1, 1);
  zcfg.stream = s;
  zcfg.attrs = attr;
  zcfg.numAttrs = 1;
  return cudaLaunchKernelEx(&zcfg, sk::zero_kernel_pdl, out, n) == cudaSuccess ? T3_OK
                                                                                : T3_ECUDA;
}

int launch_skinny_fwd(const int8_t* A, const uint8_t* Wp, int32_t* C, int64_t M, int64_t N,
                      int64_t K, int sms, int* err, cudaStream_t s) {
  sk::Params p{};
  p.A = A;
  p.Wp = Wp;
  p.C = C;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  const bool signed_digits = (M == 32);  // no spare B row for the ones
  p.NB = signed_digits ? 64 : static_cast<int>((2 * M + 1 + 15) / 16 * 16);
  p.ones_row = signed_digits ? -1 : static_cast<int>(2 * M);
  p.units_k = static_cast<int>((K + sk::UK - 1) / sk::UK);
  const int64_t tiles = (N + sk::TP - 1) / sk::TP;
  const int64_t units = static_cast<int64_t>(p.units_k) * tiles;
  if (units > 2147483647LL) return T3_EINVAL;
  p.units_total = static_cast<int>(units);
  p.err = err;
  const int64_t kbytes = (K + 3) / 4;
  CUtensorMap mw, mo, ma;
  p.use_tma_w = make_u8_map_tiled(&mw, Wp, N, kbytes, kbytes, sk::TN, sk::UB, true) ? 1 : 0;
  p.use_tma_act = make_u8_map_tiled(&ma, A, M, K, K, p.NB / 4, sk::ACT_BOX) ? 1 : 0;
  p.use_tma_out = make_i32_map_tiled(&mo, C, M, N, p.NB / 2, sk::TN, false) ? 1 : 0;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return T3_ECUDA;
  static std::atomic<bool> attr_done[64];
  if (dev < 0 || dev >= 64) return T3_EDEVICE;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(sk::skinny_fwd_kernel<false, 4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             sk::SMEM_ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(sk::skinny_fwd_kernel<false, 2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             sk::SMEM_ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(sk::skinny_fwd_kernel<true, 2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             sk::SMEM_ALLOC) != cudaSuccess)
      return T3_ECUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }

  const int zst = launch_zero_pdl(C, M * N, sms, s);
  if (zst != T3_OK) return zst;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;

  const int64_t max_pairs = sms / 2 > 0 ? sms / 2 : 1;
  const int npairs = static_cast<int>(units < max_pairs ? units : max_pairs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * npairs, 1, 1);
  cfg.blockDim = dim3(sk::kThreads, 1, 1);
  cfg.dynamicSmemBytes = sk::SMEM_ALLOC;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // four issuers while each accumulator fits in 32 columns, else two
  const cudaError_t le =
      signed_digits ? cudaLaunchKernelEx(&cfg, sk::skinny_fwd_kernel<true, 2>, p, mw, mo, ma)
      : p.NB <= 32  ? cudaLaunchKernelEx(&cfg, sk::skinny_fwd_kernel<false, 4>, p, mw, mo, ma)
                    : cudaLaunchKernelEx(&cfg, sk::skinny_fwd_kernel<false, 2>, p, mw, mo, ma);
  if (le != cudaSuccess) return T3_ECUDA;
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
