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
//     each 16-code word (even codes, then odd codes) that the activations copy.
// Schedule: a unit is 128 weight rows x 512 k per CTA.  A cluster of S CTA
// pairs (S = 1 or 2, cluster of 2S CTAs) owns one 256-row tile at a time and
// splits its reduction into S contiguous k-slices, one per pair; clusters take
// tiles cluster, cluster + clusters, ...  Each pair sums its slice in TMEM
// (runs of at most RUN_MAX units, added in int32 in shared memory), then the pairs
// other than the first send their int32 partials into the first pair's shared
// memory (st.async, counted on an mbarrier there), and the first pair adds
// them and stores the tile.  Nothing is added into C in global memory, so C
// needs no zeroing, no kernel runs before this one, and the result does not
// depend on C's old contents.
// Launch: the kernel is a programmatic dependent of whatever precedes it on
// the stream and lets its own dependents launch at once, so a CTA that finds
// an SM free sets up its barriers and TMEM before the preceding grid has
// completed; it reads its inputs and writes C only after griddepcontrol.wait
// (the preceding grid complete and its writes visible).
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
constexpr int kMaxSplit = 2;     // pairs per cluster (cluster of 4 CTAs)
constexpr int ACC_REGION = 128;                  // kIss accumulators of 128 / kIss columns
constexpr int kACol = ACC_REGION;                // then three weight buffers of 128 columns
constexpr int kStepsPerUnit = UK / 32;           // MMA K-steps per unit
// Decoders: two groups of 8 warps take alternate units, so that one group's
// per-unit waits and hand-offs overlap the other group's decode; in a group,
// two warps per TMEM lane quadrant each decode half of every row.
constexpr int kDecWarps = 16;
constexpr int kGroupWarps = kDecWarps / 2;
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
constexpr int kActIters = HALF_MAX * (UK / 16) / (kGroupWarps * 32);  // chunks per thread
constexpr int B_ATOM = (NB_MAX / 2) * 128;   // one 128-k atom of up to NB/2 rows x 128 B
constexpr int B_BUF = (UK / 128) * B_ATOM;   // 16 KB
constexpr int STAGE_OUT = (NB_MAX / 2) * TN * 4;         // [NB/2 rows m][128 int32]
// A partial of one CTA of a non-first pair: [up to 8 quads of m][128 n][4 m]
// int32, so that the 16-byte accesses of consecutive n are consecutive.
constexpr int SLOT_QUAD = TN * 16;
constexpr int SLOT_BYTES = (NB_MAX / 8) * SLOT_QUAD;
constexpr int OFF_RAW = 0;
constexpr int OFF_B = OFF_RAW + RAW_STAGES * RAW_STAGE;
constexpr int OFF_OUT = OFF_B + A_BUFS * B_BUF;
constexpr int OFF_SLOT = OFF_OUT + STAGE_OUT;
constexpr int OFF_BAR = OFF_SLOT + (kMaxSplit - 1) * SLOT_BYTES;
constexpr int N_BARS = 2 * RAW_STAGES + 2 * A_BUFS + 2 + kMaxIssuers + 2;
constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
static_assert(RAW_STAGE % 1024 == 0, "swizzled TMA destinations need 1024-byte alignment");
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
static_assert(kACol + A_BUFS * (UK / 4) <= TMEM_COLS, "TMEM budget");
static_assert(kStepsPerUnit % (4 * kMaxIssuers) == 0, "issuers split every unit in whole atoms");

struct Params {
  const int8_t* A;     // [M][K]
  const uint8_t* Wp;   // [N][ceil(K/4)]
  int32_t* C;          // [M][N], overwritten
  int M, N, K;
  int NB;              // B rows = MMA N; NB/4 activation rows per CTA, NB/2 output rows m
  int m4;              // output rows m sent between pairs: M rounded up to 4
  int ones_row;        // B row of ones (unsigned digits), or -1 (signed digits)
  int tiles;           // pair tiles of 256 weight rows
  int units_k;         // units along k per tile
  int split;           // S: pairs per cluster, each a k-slice of upp units
  int upp;             // units per pair slice: ceil(units_k / S)
  int use_tma_w, use_tma_out, use_tma_act;
  int* err;
};

// Walks this pair's units: the tiles cid, cid + ncl, ... of its cluster, and
// within each its k-slice [uk0, uk1).
struct UnitIter {
  int t, uk, uk0, uk1, ncl;
  __device__ void init(int cid, int ncl_, int uk0_, int uk1_) {
    t = cid;
    ncl = ncl_;
    uk0 = uk0_;
    uk1 = uk1_;
    uk = uk0;
  }
  __device__ bool tile_last() const { return uk + 1 == uk1; }
  __device__ void next() {
    if (++uk == uk1) {
      uk = uk0;
      t += ncl;
    }
  }
};

__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                 "=r"(v[6]), "=r"(v[7])
               : "r"(taddr));
}

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

// Arrives on `bar` in both CTAs of the pair whose even CTA has cluster rank
// `lead` once all prior MMAs of this thread are complete.
__device__ __forceinline__ void umma_commit_to_pair(uint64_t* bar, uint32_t lead) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(static_cast<uint16_t>(0x3u << lead))
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
__global__ void __launch_bounds__(kThreads, 1)
    skinny_fwd_kernel(const Params p, const __grid_constant__ CUtensorMap map_w,
                      const __grid_constant__ CUtensorMap map_out,
                      const __grid_constant__ CUtensorMap map_act) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((base_addr + 1023u) & ~1023u) - base_addr);
  uint8_t* raw = smem + OFF_RAW;
  uint8_t* bop = smem + OFF_B;
  uint8_t* stage_out = smem + OFF_OUT;
  uint8_t* slots = smem + OFF_SLOT;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* raw_full = bars;                    // TMA bytes landed
  uint64_t* raw_empty = raw_full + RAW_STAGES;  // decoders done with the stage
  uint64_t* a_full = raw_empty + RAW_STAGES;    // even CTA: both CTAs' operands ready
  uint64_t* a_empty = a_full + A_BUFS;          // both: MMAs of the buffer done (multicast)
  uint64_t* acc_full = a_empty + A_BUFS;        // both: run complete (multicast)
  uint64_t* acc_empty = acc_full + 1;           // even CTA: both epilogues drained
  uint64_t* drain_bar = acc_empty + 1;          // one per issuer, error path only
  uint64_t* part_full = drain_bar + kMaxIssuers;  // first pair: the other pairs' partials in
  uint64_t* slot_free = part_full + 1;          // other pairs: the first pair read the partials
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  constexpr int kAccStride = ACC_REGION / kIss;  // columns per accumulator (>= NB)
  constexpr int kStepsPerIssuer = kStepsPerUnit / kIss;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = tc2::cluster_rank();     // 0 .. 2S - 1
  const uint32_t rank = crank & 1u;               // CTA within the pair
  const uint32_t lead = crank & ~1u;              // the pair's even CTA
  const int qp = static_cast<int>(crank >> 1);    // pair within the cluster = k-slice
  const int csize = 2 * p.split;
  const int cid = blockIdx.x / csize, ncl = gridDim.x / csize;
  const int uk0 = qp * p.upp;
  const int uk1 = min(p.units_k, uk0 + p.upp);
  const int my_tiles = cid < p.tiles ? (p.tiles - 1 - cid) / ncl + 1 : 0;
  const int n_units = my_tiles * (uk1 - uk0);
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
      mbar_init(&raw_empty[s], kGroupWarps);
    }
    for (int s = 0; s < A_BUFS; ++s) {
      mbar_init(&a_full[s], 2 * kGroupWarps);  // one decoder group of each CTA
      mbar_init(&a_empty[s], kIss);
    }
    mbar_init(acc_full, kIss);
    mbar_init(acc_empty, 8);  // 4 epilogue warps x 2 CTAs
    for (int j = 0; j < kMaxIssuers; ++j) mbar_init(&drain_bar[j], 1);
    mbar_init(part_full, 1);  // the first pair's arm (expect_tx) + the partials' bytes
    mbar_init(slot_free, 1);  // one arrive of the first pair's CTA of the same rank
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp0) {
    tc2::tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tc2::tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // Every CTA's barriers and TMEM must exist before any remote arrive, pair
  // MMA or st.async: every role waits on this cluster phase before its first
  // such step; the producer, whose barriers are local, starts loading at once.
  cluster_arrive_relaxed();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp < kDecWarps) {
    // ------------------------------- weight decode -> TMEM, activations -> B
    const int grp = warp / kGroupWarps;          // units grp, grp + 2, ...
    const int q = warp & 3, h = (warp >> 2) & 1;  // lane quadrant, half of every row
    const int gtid = threadIdx.x - grp * kGroupWarps * 32;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    // the even CTA's decoders arrive locally; the odd CTA's arrive on the even
    // CTA's barrier.  A signal-only arrive: the operands it announces stay in
    // this SM's TMEM and shared memory, already completed (tcgen05.wait::st)
    // and fenced for the tensor core (fence.proxy.async).
    const uint32_t a_full_lead0 = tc2::peer_addr(&a_full[0], lead);
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
    if (!p.use_tma_act) grid_dependency_wait();  // the activations are read with plain loads
    UnitIter it;
    it.init(cid, ncl, uk0, uk1);
    if (grp == 1) it.next();
    for (int i = grp; i < n_units; i += 2, it.next(), it.next()) {
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
        const int ci = gtid + r * kGroupWarps * 32;
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
      // 64 bytes = 256 codes of this row's half of the unit, as two quarters
      // of 128 codes (16-byte chunks 4h .. 4h+3 of the row, in the 128-byte
      // swizzle when TMA loaded them), each decoded into 32 TMEM columns
      const uint8_t* src = stage + row * UB;
      const int swz = p.use_tma_w ? (row & 7) : 0;
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int c0 = 4 * h + 2 * qq;
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
        tc2::tmem_st_32x32b_x32(lane_addr + kACol + ab * (UK / 4) + 32 * (2 * h + qq), v);
      }
      // activations -> this CTA's half of the B operand: row 2 ml = hi
      // digits, row 2 ml + 1 = lo digits, atoms of 128 k in the 128-byte swizzle
      uint8_t* bbuf = bop + ab * B_BUF;
#pragma unroll
      for (int r = 0; r < kActIters; ++r) {
        const int ci = gtid + r * kGroupWarps * 32;
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
          tc2::mbar_arrive_cluster_relaxed(a_full_lead0 + 8u * ab);
      }
    }
  } else if (warp == kProducerWarp) {
    // ------------------------------------- packed weights and activations in
    const int64_t kbytes = (static_cast<int64_t>(p.K) + 3) / 4;
    grid_dependency_wait();  // the inputs exist: the preceding grid has completed
    uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
    bool ok = true;
    const uint32_t tx = (p.use_tma_w ? RAW_W : 0) +
                        (p.use_tma_act ? (UK / ACT_BOX) * half_rows * ACT_BOX : 0);
    UnitIter it;
    it.init(cid, ncl, uk0, uk1);
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
      it.init(cid, ncl, uk0, uk1);
      for (int i = 0; i < n_units; ++i, it.next()) {
        const int ab = i % A_BUFS;
        const uint32_t aph = (i / A_BUFS) & 1;
        ++run_len;
        const bool seg_last = (i + 1 == n_units) || it.tile_last() || (run_len == RUN_MAX);
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
        umma_commit_to_pair(&a_empty[ab], lead);
        seg_first = seg_last;
        if (seg_last) {
          umma_commit_to_pair(acc_full, lead);
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
    const uint32_t acc_empty_lead = tc2::peer_addr(acc_empty, lead);
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const bool first_pair = qp == 0;
    // a CTA of a later pair sends its partials to the first pair's CTA of the
    // same rank (cluster rank `rank`), which holds the same weight rows
    const uint32_t slot_remote =
        first_pair ? 0u : tc2::peer_addr(slots + (qp - 1) * SLOT_BYTES + nloc * 16, rank);
    const uint32_t part_full_remote = first_pair ? 0u : tc2::peer_addr(part_full, rank);
    uint32_t acc_ph = 0, part_ph = 0, free_ph = 0;
    if (p.use_tma_out && etid == 0) prefetch_tensormap(&map_out);
    cluster_wait();
    grid_dependency_wait();  // C may be read by the preceding grid: write only after it
    UnitIter it;
    it.init(cid, ncl, uk0, uk1);
    int i = 0, tile_count = 0;
    bool run_first_of_tile = true;
    // The tile's int32 partial of this CTA accumulates in the staging buffer
    // [NB/2 rows m][128 n], each thread in its own column n (thread-private
    // words, so no synchronisation between runs).
    int32_t* sb = reinterpret_cast<int32_t*>(stage_out);
    while (i < n_units) {
      // the run of units of one tile that starts at unit i
      const int t = it.t;
      int len = 1;
      while (i + len < n_units && !it.tile_last() && len < RUN_MAX) {
        it.next();
        ++len;
      }
      const bool tile_end = it.tile_last() || i + len == n_units;
      bool ok = mbar_wait(acc_full, acc_ph, abort_flag, p.err, code_base | 4);
      ok = named_bar_and(kEpiBarrier, 128, __all_sync(0xffffffffu, ok));
      if (!ok) break;
      tc_fence_after();
      if (run_first_of_tile && p.use_tma_out && first_pair) {
        // the previous tile's store has read the staging buffer
        if (etid == 0) bulk_wait_group_read<0>();
        named_bar_sync(kEpiBarrier, 128);
      }
      // Summed over the issuers' accumulators, in units of 2^-9 (scaling by
      // 512 is exact): column 2m holds the hi digits' sum of row m, column
      // 2m + 1 the lo digits' sum, column ones_row the sum of the weights.
      int32_t bias = 0;  // 128 * sum_k w for unsigned digits
      if (!kSigned) {
        uint32_t o[kIss];
#pragma unroll
        for (int a = 0; a < kIss; ++a)
          asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                       : "=r"(o[a]) : "r"(lane_base + a * kAccStride + p.ones_row));
        tmem_wait_ld();
        int32_t ones = 0;
#pragma unroll
        for (int a = 0; a < kIss; ++a) ones += __float2int_rn(__uint_as_float(o[a]) * 512.0f);
        bias = 128 * ones;
      }
      // BW columns (BW/2 rows m) of every accumulator per TMEM round trip
      constexpr int BW = 32 / kIss;
      for (int cb = 0; cb < p.NB; cb += BW) {
        uint32_t d[kIss][BW];
#pragma unroll
        for (int a = 0; a < kIss; ++a) {
          if constexpr (BW == 16)
            tmem_ld_32x32b_x16(lane_base + a * kAccStride + cb, d[a]);
          else
            tmem_ld_32x32b_x8(lane_base + a * kAccStride + cb, d[a]);
        }
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < BW / 2; ++e) {
          int32_t hi = 0, lo = 0;
#pragma unroll
          for (int a = 0; a < kIss; ++a) {
            hi += __float2int_rn(__uint_as_float(d[a][2 * e]) * 512.0f);
            lo += __float2int_rn(__uint_as_float(d[a][2 * e + 1]) * 512.0f);
          }
          const int32_t v = 16 * hi + lo - bias;
          int32_t* dst = sb + (cb / 2 + e) * TN + nloc;
          *dst = run_first_of_tile ? v : *dst + v;
        }
      }
      tc_fence_before();
      __syncwarp();
      // the accumulator reads are complete (tcgen05.wait::ld): signal only
      if (lane == 0) tc2::mbar_arrive_cluster_relaxed(acc_empty_lead);
      acc_ph ^= 1u;
      run_first_of_tile = tile_end;
      i += len;
      if (i < n_units) it.next();
      if (!tile_end) continue;
      // ---- the tile's partial of this pair is complete in the staging buffer
      if (!first_pair) {
        // the first pair has read this CTA's previous partial
        if (tile_count > 0) {
          ok = mbar_wait(slot_free, free_ph, abort_flag, p.err, code_base | 4);
          free_ph ^= 1u;
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        for (int e = 0; e < p.m4; e += 4)
          st_async_v4(slot_remote + (e / 4) * SLOT_QUAD, sb[e * TN + nloc], sb[(e + 1) * TN + nloc],
                      sb[(e + 2) * TN + nloc], sb[(e + 3) * TN + nloc], part_full_remote);
        ++tile_count;
        continue;
      }
      if (p.split > 1) {
        if (etid == 0)
          mbar_arrive_expect_tx(part_full, static_cast<uint32_t>((p.split - 1) * TN * p.m4 * 4));
        ok = mbar_wait(part_full, part_ph, abort_flag, p.err, code_base | 4);
        part_ph ^= 1u;
        if (!named_bar_and(kEpiBarrier, 128, __all_sync(0xffffffffu, ok))) break;
        for (int e = 0; e < p.m4; e += 4) {
          int4 sum = make_int4(sb[e * TN + nloc], sb[(e + 1) * TN + nloc], sb[(e + 2) * TN + nloc],
                               sb[(e + 3) * TN + nloc]);
          for (int s = 1; s < p.split; ++s) {
            const int4 x = *reinterpret_cast<const int4*>(slots + (s - 1) * SLOT_BYTES +
                                                         (e / 4) * SLOT_QUAD + nloc * 16);
            sum.x += x.x;
            sum.y += x.y;
            sum.z += x.z;
            sum.w += x.w;
          }
          sb[e * TN + nloc] = sum.x;
          sb[(e + 1) * TN + nloc] = sum.y;
          sb[(e + 2) * TN + nloc] = sum.z;
          sb[(e + 3) * TN + nloc] = sum.w;
        }
        // every partial has been read: the other pairs may send the next
        // tile's (a cluster-scope release costs its thread about a microsecond,
        // so only when the cluster has a next tile)
        if (t + ncl < p.tiles) {
          named_bar_sync(kEpiBarrier, 128);
          if (etid == 0)
            for (int s = 1; s < p.split; ++s)
              tc2::mbar_arrive_cluster(tc2::peer_addr(slot_free, 2u * s + rank));
        }
      }
      const int n0 = t * TP + static_cast<int>(rank) * TN;
      const int64_t n = static_cast<int64_t>(n0) + nloc;
      if (p.use_tma_out) {
        fence_proxy_async_smem();
        named_bar_sync(kEpiBarrier, 128);
        if (etid == 0 && n0 < p.N) {  // a tile half wholly past N stores nothing
          tma_store_2d(&map_out, stage_out, n0, 0);
          bulk_commit_group();
        }
      } else if (n < p.N) {
        for (int e = 0; e < p.M; ++e) p.C[static_cast<int64_t>(e) * p.N + n] = sb[e * TN + nloc];
      }
      ++tile_count;
    }
    if (p.use_tma_out && etid == 0) bulk_wait_group_read<0>();  // the stores finish by themselves
  }

  tc_fence_before();
  __syncthreads();
  // No cross-CTA operation is in flight any more (the even CTA has seen the
  // odd CTA's last arrive, the odd CTA the last commit, the first pair every
  // partial); the barrier keeps every CTA's shared memory and the pair's TMEM
  // allocated until all CTAs of the cluster are done with them.
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
// grid to complete before anything else, then lets the next grid launch.
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

using KernelFn = void (*)(const Params, const CUtensorMap, const CUtensorMap, const CUtensorMap);

// Kernel variant: signed digits for M = 32 (two issuers); four issuers while
// each accumulator fits in 32 columns, else two.
KernelFn pick_kernel(int M, int NB) {
  if (M == 32) return skinny_fwd_kernel<true, 2>;
  return NB <= 32 ? skinny_fwd_kernel<false, 4> : skinny_fwd_kernel<false, 2>;
}

// How many clusters of 2S CTAs can be resident at once (cached per device,
// kernel variant and S).
int max_clusters(int dev, int variant, int S, KernelFn fn) {
  static std::atomic<int> cache[64][3][kMaxSplit + 1];
  int v = cache[dev][variant][S].load(std::memory_order_acquire);
  if (v > 0) return v;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * S, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_ALLOC;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) return -1;
  cache[dev][variant][S].store(n, std::memory_order_release);
  return n;
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
  p.m4 = static_cast<int>((M + 3) / 4 * 4);
  p.ones_row = signed_digits ? -1 : static_cast<int>(2 * M);
  const int64_t units_k = (K + sk::UK - 1) / sk::UK;
  const int64_t tiles = (N + sk::TP - 1) / sk::TP;
  if (tiles * units_k > 2147483647LL) return T3_EINVAL;
  p.units_k = static_cast<int>(units_k);
  p.tiles = static_cast<int>(tiles);
  p.err = err;
  const int64_t kbytes = (K + 3) / 4;
  CUtensorMap mw, mo, ma;
  p.use_tma_w = make_u8_map_tiled(&mw, Wp, N, kbytes, kbytes, sk::TN, sk::UB, true) ? 1 : 0;
  p.use_tma_act = make_u8_map_tiled(&ma, A, M, K, K, p.NB / 4, sk::ACT_BOX) ? 1 : 0;
  p.use_tma_out = make_i32_map_tiled(&mo, C, M, N, p.NB / 2, sk::TN, false) ? 1 : 0;
  if (!p.use_tma_w) mw = p.use_tma_act ? ma : mo;  // unused copies: any initialised map
  if (!p.use_tma_act) ma = mw;
  if (!p.use_tma_out) mo = mw;

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
  const sk::KernelFn fn = sk::pick_kernel(p.M, p.NB);
  const int variant = signed_digits ? 2 : (p.NB <= 32 ? 0 : 1);

  // Split: S pairs per cluster share a tile's reduction.  Estimated time in
  // units of one pair's unit: waves of tiles x units per slice, plus about one
  // unit for the partials' exchange when S > 1.  Every pair needs a nonempty
  // slice.  Ties go to the smaller cluster.
  int best_s = 1, best_clusters = 1;
  int64_t best_cost = -1;
  for (int S = 1; S <= sk::kMaxSplit; ++S) {
    const int64_t upp = (units_k + S - 1) / S;
    if (S > units_k || (S - 1) * upp >= units_k) continue;
    const int mc = sk::max_clusters(dev, variant, S, fn);
    if (mc < 1) continue;
    const int64_t ncl = tiles < mc ? tiles : mc;
    const int64_t waves = (tiles + ncl - 1) / ncl;
    const int64_t cost = waves * upp + (S > 1 ? 1 : 0);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_s = S;
      best_clusters = static_cast<int>(ncl);
    }
  }
  if (best_cost < 0) return T3_ECUDA;  // no cluster shape can be resident
  p.split = best_s;
  p.upp = static_cast<int>((units_k + best_s - 1) / best_s);

  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2 * best_s;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * best_s * best_clusters), 1, 1);
  cfg.blockDim = dim3(sk::kThreads, 1, 1);
  cfg.dynamicSmemBytes = sk::SMEM_ALLOC;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  (void)sms;
  if (cudaLaunchKernelEx(&cfg, fn, p, mw, mo, ma) != cudaSuccess) return T3_ECUDA;
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
