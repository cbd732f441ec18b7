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
//   * swap-AB on the tensor core with 8-bit floats: D[n][.] = W^T[n][k] . B[k][.]
//     with tcgen05.mma kind::f8f6f4 (e4m3 x e4m3 -> f32), M = 128 weight rows,
//     K = 32 per instruction.  Every weight is exact in e4m3 (+1 = 0x38,
//     -1 = 0xB8).  An int8 activation a is split into a = 16*hi + lo with
//     hi in [-8, 7] and lo in [0, 15], both exact in e4m3; the hi digits of
//     the M activation rows and then their lo digits form the B operand
//     (N = 2 * 16 or 2 * 32 rows), and C = 16 * D_hi + D_lo in the epilogue.
//     An instruction costs its issuing thread about as much at N = 64 as at
//     N = 16, so doubling K per instruction (over f16) doubles the rate;
//   * the weights are decoded in registers straight into TMEM (the MMA's A
//     operand comes from TMEM, 4 e4m3 values per 32-bit column), one byte
//     permute per four weights; each unit is 128 weight rows x 512 k (a 16 KB
//     TMA box), so every SM goes through only a handful of synchronisation
//     rounds;
//   * the decode takes the even codes of a 16-code word, then the odd ones;
//     the activations are written in the same permuted reduction order, so
//     every product and sum is unchanged;
//   * the units, ordered (k-group, weight tile, k-unit), are split evenly over
//     the SMs; each run of units that shares a weight tile ends with a TMA
//     reduce-add of its int32 partial into C, which the host zeroes first.
//     Integer addition makes the result independent of the order.
//   * a run spans at most one k-group (1536 k), so each digit plane's f32 sum
//     is an integer of magnitude <= 15 * 1536 < 2^15: exact.
#include <atomic>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {
namespace sk {

constexpr int TN = 128;          // weight rows per tile (MMA M, TMEM lanes)
constexpr int UK = 512;          // reduction elements per unit
constexpr int UB = UK / 4;       // packed bytes per row per unit (128)
constexpr int GROUP = 3;         // units per activation slice (1536 k)
constexpr int GK = GROUP * UK;
constexpr int RAW_STAGES = 3;
constexpr int A_BUFS = 3;        // TMEM operand buffers of UK/4 columns
constexpr int MP_MAX = 32;
constexpr int TMEM_COLS = 512;
constexpr int kAccCol = 0;       // two accumulators of 2 * MP_MAX columns
constexpr int kACol = 128;       // three unit buffers of UK / 4 = 128 columns
constexpr int kDecGroupWarps = 8;  // one group: two warps per lane quadrant (unit halves)
constexpr int kDecGroups = 2;      // groups take alternate units
constexpr int kDecWarps = kDecGroupWarps * kDecGroups;
constexpr int kProducerWarp = kDecWarps;
constexpr int kMmaWarp = kDecWarps + 1;
constexpr int kEpiWarp0 = kDecWarps + 2;
constexpr int kThreads = 32 * (kDecWarps + 2 + 4);
constexpr int kEpiBarrier = 1;

constexpr int RAW_BYTES = TN * UB;                 // 16 KB of codes per unit
constexpr int ACT_ATOM = 2 * MP_MAX * 128;         // [hi rows; lo rows][128 e4m3] per 128 k
constexpr int ACT_ATOMS = GK / 128;                // 12 atoms = 96 KB
constexpr int STAGE_OUT = MP_MAX * TN * 4;         // [32 rows][128 int32]
constexpr int ACT_BOX = 256;                       // activation bytes per TMA box row
constexpr int RAW_ACT = MP_MAX * GK;               // int8 activation slice [32][1536]
constexpr int OFF_ACT = 0;
constexpr int OFF_RAW = OFF_ACT + ACT_ATOMS * ACT_ATOM;
constexpr int OFF_RAW_ACT = OFF_RAW + RAW_STAGES * RAW_BYTES;
constexpr int OFF_OUT = OFF_RAW_ACT + RAW_ACT;
constexpr int OFF_BAR = OFF_OUT + 2 * STAGE_OUT;
constexpr int N_BARS = 2 * RAW_STAGES + 2 * A_BUFS + 4 + 2 + 1;
constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;

struct Params {
  const int8_t* A;     // [M][K]
  const uint8_t* Wp;   // [N][ceil(K/4)]
  int32_t* C;          // [M][N], zeroed by the host
  int M, N, K, MP;
  int units_total, tiles, units_k;  // units along k per tile
  int use_tma_w, use_tma_out, use_tma_act;
  int* err;
};

// Walks units in (k-group, tile, k-unit) order; only the starting unit is
// decoded with divisions.
struct UnitIter {
  int g, t, uk;       // k-group, tile, unit within the group
  int nk;             // units in the current group
  int tiles, units_k;
  __device__ void init(const Params& p, int u) {
    tiles = p.tiles;
    units_k = p.units_k;
    const int full = tiles * GROUP;
    g = u / full;
    nk = min(GROUP, units_k - g * GROUP);
    const int rem = u - g * full;
    t = rem / nk;
    uk = rem % nk;
  }
  __device__ int k_unit() const { return g * GROUP + uk; }
  __device__ void next() {
    if (++uk == nk) {
      uk = 0;
      if (++t == tiles) {
        t = 0;
        ++g;
        nk = min(GROUP, units_k - g * GROUP);
      }
    }
  }
  __device__ bool last_of_run() const { return uk + 1 == nk; }
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

// f32 (+)= e4m3 A (TMEM) x e4m3 B (shared memory descriptor).
__device__ __forceinline__ void umma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor: e4m3 x e4m3 -> f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// Two f16 values (exact small integers) -> two e4m3 bytes in the low half.
__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
  return r;
}

// Four int8 (a word) -> their hi digits (a >> 4) and lo digits (a & 15) as
// e4m3 bytes, in the same byte order.
__device__ __forceinline__ void s8x4_to_digits_e4m3(uint32_t x, uint32_t& hi, uint32_t& lo) {
  const uint32_t u = x ^ 0x80808080u;              // a + 128
  const uint32_t uh = (u >> 4) & 0x0F0F0F0Fu;      // hi + 8
  const uint32_t ul = u & 0x0F0F0F0Fu;             // lo
  const uint32_t h01 = hsub2(prmt(uh, 0x64646464u, 0x4140u), 0x64086408u);  // 1024+v - 1032
  const uint32_t h23 = hsub2(prmt(uh, 0x64646464u, 0x4342u), 0x64086408u);
  const uint32_t l01 = hsub2(prmt(ul, 0x64646464u, 0x4140u), 0x64006400u);
  const uint32_t l23 = hsub2(prmt(ul, 0x64646464u, 0x4342u), 0x64006400u);
  hi = f16x2_to_e4m3x2(h01) | (f16x2_to_e4m3x2(h23) << 16);
  lo = f16x2_to_e4m3x2(l01) | (f16x2_to_e4m3x2(l23) << 16);
}

// 16 activations -> the e4m3 hi and lo digit words of one 16-element group,
// in the decode's permuted order (even bytes, then odd bytes).
__device__ __forceinline__ void act16_to_planes(const uint4 x, uint4& hi, uint4& lo) {
  const uint32_t y0 = prmt(x.x, x.y, 0x6420u), y1 = prmt(x.z, x.w, 0x6420u);
  const uint32_t y2 = prmt(x.x, x.y, 0x7531u), y3 = prmt(x.z, x.w, 0x7531u);
  s8x4_to_digits_e4m3(y0, hi.x, lo.x);
  s8x4_to_digits_e4m3(y1, hi.y, lo.y);
  s8x4_to_digits_e4m3(y2, hi.z, lo.z);
  s8x4_to_digits_e4m3(y3, hi.w, lo.w);
}

// Activations of units [uk0, uk1) of k-group g -> e4m3 digit planes in shared
// memory: row m holds the hi digits of activation row m, row MP+m its lo
// digits, each 16-element group in the decode's permuted order.  Rows of absent
// activations get digit 0.  The source is the raw slice the producer loaded
// with TMA (rows MP x GK bytes, zero outside the matrix) or, when A cannot be a
// TMA source, global memory directly.
__device__ __forceinline__ void convert_act(const Params& p, uint8_t* act, const uint8_t* raw_act,
                                            int g, int uk0, int uk1, int tid, int nthreads) {
  const int k_base = g * GK + uk0 * UK;
  const int chunks_per_row = (uk1 - uk0) * (UK / 16);
  const int total = p.MP * chunks_per_row;
  for (int i = tid; i < total; i += nthreads) {
    const int m = i / chunks_per_row, c = i % chunks_per_row;
    const int kk = uk0 * UK + 16 * c;  // offset within the group
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (p.use_tma_act) {
      // box b holds k in [256 b, 256 b + 256) of all MP_MAX rows
      x = *reinterpret_cast<const uint4*>(raw_act + (kk >> 8) * (ACT_BOX * MP_MAX) + m * ACT_BOX +
                                          (kk & (ACT_BOX - 1)));
    } else if (m < p.M) {
      const int64_t k0 = static_cast<int64_t>(k_base) + 16 * c;
      const int8_t* src = p.A + static_cast<int64_t>(m) * p.K + k0;
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      for (int j = 0; j < 16; ++j)
        if (k0 + j < p.K)
          w[j >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(__ldg(src + j))) << (8 * (j & 3));
      x = make_uint4(w[0], w[1], w[2], w[3]);
    }
    uint4 hi, lo;
    act16_to_planes(x, hi, lo);
    uint8_t* atom = act + (kk >> 7) * ACT_ATOM;
    const int chunk = (kk & 127) >> 4;
    *reinterpret_cast<uint4*>(atom + tc::sw128(m, chunk)) = hi;
    *reinterpret_cast<uint4*>(atom + tc::sw128(p.MP + m, chunk)) = lo;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    skinny_fwd_kernel(const Params p, const __grid_constant__ CUtensorMap map_w,
                      const __grid_constant__ CUtensorMap map_out,
                      const __grid_constant__ CUtensorMap map_act) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((base_addr + 1023u) & ~1023u) - base_addr);
  uint8_t* act = smem + OFF_ACT;
  uint8_t* raw = smem + OFF_RAW;
  uint8_t* raw_act = smem + OFF_RAW_ACT;
  uint8_t* stage_out = smem + OFF_OUT;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + RAW_STAGES;
  uint64_t* a_full = raw_empty + RAW_STAGES;
  uint64_t* a_empty = a_full + A_BUFS;
  uint64_t* acc_full = a_empty + A_BUFS;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* act_full = acc_empty + 2;
  uint64_t* drain_bar = act_full + 1;
  uint64_t* act_raw_full = drain_bar + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u0 = static_cast<int>(static_cast<int64_t>(p.units_total) * blockIdx.x / gridDim.x);
  const int u1 =
      static_cast<int>(static_cast<int64_t>(p.units_total) * (blockIdx.x + 1) / gridDim.x);
  const int n_units = u1 - u0;
  constexpr int code_base = 4 << 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW_STAGES; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kDecGroupWarps);
    }
    for (int s = 0; s < A_BUFS; ++s) {
      mbar_init(&a_full[s], kDecGroupWarps);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 4);
    }
    mbar_init(act_full, 1);
    mbar_init(drain_bar, 1);
    mbar_init(act_raw_full, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // The first k-group's activation slice is converted by the decoder and
  // epilogue warps together (384 threads): nothing else can run before it.
  constexpr int kCoopThreads = (kDecWarps + 4) * 32;
  const bool coop = (warp < kDecWarps) || (warp >= kEpiWarp0);
  int first_g = -1;
  if (n_units > 0) {
    UnitIter it0;
    it0.init(p, u0);
    first_g = it0.g;
    if (coop) {
      const int ctid = (warp < kDecWarps) ? threadIdx.x : threadIdx.x - 64;  // 0..kCoop-1
      int lo = it0.uk, hi = it0.uk + 1;
      UnitIter scan = it0;
      for (int j = 1; j < n_units; ++j) {
        scan.next();
        if (scan.g != first_g) break;
        lo = min(lo, scan.uk);
        hi = max(hi, scan.uk + 1);
      }
      bool okr = true;
      if (p.use_tma_act) okr = mbar_wait(act_raw_full, 0, abort_flag, p.err, code_base | 4);
      okr = named_bar_and(2, kCoopThreads, __all_sync(0xffffffffu, okr));
      if (okr) {
        convert_act(p, act, raw_act, first_g, lo, hi, ctid, kCoopThreads);
        fence_proxy_async_smem();
      }
      named_bar_sync(2, kCoopThreads);
      if (ctid == 0) mbar_arrive(act_full);
    }
  }

  if (warp < kDecWarps) {
    // ------------------------------------------------ weight decode -> TMEM
    const int q = warp & 3, h = (warp >> 2) & 1;  // lane quadrant, half of the unit
    const int grp = warp / kDecGroupWarps;          // this group's units: i % kDecGroups == grp
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    for (int i = grp; i < n_units; i += kDecGroups) {
      const int rs = i % RAW_STAGES, ab = i % A_BUFS;  // compile-time divisors
      const uint32_t rph = (i / RAW_STAGES) & 1, aph = (i / A_BUFS) & 1;
      bool ok = mbar_wait(&raw_full[rs], rph, abort_flag, p.err, code_base | 2) &&
                mbar_wait(&a_empty[ab], aph ^ 1u, abort_flag, p.err, code_base | 2);
      if (!__all_sync(0xffffffffu, ok)) break;
      // 64 bytes = 16 words = 256 codes of this row's half of the unit: 16-byte
      // chunks 4h..4h+3 of the row, stored in the 128-byte swizzle when TMA
      // loaded them (so that the 32 rows of a warp hit distinct banks)
      const uint8_t* src = raw + rs * RAW_BYTES + row * UB;
      const int swz = p.use_tma_w ? (row & 7) : 0;
      const uint32_t col0 = kACol + ab * (UK / 4) + 64 * h;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int c0 = 4 * h + 2 * part;
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
        tc2::tmem_st_32x32b_x32(lane_addr + col0 + 32 * part, v);
      }
      tc2::tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&raw_empty[rs]);
        mbar_arrive(&a_full[ab]);
      }
    }
  } else if (warp == kProducerWarp) {
    // --------------------------------------------------- packed weights in
    if (lane == 0 && p.use_tma_w) prefetch_tensormap(&map_w);
    uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
    bool ok = true;
    const int64_t kbytes = (static_cast<int64_t>(p.K) + 3) / 4;
    if (lane == 0 && p.use_tma_act) prefetch_tensormap(&map_act);
    UnitIter it;
    it.init(p, u0);
    int act_g = -1;
    uint32_t act_loads = 0;
    for (int i = 0; i < n_units; ++i, it.next()) {
      if (p.use_tma_act && it.g != act_g) {
        // The raw slice of a new group: the converters of the previous group
        // have finished with the buffer once the MMA has consumed its units,
        // which the raw_empty wait of the current unit does not prove, so wait
        // for the conversion to be published (act_full) first.
        if (lane == 0 && act_loads > 0)
          ok = mbar_wait(act_full, (act_loads - 1) & 1u, abort_flag, p.err, code_base | 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(act_raw_full, RAW_ACT);
          for (int b = 0; b < GK / ACT_BOX; ++b)
            tma_load_2d(raw_act + b * ACT_BOX * MP_MAX, &map_act, act_raw_full,
                        it.g * GK + b * ACT_BOX, 0);
        }
        ++act_loads;
        act_g = it.g;
      }
      if (lane == 0)
        ok = mbar_wait(&raw_empty[stage], phase ^ 1u, abort_flag, p.err, code_base | 1);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      uint8_t* dst = raw + stage * RAW_BYTES;
      const int x0 = it.k_unit() * UB, y0 = it.t * TN;
      if (!p.use_tma_w) {
        tc::manual_box(dst, p.Wp, kbytes, p.N, kbytes, y0, x0, TN, UB, lane);
        __threadfence_block();
        __syncwarp();
      }
      if (lane == 0) {
        if (p.use_tma_w) {
          mbar_arrive_expect_tx(&raw_full[stage], RAW_BYTES);
          tma_load_2d(dst, &map_w, &raw_full[stage], x0, y0);
        } else {
          mbar_arrive(&raw_full[stage]);
        }
      }
      issued_mask |= 1u << stage;
      issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
      if (++stage == RAW_STAGES) { stage = 0; phase ^= 1u; }
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
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_e4m3_f32(TN, 2 * p.MP);
      uint32_t acc_b = 0, acc_ph = 0, act_ph = 0;
      int cur_g = -1;
      bool ok = true, issued_any = false, seg_first = true;
      UnitIter it;
      it.init(p, u0);
      for (int i = 0; i < n_units; ++i, it.next()) {
        const int ab = i % A_BUFS;
        const uint32_t aph = (i / A_BUFS) & 1;
        const bool seg_last = (i + 1 == n_units) || it.last_of_run();
        if (seg_first) {
          ok = mbar_wait(&acc_empty[acc_b], acc_ph ^ 1u, abort_flag, p.err, code_base | 3);
          if (ok && it.g != cur_g) {
            ok = mbar_wait(act_full, act_ph, abort_flag, p.err, code_base | 3);
            act_ph ^= 1u;
            cur_g = it.g;
          }
        }
        if (ok) ok = mbar_wait(&a_full[ab], aph, abort_flag, p.err, code_base | 3);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + kAccCol + acc_b * (2 * MP_MAX);
        const uint32_t a_tmem = tmem_base + kACol + ab * (UK / 4);
        // descriptor of k-step j = base + (atom j/4, 32-byte step j%4): only the
        // 14-bit start-address field changes, by (offset >> 4)
        const uint64_t bdesc0 = smem_desc_k_sw128(smem_addr(act + it.uk * (UK / 128) * ACT_ATOM));
        umma_f8_ts(d_tmem, a_tmem, bdesc0, idesc, seg_first ? 0u : 1u);
#pragma unroll
        for (int j = 1; j < UK / 32; ++j)
          umma_f8_ts(d_tmem, a_tmem + 8 * j,
                     bdesc0 + static_cast<uint64_t>(((j >> 2) * ACT_ATOM + 32 * (j & 3)) >> 4),
                     idesc, 1u);
        issued_any = true;
        umma_commit(&a_empty[ab]);
        seg_first = seg_last;
        if (seg_last) {
          umma_commit(&acc_full[acc_b]);
          if (++acc_b == 2) { acc_b = 0; acc_ph ^= 1u; }
        }
      }
      if (!ok && issued_any) {
        umma_commit(drain_bar);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------- activation slices and epilogue
    const int q = warp & 3;
    const int etid = threadIdx.x - kEpiWarp0 * 32;
    const int nloc = q * 32 + lane;
    uint32_t acc_b = 0, acc_ph = 0, slab = 0, act_raw_ph = 1;  // phase 0 was the first group
    int cur_g = first_g;
    if (p.use_tma_out && etid == 0) prefetch_tensormap(&map_out);
    UnitIter it;
    it.init(p, u0);
    int i = 0;
    while (i < n_units) {
      // the run of units that shares (k-group, tile) with unit i
      const int g = it.g, t = it.t, uk_first = it.uk;
      int len = 1;
      while (i + len < n_units && !it.last_of_run()) {
        it.next();
        ++len;
      }
      const int uk_last = it.uk;
      if (g != cur_g) {
        // k-units of this group that this CTA's remaining runs touch
        int lo = uk_first, hi = uk_last + 1;
        UnitIter scan = it;
        for (int j = i + len; j < n_units; ++j) {
          scan.next();
          if (scan.g != g) break;
          lo = min(lo, scan.uk);
          hi = max(hi, scan.uk + 1);
        }
        if (p.use_tma_act) {
          bool okr = mbar_wait(act_raw_full, act_raw_ph, abort_flag, p.err, code_base | 4);
          okr = named_bar_and(kEpiBarrier, 128, __all_sync(0xffffffffu, okr));
          if (!okr) break;
          act_raw_ph ^= 1u;
        }
        convert_act(p, act, raw_act, g, lo, hi, etid, 128);
        fence_proxy_async_smem();
        named_bar_sync(kEpiBarrier, 128);
        if (etid == 0) mbar_arrive(act_full);
        cur_g = g;
      }
      bool ok = mbar_wait(&acc_full[acc_b], acc_ph, abort_flag, p.err, code_base | 4);
      ok = named_bar_and(kEpiBarrier, 128, __all_sync(0xffffffffu, ok));
      if (!ok) break;
      tc_fence_after();
      // C = 16 * (hi digit plane) + (lo digit plane), both exact integers.
      // Columns [0, MP) hold the hi plane, [MP, 2 MP) the lo plane.
      const uint32_t acc_addr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kAccCol + acc_b * (2 * MP_MAX);
      const int64_t n = static_cast<int64_t>(t) * TN + nloc;
      uint8_t* buf = stage_out + (slab & 1) * STAGE_OUT;
      if (p.use_tma_out) {
        if (etid == 0) bulk_wait_group_read<1>();
        named_bar_sync(kEpiBarrier, 128);
      }
      int32_t* sb = reinterpret_cast<int32_t*>(buf);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // rows m in [16 half, 16 half + 16): hi at column m, lo at column MP + m
        uint32_t dh[16], dl[16];
        tmem_ld_32x32b_x16(acc_addr + 16 * half, dh);
        tmem_ld_32x32b_x16(acc_addr + p.MP + 16 * half, dl);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = 16 * half + j;
          const int32_t v = 16 * tc::f32_bits_to_i32(dh[j]) + tc::f32_bits_to_i32(dl[j]);
          if (p.use_tma_out) {
            if (m < p.MP) sb[m * TN + nloc] = v;
          } else if (n < p.N && m < p.M) {
            atomicAdd(p.C + static_cast<int64_t>(m) * p.N + n, v);
          }
        }
        if (p.MP == 16) break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc_b]);
      if (++acc_b == 2) { acc_b = 0; acc_ph ^= 1u; }
      if (p.use_tma_out) {
        fence_proxy_async_smem();
        named_bar_sync(kEpiBarrier, 128);
        if (etid == 0) {
          tma_reduce_add_2d(&map_out, buf, t * TN, 0);
          bulk_commit_group();
        }
        ++slab;
      }
      i += len;
      if (i < n_units) it.next();
    }
    if (p.use_tma_out && etid == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace sk

int launch_skinny_fwd(const int8_t* A, const uint8_t* Wp, int32_t* C, int64_t M, int64_t N,
                      int64_t K, int sms, int* err, cudaStream_t s) {
  sk::Params p{};
  p.A = A;
  p.Wp = Wp;
  p.C = C;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.MP = M <= 16 ? 16 : 32;
  p.units_k = static_cast<int>((K + sk::UK - 1) / sk::UK);
  p.tiles = static_cast<int>((N + sk::TN - 1) / sk::TN);
  const int64_t units = static_cast<int64_t>(p.units_k) * p.tiles;
  if (units > 2147483647LL) return T3_EINVAL;
  p.units_total = static_cast<int>(units);
  p.err = err;
  const int64_t kbytes = (K + 3) / 4;
  CUtensorMap mw, mo, ma;
  p.use_tma_w = make_u8_map_tiled(&mw, Wp, N, kbytes, kbytes, sk::TN, sk::UB, true) ? 1 : 0;
  p.use_tma_act = make_u8_map_tiled(&ma, A, M, K, K, sk::MP_MAX, sk::ACT_BOX) ? 1 : 0;
  p.use_tma_out = make_i32_map_tiled(&mo, C, M, N, p.MP, sk::TN, false) ? 1 : 0;
  if (cudaMemsetAsync(C, 0, static_cast<size_t>(M) * N * sizeof(int32_t), s) != cudaSuccess)
    return T3_ECUDA;
  int grid = static_cast<int>(units < sms ? units : sms);
  if (grid < 1) grid = 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return T3_ECUDA;
  static std::atomic<bool> attr_done[64];
  if (dev < 0 || dev >= 64) return T3_EDEVICE;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(sk::skinny_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             sk::SMEM_ALLOC) != cudaSuccess)
      return T3_ECUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  sk::skinny_fwd_kernel<<<grid, sk::kThreads, sk::SMEM_ALLOC, s>>>(p, mw, mo, ma);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
