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
//   * swap-AB on the tensor core: D[n][m] = W^T[n][k] . A^T[k][m] with
//     tcgen05.mma kind::f16, M = 128 weight rows, N = 16 or 32 activation rows;
//   * the weights are decoded in registers straight into TMEM (the MMA's A
//     operand comes from TMEM), so the 8x-expanded weights never touch shared
//     memory; each unit is 128 weight rows x 384 k (a 12 KB TMA box), so that
//     every SM goes through only a handful of synchronisation rounds;
//   * the decode pairs code j with code j+4 of each 16-code word (two byte
//     permutes per four weights); the activations are written in the same
//     permuted reduction order, so every product and sum is unchanged;
//   * the units, ordered (k-group, weight tile, k-unit), are split evenly over
//     the SMs; each run of units that shares a weight tile ends with a TMA
//     reduce-add of its int32 partial into C, which the host zeroes first.
//     Integer addition makes the result independent of the order.
//   * a run spans at most one k-group (1536 k), so its f32 sum is an integer of
//     magnitude <= 128 * 1536 < 2^18 and converts to int32 exactly.
#include <atomic>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {
namespace sk {

constexpr int TN = 128;          // weight rows per tile (MMA M, TMEM lanes)
constexpr int UK = 384;          // reduction elements per unit
constexpr int UB = UK / 4;       // packed bytes per row per unit (96)
constexpr int GROUP = 4;         // units per activation slice (1536 k)
constexpr int GK = GROUP * UK;
constexpr int RAW_STAGES = 4;
constexpr int A_BUFS = 2;        // TMEM operand buffers of UK/2 columns
constexpr int MP_MAX = 32;
constexpr int TMEM_COLS = 512;
constexpr int kAccCol = 0;       // two accumulators of MP_MAX columns
constexpr int kACol = 64;        // two unit buffers of 192 columns
constexpr int kDecWarps = 8;     // two per lane quadrant: halves of the unit
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kEpiWarp0 = 10;
constexpr int kThreads = 448;
constexpr int kEpiBarrier = 1;

constexpr int RAW_BYTES = TN * UB;                 // 12 KB of codes per unit
constexpr int ACT_ATOM = MP_MAX * 128;             // [32 rows][64 f16] per 64 k
constexpr int ACT_ATOMS = GK / 64;                 // 24 atoms = 96 KB
constexpr int STAGE_OUT = MP_MAX * TN * 4;         // [32 rows][128 int32]
constexpr int OFF_ACT = 0;
constexpr int OFF_RAW = OFF_ACT + ACT_ATOMS * ACT_ATOM;
constexpr int OFF_OUT = OFF_RAW + RAW_STAGES * RAW_BYTES;
constexpr int OFF_BAR = OFF_OUT + 2 * STAGE_OUT;
constexpr int N_BARS = 2 * RAW_STAGES + 2 * A_BUFS + 4 + 2;
constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;

struct Params {
  const int8_t* A;     // [M][K]
  const uint8_t* Wp;   // [N][ceil(K/4)]
  int32_t* C;          // [M][N], zeroed by the host
  int M, N, K, MP;
  int units_total, tiles, units_k;  // units along k per tile
  int use_tma_w, use_tma_out;
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

// 16 codes (one word, code i at bits 2i) -> 8 f16x2 words in the permuted
// reduction order: word 2j = (code j, code j+4), word 2j+1 = (code j+8, code j+12).
__device__ __forceinline__ void decode16_pairs(uint32_t x, uint32_t* o) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t sh = (j < 3) ? (x << (4 - 2 * j)) : (x >> 2);
    const uint32_t s = (sh & 0x30303030u) | 0x04040404u;
    o[2 * j] = prmt(tc::kF16HiTable, 0u, s);
    o[2 * j + 1] = prmt(tc::kF16HiTable, 0u, s >> 16);
  }
}

__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Activations of units [uk0, uk1) of k-group g -> f16 atoms in shared memory,
// rows m < M (rows up to MP stay zero), in the decode's permuted order.  Each
// thread loads a batch of 16-byte chunks before converting any.
__device__ __forceinline__ void convert_act(const Params& p, uint8_t* act, int g, int uk0, int uk1,
                                            int tid) {
  constexpr int kBatch = 8;
  const int k_base = g * GK + uk0 * UK;
  const int chunks_per_row = (uk1 - uk0) * (UK / 16);
  const int total = p.MP * chunks_per_row;
  const bool vec = (p.K % 16 == 0) && (reinterpret_cast<uintptr_t>(p.A) % 16 == 0);
  for (int base = 0; base < total; base += 128 * kBatch) {
    uint4 x[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int i = base + b * 128 + tid;
      x[b] = make_uint4(0u, 0u, 0u, 0u);
      if (i >= total) continue;
      const int m = i / chunks_per_row, c = i % chunks_per_row;
      const int64_t k0 = static_cast<int64_t>(k_base) + 16 * c;
      if (m >= p.M) continue;
      const int8_t* src = p.A + static_cast<int64_t>(m) * p.K + k0;
      if (vec && k0 + 16 <= p.K) {
        x[b] = __ldg(reinterpret_cast<const uint4*>(src));
      } else {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        for (int j = 0; j < 16; ++j)
          if (k0 + j < p.K)
            w[j >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(__ldg(src + j))) << (8 * (j & 3));
        x[b] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int i = base + b * 128 + tid;
      if (i >= total) continue;
      const int m = i / chunks_per_row, c = i % chunks_per_row;
      const int kk = uk0 * UK + 16 * c;  // offset within the group
      uint32_t Y[4];
      tc::transpose4x4(x[b].x, x[b].y, x[b].z, x[b].w, Y);  // reduction order 0,4,8,12,1,5,...
      uint4 o0, o1;
      tc::s8x4_to_f16(Y[0], o0.x, o0.y);
      tc::s8x4_to_f16(Y[1], o0.z, o0.w);
      tc::s8x4_to_f16(Y[2], o1.x, o1.y);
      tc::s8x4_to_f16(Y[3], o1.z, o1.w);
      uint8_t* atom = act + (kk >> 6) * ACT_ATOM;
      const int sub = (kk & 63) >> 4;
      *reinterpret_cast<uint4*>(atom + tc::sw128(m, 2 * sub)) = o0;
      *reinterpret_cast<uint4*>(atom + tc::sw128(m, 2 * sub + 1)) = o1;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    skinny_fwd_kernel(const Params p, const __grid_constant__ CUtensorMap map_w,
                      const __grid_constant__ CUtensorMap map_out) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((base_addr + 1023u) & ~1023u) - base_addr);
  uint8_t* act = smem + OFF_ACT;
  uint8_t* raw = smem + OFF_RAW;
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
      mbar_init(&raw_empty[s], kDecWarps);
    }
    for (int s = 0; s < A_BUFS; ++s) {
      mbar_init(&a_full[s], kDecWarps);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 4);
    }
    mbar_init(act_full, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  // rows MP..31 of the activation atoms are never written: keep them zero
  for (int i = threadIdx.x; i < ACT_ATOMS * ACT_ATOM / 16; i += kThreads)
    reinterpret_cast<uint4*>(act)[i] = make_uint4(0, 0, 0, 0);
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp < kDecWarps) {
    // ------------------------------------------------ weight decode -> TMEM
    const int q = warp & 3, h = warp >> 2;  // lane quadrant, half of the unit
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    for (int i = 0; i < n_units; ++i) {
      const int rs = i & (RAW_STAGES - 1), ab = i & (A_BUFS - 1);
      const uint32_t rph = (i / RAW_STAGES) & 1, aph = (i / A_BUFS) & 1;
      bool ok = mbar_wait(&raw_full[rs], rph, abort_flag, p.err, code_base | 2) &&
                mbar_wait(&a_empty[ab], aph ^ 1u, abort_flag, p.err, code_base | 2);
      if (!__all_sync(0xffffffffu, ok)) break;
      // 48 bytes = 12 words = 192 codes of this row's half of the unit
      const uint8_t* src = raw + rs * RAW_BYTES + row * UB + 48 * h;
      const uint32_t col0 = kACol + ab * (UK / 2) + 96 * h;
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        const uint4 x = *reinterpret_cast<const uint4*>(src + 16 * part);
        uint32_t v[32];
        decode16_pairs(x.x, v);
        decode16_pairs(x.y, v + 8);
        decode16_pairs(x.z, v + 16);
        decode16_pairs(x.w, v + 24);
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
    UnitIter it;
    it.init(p, u0);
    for (int i = 0; i < n_units; ++i, it.next()) {
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
      const uint32_t idesc = idesc_f16_f32(TN, p.MP);
      uint32_t acc_b = 0, acc_ph = 0, act_ph = 0;
      int cur_g = -1;
      bool ok = true, issued_any = false, seg_first = true;
      UnitIter it;
      it.init(p, u0);
      for (int i = 0; i < n_units; ++i, it.next()) {
        const int ab = i & (A_BUFS - 1);
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
        const uint32_t b0 = smem_addr(act + it.uk * (UK / 64) * ACT_ATOM);
        const uint32_t d_tmem = tmem_base + kAccCol + acc_b * MP_MAX;
        const uint32_t a_tmem = tmem_base + kACol + ab * (UK / 2);
#pragma unroll 4
        for (int j = 0; j < UK / 16; ++j)
          umma_f16_ts(d_tmem, a_tmem + 8 * j,
                      smem_desc_k_sw128(b0 + (j >> 2) * ACT_ATOM + 32 * (j & 3)), idesc,
                      (!seg_first || j > 0) ? 1u : 0u);
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
    uint32_t acc_b = 0, acc_ph = 0, slab = 0;
    int cur_g = -1;
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
        convert_act(p, act, g, lo, hi, etid);
        fence_proxy_async_smem();
        named_bar_sync(kEpiBarrier, 128);
        if (etid == 0) mbar_arrive(act_full);
        cur_g = g;
      }
      bool ok = mbar_wait(&acc_full[acc_b], acc_ph, abort_flag, p.err, code_base | 4);
      ok = named_bar_and(kEpiBarrier, 128, __all_sync(0xffffffffu, ok));
      if (!ok) break;
      tc_fence_after();
      uint32_t val[32];
      tmem_ld_32x32b_x32(
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kAccCol + acc_b * MP_MAX, val);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc_b]);
      if (++acc_b == 2) { acc_b = 0; acc_ph ^= 1u; }
      const int64_t n = static_cast<int64_t>(t) * TN + nloc;
      if (p.use_tma_out) {
        uint8_t* buf = stage_out + (slab & 1) * STAGE_OUT;
        if (etid == 0) bulk_wait_group_read<1>();
        named_bar_sync(kEpiBarrier, 128);
        int32_t* sb = reinterpret_cast<int32_t*>(buf);
#pragma unroll
        for (int m = 0; m < MP_MAX; ++m)
          if (m < p.MP) sb[m * TN + nloc] = tc::f32_bits_to_i32(val[m]);
        fence_proxy_async_smem();
        named_bar_sync(kEpiBarrier, 128);
        if (etid == 0) {
          tma_reduce_add_2d(&map_out, buf, t * TN, 0);
          bulk_commit_group();
        }
        ++slab;
      } else if (n < p.N) {
#pragma unroll
        for (int m = 0; m < MP_MAX; ++m)
          if (m < p.M)
            atomicAdd(p.C + static_cast<int64_t>(m) * p.N + n, tc::f32_bits_to_i32(val[m]));
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
  CUtensorMap mw, mo;
  p.use_tma_w = make_u8_map_tiled(&mw, Wp, N, kbytes, kbytes, sk::TN, sk::UB) ? 1 : 0;
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
  sk::skinny_fwd_kernel<<<grid, sk::kThreads, sk::SMEM_ALLOC, s>>>(p, mw, mo);
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

}  // namespace t3
