// t3_api.cu -- the C ABI: argument checks, the host packer, TMA descriptors,
// launches and the device error word.  See include/t3.h for the contract.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {

// One error word per device (a __device__ variable has one instance per
// device context).  Kernels receive its address; t3_last_device_error reads
// and clears it.
__device__ int g_error_word;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}


bool make_u8_map_tiled(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                       int box_rows, int box_cols, bool swizzle128) {
  std::memset(map, 0, sizeof(*map));
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || ld % 16 != 0) return false;
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) std::memset(map, 0, sizeof(*map));
  return r == CUDA_SUCCESS;
}

bool make_i32_map_tiled(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                        int box_rows, int box_cols, bool swizzle128) {
  std::memset(map, 0, sizeof(*map));
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || (cols * 4) % 16 != 0) return false;
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 4)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) std::memset(map, 0, sizeof(*map));
  return r == CUDA_SUCCESS;
}

// bf16 matrix [rows][cols] (cols elements of 2 bytes per row) as 16-bit
// elements, boxes of box_cols x box_rows in the 128-byte swizzle.
bool make_u16_map_tiled(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                        int box_rows, int box_cols) {
  std::memset(map, 0, sizeof(*map));
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || (cols * 2) % 16 != 0) return false;
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) std::memset(map, 0, sizeof(*map));
  return r == CUDA_SUCCESS;
}

// Output tensor map of the pair pipeline for output kind `kind` (tc2::kOutI32
// or a T3_OUT_* kind): boxes of 32 columns x 128 rows; int32 and float rows
// in the 128-byte swizzle, bf16 rows (64 bytes) unswizzled.
bool make_out_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int kind) {
  if (kind == tc2::kOutI32) return make_i32_map_tiled(map, base, rows, cols, 128, 32, true);
  std::memset(map, 0, sizeof(*map));
  const int64_t esize = (kind == T3_OUT_BF16) ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || (cols * esize) % 16 != 0) return false;
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * esize)};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map,
                  kind == T3_OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  kind == T3_OUT_BF16 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) std::memset(map, 0, sizeof(*map));
  return r == CUDA_SUCCESS;
}

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = 2147483647LL;           // TMA coordinates are int32
constexpr int64_t kMaxTernaryReduction = 16777215;  // 128 * K <= INT32_MAX
constexpr int64_t kMaxInt8Reduction = 131071;       // 16384 * M <= INT32_MAX
// What splitting a pair pipeline's last wave costs, in stages of one pair
// (~0.7 us each), fitted to measurements: the split kernel runs ~5 % slower
// per stage than the whole-tile one, and each piece ends in an accumulator
// flush that adds rather than stores, which short pieces cannot hide.  The
// zeroing grid and the dependent launch before it cost nothing measurable.
constexpr int64_t kSplitCostStages = 8;
constexpr int64_t kSmallM = 32;                     // forward rows served by the small-M path
constexpr int64_t kGemvM = 8;                       // of those, at most the rows the CUDA cores serve
constexpr int64_t kGemvSmallBytes = 4 << 20;        // packed weights up to which they serve 3..8 rows

struct DeviceInfo {
  bool ready = false;
  int status = T3_OK;
  int sms = 0;
  int* err_word = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

int device_info(const DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return T3_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return T3_EDEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return T3_ECUDA;
    if (major != 10 || minor != 3) {
      d.status = T3_EDEVICE;  // built for sm_103a only
    } else if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err_word), g_error_word) !=
               cudaSuccess) {
      return T3_ECUDA;
    }
    d.ready = true;
  }
  *out = &d;
  return d.status;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// One CTA waits on a barrier that nothing completes, with the pipelines' wait
// (suspend hints, abort flag, error word) but a limit of limit_ns: it must
// give up, record (10 << 8) | 2 in the error word and return.
__global__ void wait_selftest_kernel(int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait_limit(&bar, 0, &abort_flag, err, (10 << 8) | 2, limit_ns);
}

// The CTA-pair pipeline for the forward (OP = kOpFwd: act = A [M][K], weights
// packed along K) or dX (act = dY [M][N], reduction N), for operands of any
// alignment.  A scaled output kind needs bulk stores and the reduction in one
// exact chunk: otherwise it returns T3_EINVAL without launching, and the
// caller computes the exact int32 product and then t3_dequant_i32.
template <int OP>
int run_tc2(const int8_t* act, const uint8_t* Wp, void* out, int64_t M, int64_t N, int64_t K,
            cudaStream_t stream, int out_kind = tc2::kOutI32, const float* row_scale = nullptr,
            const float* col_scale = nullptr) {
  const DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != T3_OK) return st;
  const int64_t KB = (K + 3) / 4;
  const int64_t act_cols = (OP == kOpFwd) ? K : N;
  const int64_t out_cols = (OP == kOpFwd) ? N : K;
  CUtensorMap ma, mw, mo;
  // Operands TMA cannot address (row strides or bases not 16-byte aligned)
  // are loaded by their converters from global memory instead; an int32
  // output that cannot take bulk stores is written with plain stores.
  const bool a_ok = make_u8_map_tiled(&ma, act, M, act_cols, act_cols, 128, tc2::BK, true);
  const bool w_ok = (OP == kOpFwd)
                        ? make_u8_map_tiled(&mw, Wp, N, KB, KB, tc2::BNH, tc2::BK / 4)
                        : make_u8_map_tiled(&mw, Wp, N, KB, KB, tc2::BK, tc2::BN / 4);
  const bool out_ok = make_out_map(&mo, out, M, out_cols, out_kind);
  if (!out_ok && out_kind != tc2::kOutI32) return T3_EINVAL;  // scaled output needs bulk stores
  if (!a_ok) ma = w_ok ? mw : mo;  // unused copies: any initialised map
  if (!w_ok) mw = ma;
  if (out_kind != tc2::kOutI32 && ceil_div(act_cols, tc2::BK) > tc2::kChunkStages) return T3_EINVAL;
  tc2::Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.out_rows = M;
  p.out_cols = out_cols;
  p.num_stages = ceil_div(act_cols, tc2::BK);
  const int64_t tiles_r = ceil_div(M, tc2::BMP), tiles_c = ceil_div(out_cols, tc2::BN);
  if (tiles_r * tiles_c > kMaxDim) return T3_EINVAL;
  p.tiles_r = static_cast<int>(tiles_r);
  p.tiles_c = static_cast<int>(tiles_c);
  p.out = static_cast<int32_t*>(out);
  p.use_tma_out = out_ok ? 1 : 0;
  p.out_kind = out_kind;
  p.row_scale = row_scale;
  p.col_scale = col_scale;
  p.wp = Wp;
  p.kb_bytes = KB;
  p.w_tma = w_ok ? 1 : 0;
  p.w_vec4 = (KB % 4 == 0) && (reinterpret_cast<uintptr_t>(Wp) % 4 == 0);
  p.act = act;
  p.act_rows = M;
  p.act_cols = act_cols;
  p.act_vec4 = (act_cols % 4 == 0) && (reinterpret_cast<uintptr_t>(act) % 4 == 0);
  p.a_tma = a_ok ? 1 : 0;
  // the weights-from-global instantiation loads whole words only
  p.mode = (a_ok && w_ok) ? tc2::kModeTma
           : (a_ok && p.w_vec4) ? tc2::kModeWGlobal
                                : tc2::kModeAGlobal;
  p.err = dev->err_word;
  // Schedule.  Whole tiles dealt round-robin keep the busiest pair busy for
  // ceil(T / P) tiles of S stages.  Dealing only the full waves that way and
  // splitting the stages of the remaining tiles evenly over all pairs
  // (stream-K) takes floor(T / P) tiles plus ceil(rem * S / P) stages, and
  // costs the zeroing of those tiles' rows and one more partial-tile flush
  // per pair, counted as kSplitCostStages.  A scaled epilogue needs a tile's
  // whole sum, so it keeps whole tiles, and so do the global-load modes.
  const int64_t num_tiles = tiles_r * tiles_c;
  const int64_t max_pairs = std::max(dev->sms / 2, 1);
  const int64_t waves = num_tiles / max_pairs, rem = num_tiles % max_pairs;
  int64_t dp_tiles = num_tiles;
  if (out_kind == tc2::kOutI32 && p.mode == tc2::kModeTma && rem != 0) {
    const int64_t t_whole = (waves + 1) * p.num_stages;
    const int64_t t_split =
        (waves * p.num_stages + ceil_div(rem * p.num_stages, max_pairs)) * 21 / 20 +
        kSplitCostStages;
    if (t_split < t_whole) dp_tiles = waves * max_pairs;
  }
  p.dp_tiles = static_cast<int>(dp_tiles);
  const bool split = dp_tiles < num_tiles;
  if (split) {
    // the split kernel's attributes first, so that a failure there leaves the
    // output untouched
    st = (OP == kOpFwd) ? prepare_tc2_fwd() : prepare_tc2_dx();
    if (st != T3_OK) return st;
    // from the first tile row that holds a split tile to the end
    const int64_t row0 = (dp_tiles / tiles_c) * tc2::BMP;
    st = launch_zero_pdl(static_cast<int32_t*>(out) + row0 * out_cols, (M - row0) * out_cols,
                         dev->sms, stream);
    if (st != T3_OK) return st;
  }
  const int64_t pairs = split ? max_pairs : std::min(num_tiles, max_pairs);
  const int grid = static_cast<int>(2 * pairs);
  return (OP == kOpFwd) ? launch_tc2_fwd(p, ma, mw, mo, grid, stream)
                        : launch_tc2_dx(p, ma, mw, mo, grid, stream);
}

// The CTA-pair dW pipeline, for operands and output of any alignment.
int run_dw2(const int8_t* A, const int8_t* dY, int32_t* dW, int64_t M, int64_t N, int64_t K,
            cudaStream_t stream) {
  const DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != T3_OK) return st;
  CUtensorMap ma, mdy, mo;
  // operands TMA cannot address are loaded by the converters themselves, and
  // a dW that cannot take bulk adds gets per-element atomic adds
  const bool a_ok = make_u8_map_tiled(&ma, A, M, K, K, dw2::BK, 128);
  const bool dy_ok = make_u8_map_tiled(&mdy, dY, M, N, N, dw2::BK, 128);
  const bool out_ok = make_i32_map_tiled(&mo, dW, K, N, 128, 32, true);
  if (!a_ok) ma = dy_ok ? mdy : mo;  // unused copies: any initialised map
  if (!dy_ok) mdy = ma;
  if (!out_ok) mo = ma;
  dw2::Params p{};
  p.a = A;
  p.dy = dY;
  p.a_vec4 = (K % 4 == 0) && (reinterpret_cast<uintptr_t>(A) % 4 == 0);
  p.dy_vec4 = (N % 4 == 0) && (reinterpret_cast<uintptr_t>(dY) % 4 == 0);
  p.out = dW;
  p.use_tma_out = out_ok ? 1 : 0;
  p.global_ops = (a_ok && dy_ok) ? 0 : 1;
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_stages = ceil_div(M, dw2::BK);
  const int64_t tiles_r = ceil_div(K, dw2::BMP), tiles_c = ceil_div(N, dw2::BN);
  if (tiles_r * tiles_c > kMaxDim) return T3_EINVAL;
  p.tiles_r = static_cast<int>(tiles_r);
  p.tiles_c = static_cast<int>(tiles_c);
  p.num_chunks = static_cast<int>(ceil_div(M, dw2::kChunkElems));
  p.err = dev->err_word;
  // (tile, chunk) units, dealt evenly to at most one pair per two SMs
  const int64_t units = tiles_r * tiles_c * p.num_chunks;
  const int64_t pairs = std::min<int64_t>(units, std::max(dev->sms / 2, 1));
  st = launch_zero_pdl(dW, K * N, dev->sms, stream);
  if (st != T3_OK) return st;
  return launch_dw2(p, ma, mdy, mo, static_cast<int>(2 * pairs), stream);
}

bool valid_out_kind(int kind) {
  return kind == T3_OUT_F32 || kind == T3_OUT_BF16 || kind == T3_OUT_F32_ADD;
}

// The scaled products where the pair pipeline cannot scale in its epilogue:
// the exact int32 product into `workspace` (or, for float output without
// accumulation, into the output buffer itself, converted in place), then
// the dequantization.  bf16 and "+=" outputs need the workspace.
template <class Product>
int scaled_two_pass(Product product, void* out, int64_t rows, int64_t cols, const float* row_scale,
                    const float* col_scale, int kind, int32_t* workspace, cudaStream_t stream) {
  int32_t* x = workspace ? workspace : (kind == T3_OUT_F32 ? static_cast<int32_t*>(out) : nullptr);
  if (!x) return T3_EINVAL;
  int st = product(x);
  if (st != T3_OK) return st;
  const DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != T3_OK) return st;
  return launch_dequant(x, out, rows, cols, row_scale, col_scale, kind, dev->sms, stream);
}

// Products of at most this many multiply-adds run on the CUDA cores
// (t3_small.cu) when an operand's rows are not 4-byte aligned, and of at most
// an eighth of it otherwise: the CTA-pair pipelines load rows that are not
// even word-aligned byte by byte (the pages' HSLM layers, widths 243 and 729
// at 1782 rows: 15-26 us on the CUDA cores against 21-74 us), while with TMA
// or word loads they stay ahead down to a few 10^7 (the same layers padded to
// 256 and 736: 8.5-14.6 against 13-18 us).  Set with
// t3_set_small_product_limit.
std::atomic<int64_t> g_small_macs{int64_t{1} << 29};

bool small_product(int64_t a, int64_t b, int64_t c, bool aligned) {
  int64_t lim = g_small_macs.load(std::memory_order_relaxed);
  if (aligned) lim /= 8;
  return static_cast<__int128>(a) * b * c <= static_cast<__int128>(lim);
}

// Rows of `len` bytes from `base`, every one starting on a 4-byte boundary.
bool word_rows(const void* base, int64_t len) {
  return len % 4 == 0 && reinterpret_cast<uintptr_t>(base) % 4 == 0;
}

int run_small(int op, const int8_t* x, const int8_t* y, const uint8_t* wp, int32_t* out, int64_t M,
              int64_t N, int64_t K, cudaStream_t stream) {
  const DeviceInfo* dev = nullptr;
  const int st = device_info(&dev);
  if (st != T3_OK) return st;
  return launch_small(op, x, y, wp, out, M, N, K, dev->sms, stream);
}

bool bad_dims(int64_t M, int64_t N, int64_t K) {
  return M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim;
}

// Empty reduction: the output is all zeros.
int zero_fill(int32_t* out, int64_t rows, int64_t cols, cudaStream_t s) {
  if (!out) return T3_EINVAL;
  return cudaMemsetAsync(out, 0, static_cast<size_t>(rows) * cols * sizeof(int32_t), s) ==
                 cudaSuccess
             ? T3_OK
             : T3_ECUDA;
}

}  // namespace
}  // namespace t3

using namespace t3;

extern "C" {

int t3_pack_ternary(const int8_t* w, uint8_t* wp, int64_t K, int64_t N) {
  if (K < 0 || N < 0) return T3_EINVAL;
  if (K == 0 || N == 0) return T3_OK;
  if (!w || !wp) return T3_EINVAL;
  const int64_t total = K * N;
  for (int64_t i = 0; i < total; ++i)
    if (w[i] < -1 || w[i] > 1) return T3_EVALUE;
  const int64_t KB = (K + 3) / 4;
  for (int64_t kb = 0; kb < KB; ++kb) {
    const int64_t k0 = 4 * kb;
    const int nk = static_cast<int>(K - k0 < 4 ? K - k0 : 4);
    for (int64_t n = 0; n < N; ++n) {
      uint32_t byte = 0;
      for (int j = 0; j < nk; ++j) {
        const int8_t v = w[(k0 + j) * N + n];
        const uint32_t code = v == 1 ? 1u : (v == -1 ? 2u : 0u);
        byte |= code << (2 * j);
      }
      wp[n * KB + kb] = static_cast<uint8_t>(byte);
    }
  }
  return T3_OK;
}

int t3_gemm_fwd(const int8_t* A, const uint8_t* Wp, int32_t* C, int64_t M, int64_t N, int64_t K,
                t3_stream_t stream) {
  if (bad_dims(M, N, K)) return T3_EINVAL;
  if (M == 0 || N == 0) return T3_OK;
  if (K == 0) return zero_fill(C, M, N, stream);
  if (!A || !Wp || !C) return T3_EINVAL;
  if (K > kMaxTernaryReduction) return T3_EOVERFLOW;
  if (M <= kSmallM) {
    const DeviceInfo* dev = nullptr;
    int st = device_info(&dev);
    if (st != T3_OK) return st;
    // the CUDA-core path: one or two rows, or up to eight over few weights
    // (measured: it beats the tensor cores there; the tensor cores win from
    // four rows at N = K = 8192)
    if (M <= 2 || (M <= kGemvM && N * ((K + 3) / 4) <= kGemvSmallBytes)) {
      st = launch_gemv_fwd(A, Wp, C, M, N, K, dev->sms, stream);
      if (st != T3_EINVAL) return st;
    }
    // packed rows the small-M kernel's TMA cannot address: it would load them
    // byte by byte in one warp
    const bool wp_tma =
        ((K + 3) / 4) % 16 == 0 && reinterpret_cast<uintptr_t>(Wp) % 16 == 0;
    if (!wp_tma && small_product(M, N, K, false))
      return run_small(1, A, nullptr, Wp, C, M, N, K, stream);
    return launch_skinny_fwd(A, Wp, C, M, N, K, dev->sms, dev->err_word, stream);
  }
  if (small_product(M, N, K, word_rows(A, K) && word_rows(Wp, (K + 3) / 4)))
    return run_small(1, A, nullptr, Wp, C, M, N, K, stream);
  return run_tc2<kOpFwd>(A, Wp, C, M, N, K, stream);
}

int t3_gemm_bwd_dx(const int8_t* dY, const uint8_t* Wp, int32_t* dX, int64_t M, int64_t N,
                   int64_t K, t3_stream_t stream) {
  if (bad_dims(M, N, K)) return T3_EINVAL;
  if (M == 0 || K == 0) return T3_OK;
  if (N == 0) return zero_fill(dX, M, K, stream);
  if (!dY || !Wp || !dX) return T3_EINVAL;
  if (N > kMaxTernaryReduction) return T3_EOVERFLOW;
  if (small_product(M, N, K, word_rows(dY, N) && word_rows(Wp, (K + 3) / 4)))
    return run_small(2, dY, nullptr, Wp, dX, M, N, K, stream);
  return run_tc2<kOpDx>(dY, Wp, dX, M, N, K, stream);
}

int t3_gemm_bwd_dw(const int8_t* A, const int8_t* dY, int32_t* dW, int64_t M, int64_t N,
                   int64_t K, t3_stream_t stream) {
  if (bad_dims(M, N, K)) return T3_EINVAL;
  if (K == 0 || N == 0) return T3_OK;
  if (M == 0) return zero_fill(dW, K, N, stream);
  if (!A || !dY || !dW) return T3_EINVAL;
  if (M > kMaxInt8Reduction) return T3_EOVERFLOW;
  if (small_product(M, N, K, word_rows(A, K) && word_rows(dY, N)))
    return run_small(3, A, dY, nullptr, dW, M, N, K, stream);
  return run_dw2(A, dY, dW, M, N, K, stream);
}

int t3_pack_ternary_device(const int8_t* w, uint8_t* wp, int64_t K, int64_t N,
                           t3_stream_t stream) {
  if (K < 0 || N < 0 || K > kMaxDim || N > kMaxDim) return T3_EINVAL;
  if (K == 0 || N == 0) return T3_OK;
  if (!w || !wp) return T3_EINVAL;
  const DeviceInfo* dev = nullptr;
  const int st = device_info(&dev);
  if (st != T3_OK) return st;
  return launch_pack_device(w, wp, K, N, dev->sms, dev->err_word, stream);
}

int t3_quantize_rows_bf16(const void* x, int8_t* q, float* row_scale, int64_t M, int64_t K,
                          t3_stream_t stream) {
  if (M < 0 || K < 0 || M > kMaxDim || K > kMaxDim) return T3_EINVAL;
  if (M == 0) return T3_OK;
  if (!row_scale || (K > 0 && (!x || !q))) return T3_EINVAL;
  const DeviceInfo* dev = nullptr;
  const int st = device_info(&dev);
  if (st != T3_OK) return st;
  return launch_quant_rows(x, q, row_scale, M, K, dev->sms, stream);
}

int t3_dequant_i32(const int32_t* x, void* out, int64_t rows, int64_t cols,
                   const float* row_scale, const float* col_scale, int out_kind,
                   t3_stream_t stream) {
  if (rows < 0 || cols < 0 || !valid_out_kind(out_kind)) return T3_EINVAL;
  if (rows == 0 || cols == 0) return T3_OK;
  if (!x || !out) return T3_EINVAL;
  if (out_kind != T3_OUT_F32 && static_cast<const void*>(x) == out) return T3_EINVAL;
  const DeviceInfo* dev = nullptr;
  const int st = device_info(&dev);
  if (st != T3_OK) return st;
  return launch_dequant(x, out, rows, cols, row_scale, col_scale, out_kind, dev->sms, stream);
}

int t3_gemm_fwd_scaled(const int8_t* A, const uint8_t* Wp, void* C, int64_t M, int64_t N,
                       int64_t K, const float* row_scale, const float* col_scale, int out_kind,
                       int32_t* workspace, t3_stream_t stream) {
  if (bad_dims(M, N, K) || !valid_out_kind(out_kind)) return T3_EINVAL;
  if (M == 0 || N == 0) return T3_OK;
  if (!C) return T3_EINVAL;
  if (K > 0 && (!A || !Wp)) return T3_EINVAL;
  if (K > kMaxTernaryReduction) return T3_EOVERFLOW;
  if (M > kSmallM && K > 0) {
    const int st = run_tc2<kOpFwd>(A, Wp, C, M, N, K, stream, out_kind, row_scale, col_scale);
    if (st != T3_EINVAL) return st;
  }
  return scaled_two_pass(
      [&](int32_t* x) { return t3_gemm_fwd(A, Wp, x, M, N, K, stream); }, C, M, N, row_scale,
      col_scale, out_kind, workspace, stream);
}

int t3_gemm_bwd_dx_scaled(const int8_t* dY, const uint8_t* Wp, void* dX, int64_t M, int64_t N,
                          int64_t K, const float* row_scale, const float* col_scale, int out_kind,
                          int32_t* workspace, t3_stream_t stream) {
  if (bad_dims(M, N, K) || !valid_out_kind(out_kind)) return T3_EINVAL;
  if (M == 0 || K == 0) return T3_OK;
  if (!dX) return T3_EINVAL;
  if (N > 0 && (!dY || !Wp)) return T3_EINVAL;
  if (N > kMaxTernaryReduction) return T3_EOVERFLOW;
  if (N > 0) {
    const int st = run_tc2<kOpDx>(dY, Wp, dX, M, N, K, stream, out_kind, row_scale, col_scale);
    if (st != T3_EINVAL) return st;
  }
  return scaled_two_pass(
      [&](int32_t* x) { return t3_gemm_bwd_dx(dY, Wp, x, M, N, K, stream); }, dX, M, K,
      row_scale, col_scale, out_kind, workspace, stream);
}

int t3_gemm_bwd_dw_scaled(const int8_t* A, const int8_t* dY, void* dW, int64_t M, int64_t N,
                          int64_t K, const float* row_scale, const float* col_scale, int out_kind,
                          int32_t* workspace, t3_stream_t stream) {
  if (bad_dims(M, N, K) || !valid_out_kind(out_kind)) return T3_EINVAL;
  if (K == 0 || N == 0) return T3_OK;
  if (!dW) return T3_EINVAL;
  if (M > 0 && (!A || !dY)) return T3_EINVAL;
  if (M > kMaxInt8Reduction) return T3_EOVERFLOW;
  return scaled_two_pass(
      [&](int32_t* x) { return t3_gemm_bwd_dw(A, dY, x, M, N, K, stream); }, dW, K, N, row_scale,
      col_scale, out_kind, workspace, stream);
}

int64_t t3_set_small_product_limit(int64_t macs) {
  return g_small_macs.exchange(macs < 0 ? 0 : macs);
}

}  // extern "C"

extern "C" {

const char* t3_status_string(int status) {
  switch (status) {
    case T3_OK: return "T3_OK: success";
    case T3_EINVAL: return "T3_EINVAL: null pointer or invalid size";
    case T3_EVALUE: return "T3_EVALUE: weight outside {-1, 0, +1}";
    case T3_EOVERFLOW: return "T3_EOVERFLOW: reduction too long for an exact int32 result";
    case T3_ECUDA: return "T3_ECUDA: a CUDA call failed";
    case T3_ETIMEOUT: return "T3_ETIMEOUT: a bounded device wait gave up";
    case T3_EDEVICE: return "T3_EDEVICE: no usable sm_103 device";
    default: return "unknown t3 status";
  }
}

int t3_last_device_error(t3_stream_t stream, int32_t* detail) {
  if (detail) *detail = 0;
  const DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != T3_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return T3_ECUDA;
  int value = 0;
  if (cudaMemcpy(&value, dev->err_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return T3_ECUDA;
  if (value != 0) {
    const int zero = 0;
    if (cudaMemcpy(dev->err_word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return T3_ECUDA;
  }
  if (detail) *detail = value;
  if (value == 0) return T3_OK;
  return (value & 0xFF) == 6 ? T3_EVALUE : T3_ETIMEOUT;  // role 6: an invalid input value
}

int t3_gemm_fwd_bf16(const void* X, const uint8_t* Wp, int32_t* C, float* row_scale,
                     float* row_inv, int64_t M, int64_t N, int64_t K, t3_stream_t stream) {
  if (bad_dims(M, N, K)) return T3_EINVAL;
  if (M == 0) return T3_OK;
  if (!row_scale || !row_inv || (K > 0 && !X)) return T3_EINVAL;
  if (K > kMaxTernaryReduction) return T3_EOVERFLOW;
  // the fused kernel's shapes, checked before any CUDA call
  if (N > 0 && K > 0 &&
      (M <= kSmallM || K % 64 != 0 || reinterpret_cast<uintptr_t>(X) % 16 != 0 ||
       reinterpret_cast<uintptr_t>(Wp) % 16 != 0))
    return T3_EINVAL;
  const DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != T3_OK) return st;
  if (K == 0) {  // zero rows: scales 0, and the empty reduction writes zeros
    if (cudaMemsetAsync(row_scale, 0, M * sizeof(float), stream) != cudaSuccess ||
        cudaMemsetAsync(row_inv, 0, M * sizeof(float), stream) != cudaSuccess)
      return T3_ECUDA;
    return N == 0 ? T3_OK : zero_fill(C, M, N, stream);
  }
  if (N > 0 && (!Wp || !C)) return T3_EINVAL;
  // the fused kernel's shapes: checked before anything is launched
  const int64_t KB = (K + 3) / 4;
  CUtensorMap ma, mw, mo;
  if (N > 0) {
    if (!make_u16_map_tiled(&ma, X, M, K, 128, tc2::BK / 2)) return T3_EINVAL;
    if (!make_u8_map_tiled(&mw, Wp, N, KB, KB, tc2::BNH, tc2::BK / 4)) return T3_EINVAL;
    if (!make_out_map(&mo, C, M, N, tc2::kOutI32)) mo = mw;  // plain stores
  }
  st = launch_row_scales(X, row_scale, row_inv, M, K, dev->sms, stream);
  if (st != T3_OK || N == 0) return st;
  tc2::Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.out_rows = M;
  p.out_cols = N;
  p.num_stages = ceil_div(K, tc2::BK);
  const int64_t tiles_r = ceil_div(M, tc2::BMP), tiles_c = ceil_div(N, tc2::BN);
  if (tiles_r * tiles_c > kMaxDim) return T3_EINVAL;
  p.tiles_r = static_cast<int>(tiles_r);
  p.tiles_c = static_cast<int>(tiles_c);
  p.out = C;
  p.use_tma_out = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && (N * 4) % 16 == 0) ? 1 : 0;
  p.out_kind = tc2::kOutI32;
  p.wp = Wp;
  p.kb_bytes = KB;
  p.w_tma = 1;
  p.w_vec4 = 1;
  p.act = nullptr;
  p.act_rows = M;
  p.act_cols = K;
  p.a_tma = 1;
  p.mode = tc2::kModeBf16;
  p.dp_tiles = static_cast<int>(tiles_r * tiles_c);
  p.row_inv = row_inv;
  p.err = dev->err_word;
  const int64_t pairs = std::min<int64_t>(tiles_r * tiles_c, std::max(dev->sms / 2, 1));
  return launch_tc2_fwd_bf16(p, ma, mw, mo, static_cast<int>(2 * pairs), stream);
}

int t3_selftest_wait_timeout(int64_t limit_ns, t3_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > static_cast<int64_t>(kWaitLimitNs)) return T3_EINVAL;
  const DeviceInfo* dev = nullptr;
  const int st = device_info(&dev);
  if (st != T3_OK) return st;
  wait_selftest_kernel<<<1, 32, 0, stream>>>(dev->err_word, static_cast<uint64_t>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? T3_OK : T3_ECUDA;
}

int t3_version(void) { return 200; }

}  // extern "C"
