// t3_noalloc.cu -- t3_gemm_bwd_dw_scaled_noalloc: the scaled dW whose int32
// intermediate lives in a fixed device buffer of the library.  See
// include/t3.h for the contract.
//
// The buffer has a translation unit of its own: with CUDA's lazy module
// loading, a module's device variables are allocated when the module is first
// used on a device, so only a process that calls this entry point (and thereby
// resolves the buffer's address) reserves its 32 MiB; the other entry points
// never touch this module.
#include <atomic>

#include "t3.h"
#include "t3_internal.h"

namespace t3 {
namespace {

// 8 Mi int32 entries (32 MiB) per device, enough for dW up to K * N =
// 8,388,608 (the 1280 x 3456 layer's dW has 4,423,680).  Nothing in it has to
// start at zero: the dW product writes every entry of its K x N block before
// the dequantization reads it.  Every call on a device shares it.
constexpr int64_t kNoAllocWorkspaceEntries = 8LL * 1024 * 1024;
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = 2147483647LL;
std::atomic<int32_t*> g_noalloc_addr[kMaxDevices];  // resolved once per device

}  // namespace

static __device__ __align__(256) int32_t g_noalloc_workspace[kNoAllocWorkspaceEntries];

}  // namespace t3

using namespace t3;

extern "C" int t3_gemm_bwd_dw_scaled_noalloc(const int8_t* A, const int8_t* dY, void* dW,
                                             int64_t M, int64_t N, int64_t K,
                                             const float* row_scale, const float* col_scale,
                                             int out_kind, t3_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return T3_EINVAL;
  if (out_kind != T3_OUT_F32 && out_kind != T3_OUT_BF16 && out_kind != T3_OUT_F32_ADD)
    return T3_EINVAL;
  if (K == 0 || N == 0) return T3_OK;
  if (K * N > kNoAllocWorkspaceEntries) return T3_EINVAL;  // checked before any CUDA call
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return T3_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return T3_EDEVICE;
  int32_t* ws = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (!ws) {
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ws), g_noalloc_workspace) != cudaSuccess)
      return T3_ECUDA;
    g_noalloc_addr[dev].store(ws, std::memory_order_release);
  }
  return t3_gemm_bwd_dw_scaled(A, dY, dW, M, N, K, row_scale, col_scale, out_kind, ws, stream);
}
