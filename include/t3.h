/*
 * t3.h -- C ABI of the ternary-weight x int8 GEMM library for GB300 (sm_103a).
 *
 * Three integer products of a ternary-weight layer and the packer of its
 * weights.  All results are exact int32; there is no rounding, no scale and no
 * tolerance on this path.
 *
 * Sources (web pages, cited by title and section):
 *   [fwd] "t27c PTX backend: ternary x int8 GEMM kernel emitted by a .t27 spec
 *         (int8 mma.sync), ptx-run glue", section "What this adds": C = A x W
 *         with int8 A and ternary W held as 2-bit codes, each decoded as
 *         (c & 1) - ((c >> 1) & 1), i.e. 0 -> 0, 1 -> +1, 2 -> -1, 3 -> 0.
 *   [bwd] "spec(igla): hslm_bwd_ptx -- HSLM backward dX and dW as int8
 *         tensor-core PTX written by t27", kernel 1 (dX = dY x W^T, W ternary
 *         in the same code layout) and kernel 2 (dW = X^T x dY summed over
 *         rows, int32 accumulation, reduction length <= 131071).
 *
 * Layouts (all row-major and densely packed, no row padding):
 *   A  int8  [M][K]          activations
 *   Wp uint8 [N][ceil(K/4)]  packed weights: the code of W[k][n] is at bits
 *                            2*(k%4) of byte k/4 of row n; positions k >= K of
 *                            the last byte of a row are ignored by every call.
 *   C  int32 [M][N]          forward output
 *   dY int8  [M][N]          output gradient
 *   dX int32 [M][K]          input gradient
 *   dW int32 [K][N]          weight gradient
 *
 * Ownership and threading:
 *   - The caller owns every buffer.  The GEMM calls take DEVICE pointers (any
 *     memory the current device can read/write), enqueue their work on
 *     `stream` and return without waiting; the results are ready once the
 *     stream reaches that point.  The library allocates no device memory per
 *     call.
 *   - Outputs are overwritten, never accumulated into.
 *   - A call whose output is empty (no rows or no columns) does nothing and
 *     returns T3_OK.  A call whose reduction is empty (K = 0 for the forward,
 *     N = 0 for dX, M = 0 for dW) writes zeros to its output.
 *   - Argument errors are reported before anything is launched; nothing is
 *     written then.  After T3_ECUDA (a launch or attribute call failed) the
 *     contents of the output are undefined: a call that queues a zeroing
 *     kernel before its product may have queued it already.  No C++
 *     exception crosses this interface and the device code never traps.
 *   - Calls may be made from several host threads; each call is independent.
 *   - Per-device state (the device error word's address, kernel attributes,
 *     the no-alloc buffer's address) is resolved once per device and process.
 *     It does not survive cudaDeviceReset: do not call the library on a device
 *     again in a process that reset it.
 */
#ifndef T3_H_
#define T3_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (the same type as cudaStream_t / CUstream); NULL is the
 * legacy default stream. */
typedef struct CUstream_st* t3_stream_t;

typedef enum {
  T3_OK = 0,
  T3_EINVAL = -1,     /* null pointer with a non-empty shape, negative size   */
  T3_EVALUE = -2,     /* t3_pack_ternary: a weight outside {-1, 0, +1}        */
  T3_EOVERFLOW = -3,  /* a reduction too long for an exact int32 result       */
  T3_ECUDA = -4,      /* a CUDA runtime/driver call failed (launch, attribute) */
  T3_ETIMEOUT = -5,   /* a bounded device-side wait gave up (see below)       */
  T3_EDEVICE = -6     /* no usable sm_103 device for this call               */
} t3_status;

/*
 * t3_pack_ternary -- [fwd] "What this adds" (the 2-bit weight codes).
 *   w   HOST int8 [K][N], every value in {-1, 0, +1} (W as it appears in A x W)
 *   wp  HOST uint8 [N][ceil(K/4)], written in full: code 1 for +1, 2 for -1,
 *       0 for 0 and for the pad positions k >= K.
 * Synchronous, host memory only.  Returns T3_EVALUE and writes nothing when a
 * value is outside {-1, 0, +1}; T3_EINVAL for negative sizes or null pointers.
 */
int t3_pack_ternary(const int8_t* w, uint8_t* wp, int64_t K, int64_t N);

/*
 * t3_pack_ternary_device -- the same packing as t3_pack_ternary, on the device.
 *   w   DEVICE int8 [K][N]; wp DEVICE uint8 [N][ceil(K/4)], written in full
 *       (pad codes 0).  Both are owned by the caller.
 * Asynchronous on `stream`.  A value outside {-1, 0, +1} packs as code 0 and
 * records (9 << 8) | 6 in the device error word: t3_last_device_error then
 * returns T3_EVALUE.  Returns T3_EINVAL, without launching, for negative
 * sizes, null pointers (with K, N > 0) or sizes above 2^31 - 1; K or N = 0 is
 * a no-op.  Training changes W every step: this keeps the packing on the GPU.
 */
int t3_pack_ternary_device(const int8_t* w, uint8_t* wp, int64_t K, int64_t N,
                           t3_stream_t stream);

/*
 * t3_gemm_fwd -- [fwd]: C[m][n] = sum_{k<K} A[m][k] * W[k][n].
 *   A [M][K], Wp [N][ceil(K/4)], C [M][N] (layouts above), device pointers.
 * Exact for every input when K <= 16777215 (|A W| <= 128 K fits int32);
 * larger K returns T3_EOVERFLOW.  M <= 32 takes the small-M path, which is
 * bound by reading the packed weights: one or two rows (and up to eight when
 * Wp is at most 4 MB) run on the CUDA cores (byte-permute decode, dp4a), the
 * rest on the tensor cores.  Either way it enqueues one kernel on `stream` as
 * a programmatic dependent of the work before it, so that its launch and set-
 * up overlap that work's end; it reads A and Wp and writes C only after all
 * earlier work on `stream` has completed.
 * For M > 32, when whole output tiles would leave most of the GPU idle over a
 * long reduction (few tiles, many reduction stages) and A and Wp are
 * TMA-addressable, the reduction of the last tiles is split over the whole
 * GPU: the call then enqueues the same pair of kernels, the first zeroing the
 * rows of C that the split part adds into.
 * Small products (M*N*K at most the limit of t3_set_small_product_limit,
 * 2^29 by default, when a row stride or base of A or Wp is not a multiple of
 * 4 bytes, else at most an eighth of it; for M <= 32 only when Wp's rows are
 * not 16-byte multiples on a 16-byte boundary)
 * run on the CUDA cores instead: 64 x 64 output tiles, the reduction split
 * over CTAs that add atomically onto a zeroed C when the tiles are few (a
 * cudaMemsetAsync and one kernel, both on `stream`, in stream order), any
 * alignment of A, Wp and C.
 */
int t3_gemm_fwd(const int8_t* A, const uint8_t* Wp, int32_t* C, int64_t M, int64_t N,
                int64_t K, t3_stream_t stream);

/*
 * t3_gemm_bwd_dx -- [bwd] kernel 1: dX[m][k] = sum_{n<N} dY[m][n] * W[k][n].
 *   dY [M][N], Wp [N][ceil(K/4)] (the forward's packed weights), dX [M][K].
 * Exact for every input when N <= 16777215; larger N returns T3_EOVERFLOW.
 * Long reductions over few output tiles are split as in t3_gemm_fwd (M > 32),
 * with a zeroing kernel before the product.  Small products run on the CUDA
 * cores as in t3_gemm_fwd.
 */
int t3_gemm_bwd_dx(const int8_t* dY, const uint8_t* Wp, int32_t* dX, int64_t M, int64_t N,
                   int64_t K, t3_stream_t stream);

/*
 * t3_gemm_bwd_dw -- [bwd] kernel 2: dW[k][n] = sum_{m<M} A[m][k] * dY[m][n].
 *   A [M][K], dY [M][N], dW [K][N].
 * int8 x int8 products reach 16384, so the reduction is exact in int32 only
 * for M <= 131071 (the pages' bound); larger M returns T3_EOVERFLOW.
 * It enqueues two kernels on `stream`: one that zeroes dW and one that adds
 * 1024-row partial sums into it; the second may start before the first ends
 * (programmatic dependent launch) but touches dW only after it, and the first
 * touches dW only after all earlier work on `stream`.  Small products run on
 * the CUDA cores as in t3_gemm_fwd.
 */
int t3_gemm_bwd_dw(const int8_t* A, const int8_t* dY, int32_t* dW, int64_t M, int64_t N,
                   int64_t K, t3_stream_t stream);

/*
 * t3_quantize_rows_bf16 -- the step before the products: bf16 activations to
 * int8 with one scale per row.  The second page feeds its int8 kernels from
 * quantized tensors and names per-row scales for dX but gives no quantizer;
 * this is symmetric absmax per row:
 *   amax = max_k |x[m][k]|, row_scale[m] = amax / 127, inv = 127 / amax
 *   (each a float division rounded to nearest),
 *   q[m][k] = rint(x[m][k] * inv)  (product rounded to a float, then to the
 *   nearest integer, ties to even), clamped to [-127, 127];
 *   a row of zeros gives q = 0 and row_scale = 0.
 *   x DEVICE bf16 [M][K] (bit patterns), q DEVICE int8 [M][K], row_scale
 *   DEVICE float [M]; all owned by the caller.  Finite inputs; a product
 *   0 * inf (amax so small that 127 / amax overflows) counts as 0.
 * Asynchronous on `stream`.  M = 0 is a no-op; K = 0 writes row_scale = 0.
 */
int t3_quantize_rows_bf16(const void* x, int8_t* q, float* row_scale, int64_t M, int64_t K,
                          t3_stream_t stream);

/*
 * t3_gemm_fwd_bf16 -- the row quantizer fused into the forward product: the
 * same result as t3_quantize_rows_bf16(X, q, row_scale) followed by
 * t3_gemm_fwd(q, Wp, C), without writing q.  A first kernel takes each row's
 * absolute maximum and writes
 *   row_scale[m] = amax / 127 and row_inv[m] = 127 / amax   (0 and 0 for a
 *   zero row; the divisions of t3_quantize_rows_bf16),
 * then the forward pair pipeline reads X as bf16 tiles and its converters
 * quantize them (q = rint(x * row_inv[m]), ties to even) on their way to the
 * tensor core:
 *   C[m][n] = sum_k q[m][k] * W[k][n]     (exact int32, as t3_gemm_fwd).
 *   X DEVICE bf16 [M][K] (bit patterns), Wp DEVICE [N][ceil(K/4)], C DEVICE
 *   int32 [M][N], row_scale and row_inv DEVICE float [M]; caller-owned.
 * The fused kernel takes M > 32, K a multiple of 64 and X, Wp 16-byte aligned
 * (bf16 and packed rows TMA can address); any other shape returns T3_EINVAL
 * without launching (quantize, then multiply, instead).  N = 0 computes the
 * scales only; K = 0 writes zero scales and a zero C.  Asynchronous on
 * `stream`.  Finite inputs, as for t3_quantize_rows_bf16.
 */
int t3_gemm_fwd_bf16(const void* X, const uint8_t* Wp, int32_t* C, float* row_scale,
                     float* row_inv, int64_t M, int64_t N, int64_t K, t3_stream_t stream);

/*
 * Scaled outputs -- the step after the products in "spec(igla): hslm_bwd_ptx
 * -- HSLM backward dX and dW as int8 tensor-core PTX written by t27": the
 * host rescales the integer results (dX by a scale per row; dW by scales per
 * column of X and of dY, i.e. per row and per column of dW), and the products
 * also have "+=" forms.  For an exact int32 result x[r][c]:
 *   y = ((float)x * row_scale[r]) * col_scale[c]
 * with each conversion and product rounded to the nearest float (ties to
 * even); a NULL scale vector stands for ones.  The output kind decides what
 * is written: T3_OUT_F32 stores y (float), T3_OUT_BF16 stores y rounded to
 * bf16 (nearest, ties to even), T3_OUT_F32_ADD sets out = out + y (float, one
 * rounding).  Scale vectors are device float arrays, owned by the caller.
 */
enum { T3_OUT_F32 = 0, T3_OUT_BF16 = 1, T3_OUT_F32_ADD = 2 };

/*
 * t3_dequant_i32 -- out[r][c] from x [rows][cols] (DEVICE int32) as above;
 *   out DEVICE [rows][cols] float or bf16; row_scale [rows], col_scale [cols].
 * x and out may be the same buffer for T3_OUT_F32 only (else T3_EINVAL).
 * Asynchronous on `stream`; rows or cols = 0 is a no-op.
 */
int t3_dequant_i32(const int32_t* x, void* out, int64_t rows, int64_t cols,
                   const float* row_scale, const float* col_scale, int out_kind,
                   t3_stream_t stream);

/*
 * t3_gemm_fwd_scaled, t3_gemm_bwd_dx_scaled, t3_gemm_bwd_dw_scaled -- the
 * products of t3_gemm_fwd / t3_gemm_bwd_dx / t3_gemm_bwd_dw with the scaled
 * output above, same operands, sizes, validation and overflow rules:
 *   fwd: C [M][N],  row_scale [M], col_scale [N];
 *   dX:  dX [M][K], row_scale [M], col_scale [K];
 *   dW:  dW [K][N], row_scale [K] (X's column scales), col_scale [N] (dY's).
 * The forward (M > 32) and dX apply the scales in the epilogue of their
 * pair pipeline when the reduction is at most 65536 long and the output rows
 * are 16-byte aligned; otherwise, and always for dW, they compute the exact
 * int32 product first and then run t3_dequant_i32.  That product goes to
 * `workspace` (DEVICE int32 with the output's rows x cols, caller-owned) or,
 * for T3_OUT_F32 when `workspace` is NULL, into the output buffer, converted
 * in place; T3_OUT_BF16 and T3_OUT_F32_ADD return T3_EINVAL there without a
 * workspace.  The result is the same on every path.
 */
int t3_gemm_fwd_scaled(const int8_t* A, const uint8_t* Wp, void* C, int64_t M, int64_t N,
                       int64_t K, const float* row_scale, const float* col_scale, int out_kind,
                       int32_t* workspace, t3_stream_t stream);
int t3_gemm_bwd_dx_scaled(const int8_t* dY, const uint8_t* Wp, void* dX, int64_t M, int64_t N,
                          int64_t K, const float* row_scale, const float* col_scale, int out_kind,
                          int32_t* workspace, t3_stream_t stream);
int t3_gemm_bwd_dw_scaled(const int8_t* A, const int8_t* dY, void* dW, int64_t M, int64_t N,
                          int64_t K, const float* row_scale, const float* col_scale, int out_kind,
                          int32_t* workspace, t3_stream_t stream);

/*
 * t3_gemm_bwd_dw_scaled_noalloc -- t3_gemm_bwd_dw_scaled whose int32
 * intermediate lives in a fixed buffer inside the library instead of a
 * caller workspace, so that neither the call nor the caller allocates device
 * memory for it.  The pages have no counterpart: it serves callers that
 * cannot provide a workspace (bf16 and "+=" outputs need one).
 *   The buffer holds 8,388,608 int32 entries (32 MiB) per device: K * N above
 *   that returns T3_EINVAL before any CUDA call.  Nothing in it has to start
 *   at zero (the dW product writes all of its K x N block first).
 *   Races: every call on a device shares the buffer, so two calls must not
 *   overlap on one device -- not on different streams, and not from several
 *   host threads without ordering; each call's stream order alone protects
 *   only calls on that stream.
 *   The first call on each device resolves the buffer's address
 *   (cudaGetSymbolAddress); make that call outside any stream capture.  The
 *   address, like all per-device state, is not valid after cudaDeviceReset.
 *   Residency: the buffer sits in a module of its own.  With CUDA's lazy
 *   module loading (the default) a device reserves its 32 MiB at the first
 *   call of this function there and keeps it until the process exits; the
 *   other entry points do not load that module.  With eager loading
 *   (CUDA_MODULE_LOADING=EAGER) every device reserves it when the library's
 *   modules load.
 * Arguments, sizes, results and other errors are those of
 * t3_gemm_bwd_dw_scaled.
 */
int t3_gemm_bwd_dw_scaled_noalloc(const int8_t* A, const int8_t* dY, void* dW, int64_t M,
                                  int64_t N, int64_t K, const float* row_scale,
                                  const float* col_scale, int out_kind, t3_stream_t stream);

/* A static, human-readable name for a status code (never NULL). */
const char* t3_status_string(int status);

/*
 * t3_last_device_error -- every pipeline wait inside the kernels is bounded
 * (about two seconds of device time).  A wait that runs out makes its kernel
 * stop early, leaving its output incomplete, and records a code in a
 * per-device error word instead of hanging the GPU.  This call synchronizes
 * `stream`, returns T3_ETIMEOUT if the word is set (T3_OK otherwise) and
 * clears it; T3_EVALUE instead when the code is the device packer's invalid
 * value.  *detail, when not NULL, receives the recorded code (0 if none):
 * bits 0-7 the role (1 producer, 2 converter, 3 MMA issuer, 4 epilogue,
 * 5 pair forwarder gave up; 6 an input value was invalid), bits 8-15 the
 * kernel (4 small-M fwd; 5 fwd, 6 dX, 7 dW on CTA pairs; 9 the device
 * packer; 10 the wait self-test below).
 */
int t3_last_device_error(t3_stream_t stream, int32_t* detail);

/*
 * t3_set_small_product_limit -- the route of t3_gemm_fwd, t3_gemm_bwd_dx and
 * t3_gemm_bwd_dw (and of their scaled forms' int32 pass): products of at most
 * `macs` multiply-adds (M*N*K) run on the CUDA cores when an operand's rows
 * are not 4-byte aligned (stride or base not a multiple of 4 bytes), of at
 * most macs / 8 when they all are; larger ones on the tensor cores.  Default
 * 2^29 (536870912); 0 sends every product to the tensor cores; negative
 * values count as 0.  Process-wide, for every device;
 * a call racing with products on other threads may see either route, and
 * both give the same exact result.  Returns the previous limit.  Host only:
 * no CUDA call, no error.
 */
int64_t t3_set_small_product_limit(int64_t macs);

/*
 * t3_selftest_wait_timeout -- exercises the bounded-wait path above without
 * any fault: one CTA waits on a pipeline barrier that nothing completes, with
 * the kernels' own wait loop but a limit of `limit_ns` nanoseconds of device
 * time instead of two seconds.  The wait gives up, records (10 << 8) | 2 in
 * the error word (unless a code is already there) and the kernel returns, so
 * the next t3_last_device_error reports T3_ETIMEOUT with that detail and the
 * device stays usable.  The pages have no counterpart: this is a check of the
 * library's failure reporting.  limit_ns must lie in [1000, 2e9], else
 * T3_EINVAL; asynchronous on `stream`.
 */
int t3_selftest_wait_timeout(int64_t limit_ns, t3_stream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
int t3_version(void);

#ifdef __cplusplus
}
#endif

#endif /* T3_H_ */
