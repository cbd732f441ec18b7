/*
 * t3_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * The plain, slow, obviously correct CPU oracle for the ternary-weight x int8
 * GEMMs.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg
 * may load it.  It shares no code, header, table or helper with the CUDA
 * library in ternary_weight_int8_t3_gb300/csrc, and the library never calls it.
 *
 * Sources (web pages; cited by title and section):
 *   [P-fwd] "t27c PTX backend: ternary x int8 GEMM kernel emitted by a .t27 spec
 *           (int8 mma.sync), ptx-run glue" (gHashTag/t27 pull 10425),
 *           section "What this adds": C = A * W with int8 A, ternary W held as
 *           2-bit codes, each code decoded as (c & 1) - ((c >> 1) & 1); the host
 *           CPU reference computes whole rows of C and a mismatch count.
 *   [P-bwd] "spec(igla): hslm_bwd_ptx -- HSLM backward dX and dW as int8
 *           tensor-core PTX written by t27" (gHashTag/t27 pull 10855),
 *           description of kernel 1 (dX = dY x W^T, W ternary, same code
 *           layout) and kernel 2 (dW = X^T x dY summed over rows, int32
 *           accumulation, reduction length <= 131071).
 *
 * Readings where the pages are silent:
 *   - code layout: the code of W[k][n] sits in byte (n * ceil(K/4) + k/4) of Wp,
 *     at bits 2*(k%4); the rows of Wp are n, each ceil(K/4) bytes, no padding.
 *   - the packer takes w as int8 [K][N] row-major and writes code 0 into the pad
 *     positions k >= K of the last byte of each row.
 *   - decoders ignore positions k >= K whatever their bits hold; code 3 is 0.
 *   - outputs are overwritten, not accumulated; every shape >= 1 is legal.
 *
 * Arithmetic: every sum is taken in int64 in the plain definition's order and
 * narrowed to int32 only after checking that it fits.  Nothing is blocked,
 * fused or reordered.  The outer loop is split across OpenMP threads when the
 * compiler supports it; each output element is still one serial int64 sum.
 */
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EVALUE -2      /* w holds a value outside {-1, 0, +1} */
#define ORACLE_EOVERFLOW -3   /* a sum does not fit in int32 */
#define ORACLE_EINVAL -1      /* negative size or null pointer */

/* The decode table, written out from the formula w = (c & 1) - ((c >> 1) & 1)
 * of [P-fwd] "What this adds": c=0 -> 0-0 = 0, c=1 -> 1-0 = +1, c=2 -> 0-1 = -1,
 * c=3 -> 1-1 = 0.  A lookup, not the bit formula, so that the oracle and a
 * bit-trick decoder do not share a mistake. */
static const int ORACLE_DECODE[4] = {0, +1, -1, 0};

int oracle_decode(int code) { return ORACLE_DECODE[code & 3]; }

static int64_t packed_row_bytes(int64_t K) { return (K + 3) / 4; }

/* The 2-bit code of W[k][n] in the packed matrix Wp (rows n, ceil(K/4) bytes). */
static int code_of(const uint8_t* Wp, int64_t K, int64_t n, int64_t k) {
  uint8_t byte = Wp[n * packed_row_bytes(K) + k / 4];
  return (byte >> (2 * (k % 4))) & 3;
}

/* W[k][n] in {-1, 0, +1}. */
static int weight_of(const uint8_t* Wp, int64_t K, int64_t n, int64_t k) {
  return ORACLE_DECODE[code_of(Wp, K, n, k)];
}

/* Packs w (int8 [K][N], values in {-1,0,+1}) into Wp ([N][ceil(K/4)] bytes).
 * The code for +1 is 1 and for -1 is 2, the codes the decode formula maps back
 * to those values; 0 gets code 0, and so do the pad positions.  Returns
 * ORACLE_EVALUE, writing nothing, if any w is outside {-1,0,+1}. */
int oracle_pack(const int8_t* w, uint8_t* Wp, int64_t K, int64_t N) {
  if (K < 0 || N < 0) return ORACLE_EINVAL;
  if (K == 0 || N == 0) return ORACLE_OK;
  if (!w || !Wp) return ORACLE_EINVAL;
  for (int64_t i = 0; i < K * N; ++i)
    if (w[i] != -1 && w[i] != 0 && w[i] != 1) return ORACLE_EVALUE;
  int64_t KB = packed_row_bytes(K);
  for (int64_t i = 0; i < N * KB; ++i) Wp[i] = 0;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      int v = w[k * N + n];
      int code = (v == 1) ? 1 : (v == -1) ? 2 : 0;
      Wp[n * KB + k / 4] |= (uint8_t)(code << (2 * (k % 4)));
    }
  }
  return ORACLE_OK;
}

/* Decodes Wp back to w (int8 [K][N]); positions k >= K are not read. */
int oracle_unpack(const uint8_t* Wp, int8_t* w, int64_t K, int64_t N) {
  if (K < 0 || N < 0) return ORACLE_EINVAL;
  if (K == 0 || N == 0) return ORACLE_OK;
  if (!w || !Wp) return ORACLE_EINVAL;
  for (int64_t k = 0; k < K; ++k)
    for (int64_t n = 0; n < N; ++n) w[k * N + n] = (int8_t)weight_of(Wp, K, n, k);
  return ORACLE_OK;
}

static int fits_i32(int64_t v) { return v >= -2147483647LL - 1 && v <= 2147483647LL; }

/* Forward, [P-fwd]: C[m][n] = sum_{k<K} A[m][k] * W[k][n] for the rows listed
 * in `rows` (all rows when rows == NULL; then nrows must be M).  Output row i
 * of C (N int32) holds row rows[i] of the product. */
int oracle_fwd_rows(const int8_t* A, const uint8_t* Wp, int32_t* C, int64_t M, int64_t N,
                    int64_t K, const int64_t* rows, int64_t nrows) {
  if (M < 0 || N < 0 || K < 0 || nrows < 0) return ORACLE_EINVAL;
  int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = rows ? rows[i] : i;
    if (m < 0 || m >= M) { bad |= 1; continue; }
    for (int64_t n = 0; n < N; ++n) {
      int64_t acc = 0;
      for (int64_t k = 0; k < K; ++k)
        acc += (int64_t)A[m * K + k] * (int64_t)weight_of(Wp, K, n, k);
      if (!fits_i32(acc)) bad |= 2;
      C[i * N + n] = (int32_t)acc;
    }
  }
  if (bad & 1) return ORACLE_EINVAL;
  if (bad & 2) return ORACLE_EOVERFLOW;
  return ORACLE_OK;
}

int oracle_fwd(const int8_t* A, const uint8_t* Wp, int32_t* C, int64_t M, int64_t N, int64_t K) {
  return oracle_fwd_rows(A, Wp, C, M, N, K, NULL, M);
}

/* Backward data, [P-bwd] kernel 1: dX[m][k] = sum_{n<N} dY[m][n] * W[k][n],
 * with the same packed W as the forward.  Rows as in oracle_fwd_rows. */
int oracle_dx_rows(const int8_t* dY, const uint8_t* Wp, int32_t* dX, int64_t M, int64_t N,
                   int64_t K, const int64_t* rows, int64_t nrows) {
  if (M < 0 || N < 0 || K < 0 || nrows < 0) return ORACLE_EINVAL;
  int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = rows ? rows[i] : i;
    if (m < 0 || m >= M) { bad |= 1; continue; }
    for (int64_t k = 0; k < K; ++k) {
      int64_t acc = 0;
      for (int64_t n = 0; n < N; ++n)
        acc += (int64_t)dY[m * N + n] * (int64_t)weight_of(Wp, K, n, k);
      if (!fits_i32(acc)) bad |= 2;
      dX[i * K + k] = (int32_t)acc;
    }
  }
  if (bad & 1) return ORACLE_EINVAL;
  if (bad & 2) return ORACLE_EOVERFLOW;
  return ORACLE_OK;
}

int oracle_dx(const int8_t* dY, const uint8_t* Wp, int32_t* dX, int64_t M, int64_t N, int64_t K) {
  return oracle_dx_rows(dY, Wp, dX, M, N, K, NULL, M);
}

/* Backward weights, [P-bwd] kernel 2: dW[k][n] = sum_{m<M} A[m][k] * dY[m][n],
 * summed over the rows m.  `rows` lists k indices (rows of dW). */
int oracle_dw_rows(const int8_t* A, const int8_t* dY, int32_t* dW, int64_t M, int64_t N,
                   int64_t K, const int64_t* rows, int64_t nrows) {
  if (M < 0 || N < 0 || K < 0 || nrows < 0) return ORACLE_EINVAL;
  int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t k = rows ? rows[i] : i;
    if (k < 0 || k >= K) { bad |= 1; continue; }
    for (int64_t n = 0; n < N; ++n) {
      int64_t acc = 0;
      for (int64_t m = 0; m < M; ++m)
        acc += (int64_t)A[m * K + k] * (int64_t)dY[m * N + n];
      if (!fits_i32(acc)) bad |= 2;
      dW[i * N + n] = (int32_t)acc;
    }
  }
  if (bad & 1) return ORACLE_EINVAL;
  if (bad & 2) return ORACLE_EOVERFLOW;
  return ORACLE_OK;
}

int oracle_dw(const int8_t* A, const int8_t* dY, int32_t* dW, int64_t M, int64_t N, int64_t K) {
  return oracle_dw_rows(A, dY, dW, M, N, K, NULL, K);
}

/* Number of OpenMP threads the oracle's loops use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  int t = 1;
#pragma omp parallel
  {
#pragma omp single
    t = omp_get_num_threads();
  }
  return t;
#else
  return 1;
#endif
}
