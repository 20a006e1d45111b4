// GEMM calls whose operands live in host memory: staging to the device in row blocks,
// overlapped with the GEMM of earlier blocks and the read-back of their D rows.
//
// A caller holding host buffers needs the copies as well as the GEMM ("Day 84: CUTLASS and
// CuTe layouts" — "Two programs": the harness moves the operands to the device, runs the
// kernel and reads D back; "CUTLASS, in depth" — "A complete Hopper GEMM": the device-level
// operator owns the launch and its workspace).  On this part the host link, not the tensor
// cores, bounds such a call, so the copies are cut to overlap:
//   copy stream "up"    B (and the bias) first, then per row block i the rows of A and C;
//   the caller's stream block i's GEMM (one call of the device entry point on the
//                       sub-matrices: M' rows, A, C and D offset by the block's first row),
//                       after block i's rows have landed;
//   copy stream "down"  block i's D rows, after block i's GEMM.
// Blocks are multiples of 256 rows, so every block's first row keeps the 16-byte alignment
// of A (either major), C and D; each block computes exactly what one call over all rows
// computes for those rows.  A row block of a K-major A is one contiguous copy, of an
// M-major A one two-dimensional copy (rows m0..m1 of each of the K columns).
//
// Device staging memory (one buffer per device, grown on demand, kept between calls) and
// the copy streams and events are owned by this file.  Calls on one device are serialised:
// each call's copies wait for the previous call to finish with the staging buffer.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gb300_gemm.h"

namespace {

constexpr int kMaxBlocks = 8;
constexpr int64_t kMinBlockRows = 1024;
constexpr int64_t kBlockAlign = 256;

struct Stage {
  std::mutex mu;
  bool ready = false;
  void* buf = nullptr;
  size_t cap = 0;
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, prev_done = nullptr, down_done = nullptr;
  cudaEvent_t landed[kMaxBlocks] = {}, computed[kMaxBlocks] = {};
  bool have_prev = false;
};

Stage g_stage[128];

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Row blocks of a call with M rows: one block below 2 * kMinBlockRows rows, else up to
// kMaxBlocks blocks of at least kMinBlockRows rows, each (but the last) a multiple of 256.
int row_blocks(int64_t M, int64_t* bounds) {
  if (M < 2 * kMinBlockRows) {
    bounds[0] = 0;
    bounds[1] = M;
    return 1;
  }
  int64_t n = M / kMinBlockRows;
  if (n > kMaxBlocks) n = kMaxBlocks;
  const int64_t rows = round_up((M + n - 1) / n, kBlockAlign);
  int count = 0;
  for (int64_t m0 = 0; m0 < M; m0 += rows) bounds[count++] = m0;
  bounds[count] = M;
  return count;
}

gb_status ensure_ready(Stage& s) {
  if (s.ready) return GB_OK;
  if (cudaStreamCreateWithFlags(&s.up, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&s.down, cudaStreamNonBlocking) != cudaSuccess)
    return GB_ERR_CUDA;
  cudaEvent_t* evs[] = {&s.start, &s.prev_done, &s.down_done};
  for (cudaEvent_t* e : evs)
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return GB_ERR_CUDA;
  for (int i = 0; i < kMaxBlocks; ++i)
    if (cudaEventCreateWithFlags(&s.landed[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.computed[i], cudaEventDisableTiming) != cudaSuccess)
      return GB_ERR_CUDA;
  s.ready = true;
  return GB_OK;
}

// Host pointers only: pinned (page-locked or registered), pageable or managed memory.
bool is_host_pointer(const void* p) {
  if (p == nullptr) return true;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return true;   // unknown to the runtime: ordinary host memory
  }
  return a.type != cudaMemoryTypeDevice;
}

// One host-operand GEMM.  The stored extents of the operands (elements), element sizes and
// the per-block launch are described by the caller.
struct HostCall {
  int64_t M, N, K;
  const void* A;
  int64_t lda;
  int majorA;
  const void* B;
  int64_t b_elems;     // elements of B's stored extent
  const void* C;
  void* D;
  const void* bias;    // N elements of c_size, or null
  float* amax;         // host float combined by max, or null
  int a_size, b_size, c_size, d_size;
};

template <typename Launch>
gb_status enqueue_host_call(Stage& s, const HostCall& h, cudaStream_t main, Launch&& launch);

template <typename Launch>
gb_status run_host_call(const HostCall& h, cudaStream_t main, Launch&& launch) {
  if (!is_host_pointer(h.A) || !is_host_pointer(h.B) || !is_host_pointer(h.C) || !is_host_pointer(h.D) ||
      !is_host_pointer(h.bias) || !is_host_pointer(h.amax))
    return GB_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= 128) return GB_ERR_CUDA;
  Stage& s = g_stage[device];
  std::lock_guard<std::mutex> lk(s.mu);
  gb_status st = ensure_ready(s);
  if (st != GB_OK) return st;
  st = enqueue_host_call(s, h, main, launch);
  // whatever was queued (all of it, or a part before an error), the caller's stream and the
  // next host-operand call on this device come after it
  cudaEventRecord(s.down_done, s.up);
  cudaStreamWaitEvent(main, s.down_done, 0);
  cudaEventRecord(s.down_done, s.down);
  cudaStreamWaitEvent(main, s.down_done, 0);
  if (cudaEventRecord(s.prev_done, main) != cudaSuccess) return GB_ERR_CUDA;
  s.have_prev = true;
  return st;
}

template <typename Launch>
gb_status enqueue_host_call(Stage& s, const HostCall& h, cudaStream_t main, Launch&& launch) {
  gb_status st = GB_OK;

  // staging layout: A, B, C, D, bias, amax, each 256-byte aligned
  const int64_t a_elems = h.K == 0 ? 0
                          : (h.majorA == GB_K_MAJOR ? (h.M - 1) * h.lda + h.K : (h.K - 1) * h.lda + h.M);
  const int64_t off_a = 0;
  const int64_t off_b = round_up(off_a + a_elems * h.a_size, 256);
  const int64_t off_c = round_up(off_b + (h.K == 0 ? 0 : h.b_elems) * h.b_size, 256);
  const int64_t off_d = round_up(off_c + (h.C ? h.M * h.N * h.c_size : 0), 256);
  const int64_t off_bias = round_up(off_d + h.M * h.N * h.d_size, 256);
  const int64_t off_amax = round_up(off_bias + (h.bias ? h.N * h.c_size : 0), 256);
  const size_t need = static_cast<size_t>(off_amax + 256);
  if (need > s.cap) {
    // growing: the old buffer may still be read by an earlier call's copies or GEMMs
    if (s.buf) {
      if (cudaDeviceSynchronize() != cudaSuccess || cudaFree(s.buf) != cudaSuccess) return GB_ERR_CUDA;
      s.buf = nullptr;
      s.cap = 0;
    }
    if (cudaMalloc(&s.buf, need) != cudaSuccess) {
      cudaGetLastError();
      s.buf = nullptr;
      return GB_ERR_CUDA;
    }
    s.cap = need;
  }
  uint8_t* base = static_cast<uint8_t*>(s.buf);
  uint8_t* A_d = base + off_a;
  uint8_t* B_d = base + off_b;
  uint8_t* C_d = h.C ? base + off_c : nullptr;
  uint8_t* D_d = base + off_d;
  uint8_t* bias_d = h.bias ? base + off_bias : nullptr;
  float* amax_d = h.amax ? reinterpret_cast<float*>(base + off_amax) : nullptr;
  const uint8_t* A_h = static_cast<const uint8_t*>(h.A);
  const uint8_t* C_h = static_cast<const uint8_t*>(h.C);
  uint8_t* D_h = static_cast<uint8_t*>(h.D);

#define GB_CK(x) \
  do {           \
    if ((x) != cudaSuccess) return GB_ERR_CUDA; \
  } while (0)
  // order: everything queued on the caller's stream before this call, and the previous
  // host-operand call on this device (any stream), before the staging buffer is rewritten
  GB_CK(cudaEventRecord(s.start, main));
  GB_CK(cudaStreamWaitEvent(s.up, s.start, 0));
  GB_CK(cudaStreamWaitEvent(s.down, s.start, 0));
  if (s.have_prev) {
    GB_CK(cudaStreamWaitEvent(s.up, s.prev_done, 0));
    GB_CK(cudaStreamWaitEvent(main, s.prev_done, 0));
  }
  if (h.K > 0) GB_CK(cudaMemcpyAsync(B_d, h.B, static_cast<size_t>(h.b_elems * h.b_size), cudaMemcpyHostToDevice, s.up));
  if (bias_d) GB_CK(cudaMemcpyAsync(bias_d, h.bias, static_cast<size_t>(h.N * h.c_size), cudaMemcpyHostToDevice, s.up));
  if (amax_d) GB_CK(cudaMemcpyAsync(amax_d, h.amax, sizeof(float), cudaMemcpyHostToDevice, s.up));

  int64_t bounds[kMaxBlocks + 1];
  const int nb = row_blocks(h.M, bounds);
  auto upload = [&](int i) -> gb_status {
    const int64_t m0 = bounds[i], m1 = bounds[i + 1];
    if (h.K > 0) {
      if (h.majorA == GB_K_MAJOR) {
        const int64_t e0 = m0 * h.lda, e1 = (m1 - 1) * h.lda + h.K;
        GB_CK(cudaMemcpyAsync(A_d + e0 * h.a_size, A_h + e0 * h.a_size, static_cast<size_t>((e1 - e0) * h.a_size),
                              cudaMemcpyHostToDevice, s.up));
      } else {
        const size_t pitch = static_cast<size_t>(h.lda * h.a_size);
        GB_CK(cudaMemcpy2DAsync(A_d + m0 * h.a_size, pitch, A_h + m0 * h.a_size, pitch,
                                static_cast<size_t>((m1 - m0) * h.a_size), static_cast<size_t>(h.K),
                                cudaMemcpyHostToDevice, s.up));
      }
    }
    if (C_d)
      GB_CK(cudaMemcpyAsync(C_d + m0 * h.N * h.c_size, C_h + m0 * h.N * h.c_size,
                            static_cast<size_t>((m1 - m0) * h.N * h.c_size), cudaMemcpyHostToDevice, s.up));
    GB_CK(cudaEventRecord(s.landed[i], s.up));
    return GB_OK;
  };
  // block i + 1 is queued for upload before block i's read-back, so that a read-back into
  // pageable memory (which returns only once it is done) does not hold up the next upload
  if ((st = upload(0)) != GB_OK) return st;
  for (int i = 0; i < nb; ++i) {
    if (i + 1 < nb && (st = upload(i + 1)) != GB_OK) return st;
    const int64_t m0 = bounds[i], m1 = bounds[i + 1];
    GB_CK(cudaStreamWaitEvent(main, s.landed[i], 0));
    const uint8_t* A_blk = h.majorA == GB_K_MAJOR ? A_d + m0 * h.lda * h.a_size : A_d + m0 * h.a_size;
    st = launch(m1 - m0, h.K > 0 ? A_blk : nullptr, h.K > 0 ? B_d : nullptr,
                C_d ? C_d + m0 * h.N * h.c_size : nullptr, D_d + m0 * h.N * h.d_size, bias_d, amax_d, main);
    if (st != GB_OK) return st;
    GB_CK(cudaEventRecord(s.computed[i], main));
    GB_CK(cudaStreamWaitEvent(s.down, s.computed[i], 0));
    GB_CK(cudaMemcpyAsync(D_h + m0 * h.N * h.d_size, D_d + m0 * h.N * h.d_size,
                          static_cast<size_t>((m1 - m0) * h.N * h.d_size), cudaMemcpyDeviceToHost, s.down));
  }
  if (amax_d) GB_CK(cudaMemcpyAsync(h.amax, amax_d, sizeof(float), cudaMemcpyDeviceToHost, s.down));
  // (the caller's stream then waits for both copy streams: D and amax are in host memory
  // when it reaches its next work)
#undef GB_CK
  return GB_OK;
}

bool valid_major(int m) { return m == GB_K_MAJOR || m == GB_MN_MAJOR; }

// The argument checks of the device entry points that do not depend on device pointers,
// made before any copy so that a call fails whole or not at all.
gb_status check_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int majorA, const void* B,
                     int64_t ldb, int majorB, float beta, const void* C, const void* D, int in_bytes) {
  if (M < 0 || N < 0 || K < 0 || !valid_major(majorA) || !valid_major(majorB)) return GB_ERR_INVALID_ARG;
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (M > lim || N > lim || K > lim) return GB_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GB_OK;
  if (D == nullptr || (beta != 0.0f && C == nullptr)) return GB_ERR_INVALID_ARG;
  if (K > 0) {
    if (A == nullptr || B == nullptr) return GB_ERR_INVALID_ARG;
    if (lda < (majorA == GB_K_MAJOR ? K : M) || ldb < (majorB == GB_K_MAJOR ? K : N)) return GB_ERR_INVALID_ARG;
    if ((lda * in_bytes) % 16 != 0 || (ldb * in_bytes) % 16 != 0) return GB_ERR_MISALIGNED;
  }
  return GB_OK;
}

int64_t b_extent(int64_t N, int64_t K, int64_t ldb, int majorB) {
  if (K == 0 || N == 0) return 0;
  return majorB == GB_K_MAJOR ? (N - 1) * ldb + K : (K - 1) * ldb + N;
}

gb_status host16(int dtype, int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda, int majorA,
                 const void* B, int64_t ldb, int majorB, float beta, const void* C, void* D, void* stream) {
  gb_status st = check_args(M, N, K, A, lda, majorA, B, ldb, majorB, beta, C, D, 2);
  if (st != GB_OK || M == 0 || N == 0) return st;
  const HostCall h{M, N, K, A, lda, majorA, B, b_extent(N, K, ldb, majorB), beta != 0.0f ? C : nullptr, D,
                   nullptr, nullptr, 2, 2, 2, 2};
  return run_host_call(h, static_cast<cudaStream_t>(stream),
                       [&](int64_t rows, const void* Ab, const void* Bb, const void* Cb, void* Db, const void*,
                           float*, cudaStream_t s) {
                         return dtype == GB_BF16
                                    ? gb_gemm_bf16(rows, N, K, alpha, Ab, lda, majorA, Bb, ldb, majorB, beta, Cb, Db, s)
                                    : gb_gemm_f16(rows, N, K, alpha, Ab, lda, majorA, Bb, ldb, majorB, beta, Cb, Db, s);
                       });
}

}  // namespace

extern "C" {

gb_status gb_gemm_f16_host(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda, int majorA,
                           const void* B, int64_t ldb, int majorB, float beta, const void* C, void* D,
                           void* stream) {
  return host16(GB_F16, M, N, K, alpha, A, lda, majorA, B, ldb, majorB, beta, C, D, stream);
}

gb_status gb_gemm_bf16_host(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda, int majorA,
                            const void* B, int64_t ldb, int majorB, float beta, const void* C, void* D,
                            void* stream) {
  return host16(GB_BF16, M, N, K, alpha, A, lda, majorA, B, ldb, majorB, beta, C, D, stream);
}

gb_status gb_gemm_fp8_host(int a_format, int b_format, int out_dtype, int64_t M, int64_t N, int64_t K, float alpha,
                           const void* A, int64_t lda, const void* B, int64_t ldb, float beta, const void* C,
                           void* D, const gb_epilogue* epi, void* stream) {
  if (a_format != GB_FP8_E4M3 && a_format != GB_FP8_E5M2) return GB_ERR_INVALID_ARG;
  if (b_format != GB_FP8_E4M3 && b_format != GB_FP8_E5M2) return GB_ERR_INVALID_ARG;
  if (out_dtype != GB_F16 && out_dtype != GB_BF16) return GB_ERR_INVALID_ARG;
  if (epi && (epi->out_format < GB_OUT_INPUT_TYPE || epi->out_format > GB_OUT_E5M2)) return GB_ERR_INVALID_ARG;
  gb_status st = check_args(M, N, K, A, lda, GB_K_MAJOR, B, ldb, GB_K_MAJOR, beta, C, D, 1);
  if (st != GB_OK || M == 0 || N == 0) return st;
  const int d_size = (epi && epi->out_format != GB_OUT_INPUT_TYPE) ? 1 : 2;
  const HostCall h{M, N, K, A, lda, GB_K_MAJOR, B, b_extent(N, K, ldb, GB_K_MAJOR), beta != 0.0f ? C : nullptr, D,
                   epi ? epi->bias : nullptr, epi ? epi->amax : nullptr, 1, 1, 2, d_size};
  return run_host_call(h, static_cast<cudaStream_t>(stream),
                       [&](int64_t rows, const void* Ab, const void* Bb, const void* Cb, void* Db, const void* bias_d,
                           float* amax_d, cudaStream_t s) {
                         gb_epilogue e{};
                         if (epi) {
                           e = *epi;
                           e.bias = bias_d;
                           e.amax = amax_d;
                         }
                         return gb_gemm_fp8(a_format, b_format, out_dtype, rows, N, K, alpha, Ab, lda, Bb, ldb, beta,
                                            Cb, Db, epi ? &e : nullptr, nullptr, 0, s);
                       });
}

gb_status gb_gemm_host_row_blocks(int64_t M, int64_t* bounds, int* count) {
  if (M < 0 || bounds == nullptr || count == nullptr) return GB_ERR_INVALID_ARG;
  *count = row_blocks(M, bounds);
  return GB_OK;
}

gb_status gb_host_staging_free(void) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= 128) return GB_ERR_CUDA;
  Stage& s = g_stage[device];
  std::lock_guard<std::mutex> lk(s.mu);
  if (s.buf) {
    if (cudaDeviceSynchronize() != cudaSuccess || cudaFree(s.buf) != cudaSuccess) return GB_ERR_CUDA;
    s.buf = nullptr;
    s.cap = 0;
  }
  return GB_OK;
}

}  // extern "C"
