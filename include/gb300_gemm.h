/*
 * gb300_gemm.h — C ABI of the sm_103a tiled GEMM  D = alpha * A * B + beta * C.
 *
 * Operation ("CUTLASS, in depth" — "The problem CUTLASS solves"): A is M x K, B is
 * K x N, C and D are M x N; 16-bit inputs (fp16 or bf16, named by the symbol), products
 * accumulated in fp32, alpha/beta applied in fp32, D rounded to nearest even.
 *
 * A CTA (or a pair of CTAs on two SMs) owns an output tile (128 x 64 or 128 x 256 for one
 * CTA; 256 x 224, 256 x 256, 256 x 448 or 256 x 512 for a pair) and walks K in steps of 64 with A/B
 * slices staged in shared memory ("CUTLASS, in depth" — "The problem CUTLASS solves",
 * tiling); tile and element addressing come from shape:stride layouts divided into (tile,
 * grid) modes ("Day 84: CUTLASS and CuTe layouts" — "A layout is a shape and a stride").
 * The form is chosen by shape ("CUTLASS, in depth" — "Worked example: tile choice and wave
 * quantisation"; gb_set_kernel_variant overrides it): narrow 128 x 64 tiles when N <= 64 or
 * when those tiles fit in one wave (one per SM), else the single CTA when M <= 128 or its
 * 128 x 256 tiles fit in one wave, else the pair width whose persistent waves of tiles cost
 * least (ceil(tiles / pairs) waves, pairs = half the device's SMs, times the measured cost of
 * a tile of that width; 224 needs K-major B; the 448- and 512-column tiles, whose epilogue
 * nothing overlaps, are left to 16-bit inputs with the plain alpha/beta epilogue).
 *
 * Operand layouts (a matrix is named after its stride-1 mode, "Layouts as Algebra" —
 * "One notation, and no more transposes"):
 *   A (M x K): GB_K_MAJOR  A(m,k) = A[m*lda + k]   (row-major, lda >= K)
 *              GB_MN_MAJOR A(m,k) = A[m + k*lda]   (column-major, lda >= M)
 *   B (K x N): GB_K_MAJOR  B(k,n) = B[n*ldb + k]   (column-major, ldb >= K)
 *              GB_MN_MAJOR B(k,n) = B[k*ldb + n]   (row-major, ldb >= N)
 *   C, D (M x N): row-major, leading dimension N.  C and D have the symbol's dtype.
 *
 * Ownership and execution: every buffer is caller-owned device memory (the *_host calls
 * below take host memory instead); the call allocates nothing, is asynchronous on
 * `stream` (a cudaStream_t; NULL is the legacy default stream) and returns once the
 * kernel is queued.  The kernel is launched with
 * programmatic stream serialisation: its set-up may overlap the end of the previous kernel
 * in the stream, and it touches global memory only after that kernel has completed (stream
 * order is kept for every buffer).  Calls may come from several host threads at once: the
 * library's host state (per-device set-up, cached plans) is kept under a lock.  The call
 * reads no C when beta == 0, and then C may be NULL.  M == 0 or N == 0 is a no-op; K == 0 gives
 * D = beta*C.
 *
 * Errors are reported before any launch (validation "can_implement", "CUTLASS, in
 * depth" — "Failure modes"; "Day 84" — "Pitfalls"):
 *   GB_ERR_INVALID_ARG      negative size, bad major, NULL operand that is needed,
 *                           leading dimension smaller than the contiguous extent, or a
 *                           size beyond the tensor-copy limits (M, N, K < 2^31).
 *   GB_ERR_MISALIGNED       a pointer not 16-byte aligned, or lda/ldb not a multiple of
 *                           8 elements (16 bytes): tile copies need 16-byte rows.
 *   GB_ERR_UNSUPPORTED_ARCH the current device is not compute capability 10.3.
 *   GB_ERR_LAUNCH           the CUDA launch or descriptor encoding failed.
 * A wait inside the kernel that runs past its limit (default 2 s) makes the kernel stop,
 * record a code in a device status word and return; gb_last_device_status reads it.
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GB_OK = 0,
  GB_ERR_INVALID_ARG = 1,
  GB_ERR_MISALIGNED = 2,
  GB_ERR_UNSUPPORTED_ARCH = 3,
  GB_ERR_LAUNCH = 4,
  GB_ERR_TIMEOUT = 5,
  GB_ERR_CUDA = 6,
  GB_ERR_SCRATCH_LIMIT = 7   /* gb_gemm_noalloc: the device needs more scratch than the
                                built-in array holds */
} gb_status;

typedef enum { GB_K_MAJOR = 0, GB_MN_MAJOR = 1 } gb_major;

typedef enum { GB_F16 = 0, GB_BF16 = 1 } gb_dtype;

/* D = alpha*A*B + beta*C with fp16 operands (fp32 accumulate). */
gb_status gb_gemm_f16(int64_t M, int64_t N, int64_t K, float alpha,
                      const void* A, int64_t lda, int majorA,
                      const void* B, int64_t ldb, int majorB,
                      float beta, const void* C, void* D, void* stream);

/* Same with bf16 operands. */
gb_status gb_gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha,
                       const void* A, int64_t lda, int majorA,
                       const void* B, int64_t ldb, int majorB,
                       float beta, const void* C, void* D, void* stream);

/* The same GEMM with a caller-owned scratch workspace, which lets the kernel split the
   K loop of some tiles across CTAs ("stream-K", after "CUTLASS, in depth" — "Kernel
   schedules": split-K and stream-K divide K across CTAs when output tiles are too few to
   fill the GPU, at the cost of a reduction and a workspace).  Each CTA first runs whole
   tiles, then an even contiguous share of the remaining (tile, stage-block) units (a
   stage-block is the k-blocks one pipeline stage holds: two for the 224- and 256-column CTA
   pairs, one for single CTAs and the 448- and 512-column pairs); the CTA that holds a tile's
   first unit adds the other CTAs' fp32 partials, in CTA order, before the epilogue.
   workspace: device memory of at least gb_gemm_workspace_bytes() bytes, 256-byte aligned,
   zero-filled before its first use and not shared by calls that may run at the same time
   (it is reused as is by later calls; each launch tags its hand-offs with a new number).
   Results equal the plain call's within the same bound; summation order differs. */
gb_status gb_gemm_f16_ws(int64_t M, int64_t N, int64_t K, float alpha,
                         const void* A, int64_t lda, int majorA,
                         const void* B, int64_t ldb, int majorB,
                         float beta, const void* C, void* D,
                         void* workspace, size_t workspace_bytes, void* stream);
gb_status gb_gemm_bf16_ws(int64_t M, int64_t N, int64_t K, float alpha,
                          const void* A, int64_t lda, int majorA,
                          const void* B, int64_t ldb, int majorB,
                          float beta, const void* C, void* D,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Workspace size for the *_ws calls on the current device (one 128 x 512 fp32 partial and
   one flag per SM).  GB_ERR_UNSUPPORTED_ARCH without a compute capability 10.3 device. */
gb_status gb_gemm_workspace_bytes(size_t* bytes);

/* Schedule for later *_ws calls (process-wide): 0 (the default) stream-K when the output
   tiles are fewer than the CTAs and the (tile, stage-block) units give every CTA at least two,
   else whole tiles; 1 whole tiles only; 2 stream-K whenever K > 0.  GB_ERR_INVALID_ARG for
   other values. */
gb_status gb_set_schedule(int schedule);

/* Fused epilogue ("CUTLASS, in depth" — "Epilogue fusion": load C, load a bias vector,
   add, activate, compute an absolute maximum for FP8 scaling, and store, on the
   accumulator before it leaves the chip).  Per output, in fp32:
     v = alpha*acc + beta*C[i,j];  v += bias[j] (if bias);  v = act(v);
     *amax = max(*amax, |v|) (if amax);  D[i,j] = round(v) to the input type, or, for an FP8
     output, round(v * out_scale) to FP8 with saturation at the largest finite value.
   bias: N values of the input type (column j of D gets bias[j]), or NULL.
   amax: a device float, combined with its current contents by max (zero it first), or NULL.
   FP8 outputs are one byte per element, row-major with leading dimension N. */
typedef enum { GB_ACT_NONE = 0, GB_ACT_RELU = 1, GB_ACT_GELU = 2 } gb_activation;
typedef enum { GB_OUT_INPUT_TYPE = 0, GB_OUT_E4M3 = 1, GB_OUT_E5M2 = 2 } gb_out_format;
typedef struct {
  const void* bias;
  int activation;     /* gb_activation; GELU is 0.5 v (1 + erf(v / sqrt 2)) */
  float* amax;
  int out_format;     /* gb_out_format */
  float out_scale;    /* used by FP8 outputs; must be finite and > 0 for them */
} gb_epilogue;

/* D = epilogue(alpha*A*B + beta*C) with fp16 (dtype GB_F16) or bf16 (GB_BF16) inputs.  epi
   NULL gives the plain call.  workspace / workspace_bytes: as for gb_gemm_f16_ws, or NULL/0
   for whole tiles only.  Errors as for gb_gemm_f16, plus GB_ERR_INVALID_ARG for an unknown
   activation or output format or a bad FP8 scale. */
gb_status gb_gemm_ex(int dtype, int64_t M, int64_t N, int64_t K, float alpha,
                     const void* A, int64_t lda, int majorA,
                     const void* B, int64_t ldb, int majorB,
                     float beta, const void* C, void* D, const gb_epilogue* epi,
                     void* workspace, size_t workspace_bytes, void* stream);

/* GEMM with 8-bit floating-point inputs ("CUTLASS, in depth" — "Epilogue fusion" and
   "Numerics": the tensor cores take FP8 operands; FP8 data carries a scale factor, and a
   GEMM without the right scales overflows).  Computes, in fp32 on the tensor cores,
     D = epilogue(alpha * A*B + beta*C)
   where A (M x K) and B (K x N) hold FP8 codes: a_format / b_format are GB_FP8_E4M3 (OCP
   E4M3: no infinities, largest finite 448) or GB_FP8_E5M2 (OCP E5M2), one byte each, and
   may differ.  Both operands are K-major: A row-major with leading dimension lda, B stored
   as its transpose (N rows of K, leading dimension ldb); lda and ldb are multiples of 16
   elements and A, B are 16-byte aligned.  Per-tensor scale factors are folded into alpha
   by the caller (alpha = alpha' * scale_A * scale_B for dequantised operands
   scale_A * A, scale_B * B).  C, D and the bias are of out_dtype (GB_F16 or GB_BF16), laid
   out as for gb_gemm_f16; epi, workspace and stream as for gb_gemm_ex (an FP8 output via
   epi->out_format gives an FP8-in, FP8-out GEMM).  Errors as for gb_gemm_ex, plus
   GB_ERR_INVALID_ARG for an unknown format or out_dtype and GB_ERR_MISALIGNED for lda or
   ldb not a multiple of 16. */
typedef enum { GB_FP8_E4M3 = 0, GB_FP8_E5M2 = 1 } gb_fp8_format;
gb_status gb_gemm_fp8(int a_format, int b_format, int out_dtype, int64_t M, int64_t N, int64_t K,
                      float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                      float beta, const void* C, void* D, const gb_epilogue* epi,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Block-scaled FP8 GEMM ("MX": the per-block scale factors of "CUTLASS, in depth" —
   "Epilogue fusion" and "Numerics", read as the OCP Microscaling format).  Every 32
   consecutive K elements of a row of A, and of a column of B, share one E8M0 scale
   2^(e - 127) (e = 255 is NaN):
     D = epilogue(alpha * sum_k (2^(sa(i,k/32)-127) A(i,k)) (2^(sb(j,k/32)-127) B(k,j)) + beta*C)
   computed on the tensor cores (kind::mxf8f6f4, fp32 accumulation).  A and B are as for
   gb_gemm_fp8 (K-major FP8 codes of a_format / b_format, lda and ldb multiples of 16).
   sfa and sfb are the scales packed by gb_mx_pack_scales (operand 0 for A with M rows,
   operand 1 for B with N rows), 16-byte aligned device buffers.  C, D, epi, workspace and
   stream as for gb_gemm_fp8.  Errors as for gb_gemm_fp8, plus GB_ERR_INVALID_ARG for a
   missing scale buffer when K > 0.  Uses the single-CTA kernel for M <= 128 and the
   CTA-pair kernel otherwise. */
gb_status gb_gemm_mxfp8(int a_format, int b_format, int out_dtype, int64_t M, int64_t N, int64_t K,
                        float alpha, const void* A, int64_t lda, const void* sfa,
                        const void* B, int64_t ldb, const void* sfb,
                        float beta, const void* C, void* D, const gb_epilogue* epi,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Packed scale factors for gb_gemm_mxfp8.  The kernels read scales in 512-byte atoms, each
   covering 128 rows (or columns) and one k-block of 128 elements (4 scales per row): scale
   (row 32j + i, scale kk of the k-block) at byte 16i + 4j + kk of the atom, i.e. the layout
   ((32,4),4):((16,4),1) from (row, scale) to bytes.  Operand 0 (A, rows = M): one atom per
   (128 rows, k-block), atom (rb, kb) at byte (rb * ceil(K/128) + kb) * 512.  Operand 1 (B,
   rows = N): 1024 bytes per (224 columns, k-block) at (nb * ceil(K/128) + kb) * 1024, the
   seven 32-column groups g of the block in atom g / 4, slot g % 4 (the eighth slot is
   padding).  Padding holds 127 (a scale of 1).
   gb_mx_scales_bytes: size of the packed buffer.  gb_mx_pack_scales: fill `dst` (device,
   that size) from `src` (device, rows x ceil(K/32) E8M0 bytes, row pitch ld_src >=
   ceil(K/32)), asynchronously on `stream`.  GB_ERR_INVALID_ARG for a bad operand, negative
   sizes or a short pitch. */
gb_status gb_mx_scales_bytes(int operand, int64_t rows, int64_t K, size_t* bytes);
gb_status gb_mx_pack_scales(int operand, int64_t rows, int64_t K, const void* src, int64_t ld_src,
                            void* dst, void* stream);

/* Allocation-free GEMM (no counterpart on the pages: an addition for callers that may not
   allocate device memory).  Some callers cannot call cudaMalloc at the point where they
   run a GEMM: code inside a runtime that owns every byte of device memory (a serving
   engine or framework plugin with a fixed memory plan), code on a latency-critical path
   where an allocation would synchronise the device, or code that only receives
   pre-allocated input and output buffers.  This entry point serves them: it computes the
   same result as gb_gemm_f16_ws / gb_gemm_bf16_ws (dtype = GB_F16 or GB_BF16), but its
   stream-K scratch lives in a static array inside this library instead of a caller
   workspace; it calls no allocating routine.
   Limits and sharing: the array holds about 40 MiB (one 128 x 512 fp32 partial and one
   flag for each of up to 160 SMs) and every GPU that loads the library keeps it until
   the process exits; a device with more SMs gets GB_ERR_SCRATCH_LIMIT.  All calls on a
   device share the one array and it keeps the last call's contents, so calls that may run
   at the same time on the GPU (different streams, overlapping launches) race and must not
   be issued.  The first call on each device looks up the array's device address and
   clears its flags (an asynchronous memset on `stream`, ahead of the call's kernel); make
   that first call before any stream capture.  Other arguments, errors and ownership as
   for gb_gemm_f16. */
gb_status gb_gemm_noalloc(int dtype, int64_t M, int64_t N, int64_t K, float alpha,
                          const void* A, int64_t lda, int majorA,
                          const void* B, int64_t ldb, int majorB,
                          float beta, const void* C, void* D, void* stream);

/* The same GEMMs with every operand in HOST memory (pinned, pageable or managed; device
   pointers are rejected with GB_ERR_INVALID_ARG): for a caller that holds its matrices on
   the host ("Day 84: CUTLASS and CuTe layouts" — "Two programs": the harness copies the
   operands in, runs the kernel and reads D back).  Layouts, alpha/beta, validation and
   results are those of gb_gemm_f16 / gb_gemm_bf16 / gb_gemm_fp8 (every output equal, bit
   for bit, to the device call's); for gb_gemm_fp8_host, epi->bias is a host array of N
   values and epi->amax a host float, both optional.
   Execution: B goes to the device first; then A's and C's rows go up in row blocks
   (gb_gemm_host_row_blocks) on a copy stream while earlier blocks are multiplied on
   `stream` and their D rows come back on a second copy stream, so the copies in both
   directions and the GEMM overlap.  The call is asynchronous on `stream`: it returns once
   the work is queued (with pageable buffers some copies finish before it returns), and D
   (and *amax) hold the result once `stream` has reached the end of the call (e.g. after
   cudaStreamSynchronize(stream)).  Work queued on `stream` before the call (e.g. writes to
   the host operands) comes first.
   Memory: unlike the device entry points, these calls use device staging memory owned by
   the library: one buffer per device for A, B, C and D, allocated on the first call and
   grown when a call needs more (growing synchronises the device), kept for later calls
   until gb_host_staging_free().  Host-operand calls on one device share it, so each call
   waits on the GPU for the previous one (on any stream) to release it.  Errors: those of
   the device entry points, checked before any copy; GB_ERR_CUDA if a copy, event or
   allocation fails. */
gb_status gb_gemm_f16_host(int64_t M, int64_t N, int64_t K, float alpha,
                           const void* A, int64_t lda, int majorA,
                           const void* B, int64_t ldb, int majorB,
                           float beta, const void* C, void* D, void* stream);
gb_status gb_gemm_bf16_host(int64_t M, int64_t N, int64_t K, float alpha,
                            const void* A, int64_t lda, int majorA,
                            const void* B, int64_t ldb, int majorB,
                            float beta, const void* C, void* D, void* stream);
gb_status gb_gemm_fp8_host(int a_format, int b_format, int out_dtype, int64_t M, int64_t N, int64_t K,
                           float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                           float beta, const void* C, void* D, const gb_epilogue* epi, void* stream);

/* Row blocks of a host-operand call with M rows: *count blocks, block i = rows
   [bounds[i], bounds[i+1]); bounds must hold 9 values.  One block when M < 2048, else up to
   8 blocks of at least 1024 rows, each but the last a multiple of 256 rows (so every block
   starts 16-byte aligned in A, C and D).  Pure host computation. */
gb_status gb_gemm_host_row_blocks(int64_t M, int64_t* bounds, int* count);

/* Free the current device's staging buffer of the host-operand calls (synchronises the
   device).  The next host-operand call allocates it again. */
gb_status gb_host_staging_free(void);

/* Synchronises `stream`, then returns GB_ERR_TIMEOUT if any kernel of this library on the
   current device recorded a wait that ran out since the last call (the raw code goes to
   *detail when detail != NULL: bits 0-7 the wait that ran out, bits 8-31 the CTA), and
   clears the record.  GB_ERR_CUDA if synchronising failed. */
gb_status gb_last_device_status(void* stream, uint32_t* detail);

/* Name of a status code. */
const char* gb_status_string(int status);

/* Host-side plan of one call: the tile grid and tensor-copy geometry the layouts give.
   Pure host computation (no GPU needed), same validation as the GEMM call except the
   pointer and device checks. */
typedef struct {
  int64_t m_tiles, n_tiles, k_blocks;   /* grid of tile_m x tile_n output tiles, K steps of 64 */
  int64_t tile_m, tile_n, tile_k;       /* 128 (single) or 256 (pair); 64, 224, 256, 448 or 512; 64 */
  int64_t a_dim[2], a_row_bytes;        /* A copy: extents (inner first), row pitch */
  int64_t a_box[2], a_boxes;            /* box extents (inner first), boxes per stage per CTA */
  int64_t b_dim[2], b_row_bytes;
  int64_t b_box[2], b_boxes;
  int64_t d_grid_stride[2];             /* D offset step per tile along M and along N */
  int64_t d_elem_stride[2];             /* D offset step per row and per column */
  uint32_t instr_desc;                  /* tensor-core instruction descriptor */
  int32_t vector_epilogue;              /* 1 when 16-byte C/D accesses are legal */
  int32_t variant;                      /* the kernel variant (see gb_set_kernel_variant) */
} gb_gemm_plan;

gb_status gb_gemm_make_plan(int dtype, int64_t M, int64_t N, int64_t K, int64_t lda, int majorA,
                            int64_t ldb, int majorB, gb_gemm_plan* plan);

/* Robustness knobs (process-wide, read when a call launches, so a change made while other
   threads launch reaches some of their calls and not others):
   the limit on every in-kernel wait, in nanoseconds (0 restores the 2 s default), and a
   test hook that makes the copy stage skip the k-block with the given running index
   (-1 disables), so that the consumer's bounded wait runs out and the timeout path is
   exercised without faulting the device. */
gb_status gb_set_wait_timeout_ns(uint64_t ns);
gb_status gb_debug_skip_k_block(int64_t k_block);

/* Kernel variant for later calls (process-wide): 0 chooses by shape (the default, as
   described at the top of this file), 1 the single-CTA 128 x 256 kernel, 2 the CTA-pair
   256 x 256 kernel, 4 the single-CTA kernel with narrow 128 x 64 tiles and eight 24 KiB
   stages (for outputs with few columns; with a workspace, stream-K spreads K over the SMs),
   5 the CTA-pair kernel with 256 x 224 tiles (K-major B; with MN-major B it runs as 2), 6
   the CTA-pair kernel with 256 x 512 tiles (two 256-column MMAs per k-block of A, one
   accumulator filling Tensor Memory, eight epilogue warps), 7 the same with 256 x 448 tiles
   (two 224-column MMAs; K-major B; with MN-major B it runs as 6).  Block-scaled FP8 has no
   form 4, 5, 6 or 7 and runs as 2 (M > 128) or 1.  Every variant copies each tile into one CTA only
   (no copy multicast).  GB_ERR_INVALID_ARG for other values (3 included). */
gb_status gb_set_kernel_variant(int variant);

/* Test hook: evaluate, on the device, the D-offset map the epilogue of `variant` (1, 2, 4, 5,
   6 or 7) uses for tile (m_tile, n_tile) of an M x N problem: out[r*tile_n + c] = offset of
   in-tile element (r, c) (r < tile_m, c < tile_n, both from gb_gemm_make_plan), or -1
   when the element lies outside M x N.  out is a device buffer of tile_m * tile_n int64.
   Asynchronous on stream. */
gb_status gb_debug_epilogue_map(int variant, int64_t M, int64_t N, int64_t m_tile,
                                int64_t n_tile, int64_t* out, void* stream);

/* Test hook: copy one pipeline stage of operand A (which = 0) or B (which = 1) of the
   single-CTA kernel for (tile, k_block) into shared memory exactly as its copy stage
   does, then write the raw shared-memory bytes to `out` (a device buffer of 16384 bytes
   for A, 32768 for B); `tile` is the M-tile for A and the N-tile for B.  Checks the
   tensor-copy geometry and the 128-byte swizzle. */
gb_status gb_debug_stage_bytes(int dtype, int which, int64_t M, int64_t N, int64_t K,
                               const void* A, int64_t lda, int majorA,
                               const void* B, int64_t ldb, int majorB,
                               int64_t tile, int64_t k_block, void* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H */
