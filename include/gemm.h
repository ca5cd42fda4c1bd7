/*
 * gemm.h -- C ABI of the GB300 dense GEMM library (libgemm.so).
 *
 * The operation is the dense matrix multiply that "bare-metal-bard"
 * (ethanyanxu.com) builds as a ladder of kernels and uses for every projection
 * of a small GPT (first and second paragraphs), in its BLAS form
 *
 *     C = alpha * op(A) * op(B) + beta * C
 *
 * computed by gemm_run in one of seven modes (gemm_mode_t): exact FP32 on
 * the CUDA cores, TF32 on the tensor cores (the mode the page's tensor-core
 * kernel uses, first paragraph), BF16 inputs on the tensor cores, or 8-bit
 * float inputs on the tensor cores in four modes -- E4M3 x E4M3, E5M2 x E5M2
 * and the two mixed pairs ("Tensor Cores: Matrix Instructions, Swizzling
 * and FP8, Measured" and "Low-Precision Kernels: INT4, INT8 and FP8
 * Matmuls, Measured" name the formats).  Three more modes, the block-scaled
 * MXFP8 (E4M3, E5M2) and NVFP4, run through gemm_run_block_scaled.  Every
 * mode accumulates in FP32 and writes FP32.  gemm_run_epilogue adds a bias,
 * GELU or GELU' to the product, and gemm_attention_forward is the fused
 * attention forward of the same GPT (third paragraph).
 *
 * Layout (all matrices row-major, element (r, c) at base[r * ld + c]):
 *   op(A) is M x K.  transA == 0: A is stored M x K, lda >= max(K, 1).
 *                    transA == 1: A is stored K x M, lda >= max(M, 1).
 *   op(B) is K x N.  transB == 0: B is stored K x N, ldb >= max(N, 1).
 *                    transB == 1: B is stored N x K, ldb >= max(K, 1).
 *   C is M x N float, ldc >= max(N, 1).
 *   A and B are float in GEMM_MODE_FP32 and GEMM_MODE_TF32 and bfloat16
 *   (raw 16-bit patterns) in GEMM_MODE_BF16.  In TF32 mode the fp32 operands
 *   are passed to the tensor cores unchanged; the hardware drops their 13 low
 *   mantissa bits.  The TF32 tensor-core instruction reads K-major operands
 *   only, so in TF32 mode an operand stored with M (or N) contiguous (A with
 *   transA == 1, B with transB == 0) is first transposed into the workspace.
 *   In the FP8 modes, A and B hold 8-bit codes of the OCP 8-bit
 *   floating-point formats: E4M3 (1 sign, 4 exponent bits with bias 7, 3
 *   mantissa bits, no infinities, S.1111.111 = NaN, largest magnitude 448)
 *   or E5M2 (5 exponent bits with bias 15, 2 mantissa bits, infinities and
 *   NaNs as in IEEE 754, largest magnitude 57344), each operand in the
 *   format its mode names; there is no per-block scale, so per-tensor scale
 *   factors go into alpha.  The FP8 kernels read K-major operands (A
 *   stored M x K, B stored N x K, the weights of a linear layer as usually
 *   kept) in place; an FP8 operand stored MN-major is first transposed into
 *   the workspace, as in TF32 mode.
 *
 * Ownership: the caller owns A, B and C, which are device memory.  A handle
 * owns its device properties, a device status word (with, beside it, the
 * per-tile arrival counters of the FP32 kernel's stream-K schedule, zero
 * between calls) and a scratch workspace (split-K partial sums, re-packed
 * and transposed operands) that grows on demand and is freed by
 * gemm_destroy.  A handle is bound to the device that was current at
 * gemm_create and must not be used from two streams at the same time.
 *
 * Errors: every call returns a status and never throws.  Arguments are checked
 * before anything is launched; a failed check launches nothing and leaves C
 * untouched.  Launch failures are reported as GEMM_ERR_CUDA.  There is no
 * fallback to the CPU or to another library.
 */
#ifndef DENSE_GEMM_GB300_GEMM_H
#define DENSE_GEMM_GB300_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_handle_s* gemm_handle_t;

typedef enum {
  GEMM_MODE_FP32 = 0, /* fp32 operands, FFMA on CUDA cores, exact fp32 products */
  GEMM_MODE_TF32 = 1, /* fp32 operands, tcgen05 kind::tf32, fp32 accumulate   */
  GEMM_MODE_BF16 = 2, /* bf16 operands, tcgen05 kind::f16, fp32 accumulate    */
  GEMM_MODE_FP8_E4M3 = 3,      /* e4m3 A and B, tcgen05 kind::f8f6f4, fp32 accumulate;
                                  K-major operands read in place (every FP8 mode)   */
  GEMM_MODE_FP8_E5M2 = 4,      /* e5m2 A and B                                          */
  GEMM_MODE_FP8_E4M3_E5M2 = 5, /* e4m3 A, e5m2 B                                        */
  GEMM_MODE_FP8_E5M2_E4M3 = 6, /* e5m2 A, e4m3 B                                        */
  /* Block-scaled modes, gemm_run_block_scaled only (gemm_run refuses them): */
  GEMM_MODE_MXFP8_E4M3 = 7,    /* e4m3 A and B, one E8M0 scale per 32 K elements,
                                  tcgen05 kind::mxf8f6f4 block_scale                   */
  GEMM_MODE_MXFP8_E5M2 = 8,    /* e5m2 A and B, E8M0 scales per 32 K                   */
  GEMM_MODE_NVFP4 = 9          /* e2m1 A and B packed two per byte, one UE4M3 scale per
                                  16 K elements, tcgen05 kind::mxf4nvf4 block_scale    */
} gemm_mode_t;

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_VALUE = 1, /* null handle/pointer, bad mode or flag, negative size, ld too small */
  GEMM_ERR_NOT_SUPPORTED = 2, /* device is not sm_103 / sm_100 class, or option not available     */
  GEMM_ERR_MISALIGNED = 3,    /* a pointer is not aligned to its element size                        */
  GEMM_ERR_CUDA = 4,          /* a CUDA runtime or driver call failed                                */
  GEMM_ERR_ALLOC = 5,         /* device memory for the handle's workspace could not be allocated    */
  GEMM_ERR_DEVICE_TIMEOUT = 6, /* a kernel gave up a bounded wait and set the device status word     */
  GEMM_ERR_TOO_LARGE = 7       /* the problem exceeds gemm_run_small_m_noalloc's limit (M > 16)      */
} gemm_status_t;

/* Kernel families the planner chooses among (gemm_set_option/GEMM_OPT_FAMILY). */
typedef enum {
  GEMM_FAMILY_AUTO = 0,
  GEMM_FAMILY_SIMT = 1,   /* register-tiled FFMA kernel (GEMM_MODE_FP32 only)           */
  GEMM_FAMILY_TC = 2,     /* persistent TMA + tcgen05 kernel (TF32/BF16/FP8)             */
  GEMM_FAMILY_SKINNY = 3, /* HBM-bound small-M kernels, M <= 16 (TF32/BF16/FP8)         */
  GEMM_FAMILY_ATTENTION = 4 /* the fused attention kernel (gemm_attention_forward)        */
} gemm_family_t;

typedef enum {
  GEMM_OPT_FAMILY = 1,   /* value: gemm_family_t; AUTO lets the planner choose            */
  GEMM_OPT_SPLIT_K = 2,  /* value: 0 = planner's choice, n >= 1 = force n slices of K      */
  GEMM_OPT_TILE_N = 3,   /* value: 0 = planner's choice; TC: 128, 192, 224 or 256 (224 and,
                            for pairs, 192 need a K-major B in BF16); SIMT: 128 or 256    */
  GEMM_OPT_PRETRANSPOSE = 4, /* SIMT: 0 = planner's choice (K-contiguous operands transposed,
                                misaligned ones re-packed into the workspace first), 1 = never
                                (operands read in place), 2 = always transpose.  TF32: 2 also
                                transposes an MN-major A that the 128-column kernel would
                                otherwise move into TMEM itself (0 and 1: it does)          */
  GEMM_OPT_PAIR = 5,         /* TC: CTA pairs issuing one 256-row MMA (tcgen05 cta_group::2;
                                tiles of 192 or more columns, two or more rows of tiles; each
                                CTA stages half of every B tile).  0 = wherever the tile width
                                and B layout allow, 1 = never                                 */
  GEMM_OPT_WAIT_LIMIT_US = 6, /* TC: how long (microseconds) a wait of the persistent tcgen05
                                 kernel on one of its pipeline barriers may last before the
                                 kernel gives up, records GEMM_ERR_DEVICE_TIMEOUT in the device
                                 status word and returns.  0 = the default, 2 seconds; at most
                                 60 s.  A limit shorter than the call's own stages take makes
                                 correct calls time out.                                       */
  GEMM_OPT_FAULT_SKIP_STAGE = 7, /* TC, a test hook for the bounded-wait path: n > 0 makes the
                                   first CTA's TMA producer of the persistent tcgen05 kernel
                                   issue no copies for the n-th pipeline stage it takes, so
                                   that the MMA's wait for that stage runs out (after the
                                   GEMM_OPT_WAIT_LIMIT_US limit); the kernel then drains its
                                   copies and MMAs in flight, frees its TMEM and returns, C is
                                   undefined, and gemm_check_device reports
                                   GEMM_ERR_DEVICE_TIMEOUT.  Forces one CTA per tile (no pairs).
                                   0 = off (the default).  Nothing faults or hangs.             */
  GEMM_OPT_SK_FIXUP = 8       /* SIMT stream-K: how the partial tiles are summed.  0 = planner's
                                 choice (by the last CTA to finish a part of each tile when
                                 every tile is cut into a few long parts, else by a separate
                                 fixup kernel), 1 = always the fixup kernel, 2 = by the last CTA
                                 wherever the tiles cut into parts number at most 1024.  The
                                 sums are the same either way (ascending k order).            */
} gemm_option_t;

/* Elementwise work fused into the GEMM's epilogue (gemm_run_epilogue), the
 * variants a transformer layer's projections need ("bare-metal-bard", second
 * paragraph: a GPT whose every matmul, GELU and layernorm kernel is written
 * from scratch).  GELU is the function's definition, x * Phi(x) with the
 * exact error function (the page names GELU without a variant). */
typedef enum {
  GEMM_ACT_NONE = 0,  /* C = alpha*op(A)*op(B) + beta*C + bias                          */
  GEMM_ACT_GELU = 1,  /* C = GELU(alpha*op(A)*op(B) + beta*C + bias): a forward layer     */
  GEMM_ACT_DGELU = 2  /* C = (alpha*op(A)*op(B) + beta*C) * GELU'(Z): the gradient through
                         a GELU whose input Z (M x N) was kept from the forward pass      */
} gemm_activation_t;

typedef struct {
  int32_t activation;  /* gemm_activation_t */
  int32_t reserved;
  const float* bias;   /* NONE / GELU: N floats added to every row of the result, or NULL;
                          must be NULL for DGELU. Device memory, 4-byte aligned.          */
  const float* aux;    /* DGELU: Z, M x N row-major with leading dimension ld_aux (>= N);
                          ignored otherwise. Device memory, 4-byte aligned.              */
  int64_t ld_aux;
} gemm_epilogue_t;

/* What the last successful gemm_run on a handle launched. */
typedef struct {
  int32_t family;        /* gemm_family_t actually used (0 when nothing was launched) */
  int32_t tile_m, tile_n, tile_k;
  int32_t split_k;       /* slices of K (1 = no split) */
  int32_t stages;        /* shared-memory pipeline depth */
  int32_t grid;          /* CTAs of the main kernel */
  int32_t kernels;       /* kernels launched by the call */
  int32_t packed;        /* bit 0: A re-packed (or transposed), bit 1: B, into the workspace */
  int32_t schedule;      /* 0 one unit per tile, 1 split-K slices, 2 stream-K (SIMT),
                            3 whole tiles then K slices for the last rows of tiles (TC) */
  int32_t cluster;       /* TC: CTAs per cluster (2 = CTA pairs); small M: K slices per cluster */
  int32_t pair_mma;      /* TC: 1 when each CTA pair issues one 256-row MMA (tcgen05 cta_group::2) */
  int32_t epilogue_fused; /* gemm_run_epilogue: 1 when the GEMM kernel itself applied the epilogue */
  int32_t sk_fixup;      /* SIMT stream-K: 1 partial tiles summed by a separate fixup kernel,
                            2 by the last CTA to finish a part of each tile (0 otherwise) */
  int32_t reserved[2];
} gemm_plan_t;

/* Create a handle on the current device.  Reads the device properties and
 * allocates the 4-byte device status word.  *out is set to NULL on failure. */
gemm_status_t gemm_create(gemm_handle_t* out);

/* Free the handle, its status word and its workspace.  Synchronizes the
 * device first so that no launched kernel still uses the workspace.
 * A NULL handle is GEMM_ERR_INVALID_VALUE. */
gemm_status_t gemm_destroy(gemm_handle_t h);

/* C = alpha * op(A) * op(B) + beta * C on `stream` (a cudaStream_t; NULL is
 * the legacy default stream).  Asynchronous: returns once the kernels are
 * enqueued.  M == 0 or N == 0 is a no-op.  K == 0 or alpha == 0 gives
 * C = beta * C without reading A or B.  beta == 0 writes C without reading it
 * (a NaN in C does not propagate).  C must not overlap A or B.  The workspace
 * may grow (cudaMalloc) on the first call that needs a larger one.
 *
 * Small M (M <= 16, transA == 0, TF32/BF16/FP8) with fewer than two waves of
 * 128-column weight tiles runs one kernel that splits K across the CTAs of a
 * thread-block cluster and sums the slices in distributed shared memory (no
 * workspace).  It is launched with programmatic dependent launch: its set-up
 * and an L2 prefetch of the weights may overlap the end of the previous
 * kernel in `stream`, but it reads and writes no memory before that kernel
 * has completed, so stream order is kept. */
gemm_status_t gemm_run(gemm_handle_t h, int mode, int transA, int transB,
                       int64_t M, int64_t N, int64_t K, float alpha,
                       const void* A, int64_t lda, const void* B, int64_t ldb,
                       float beta, float* C, int64_t ldc, void* stream);

/* gemm_run with the elementwise epilogue `*ep` applied to every element of
 * the result, once, after split-K or stream-K partial sums are added.  In
 * TF32 and BF16 mode with A read K-major (transA == 0, or an A the plan
 * transposes) the tensor-core kernel applies it itself between its
 * accumulator load and its store (and the slice reduction for rows whose K
 * is split); otherwise it is applied inside the split-K reduction when the
 * call has one that writes all of C, or in one pass over C right after the
 * GEMM, in the same stream.  GELU is computed as x * Phi(x) with Phi from
 * the Abramowitz-Stegun 7.1.26 approximation of erfc (|error| <= 1.5e-7).
 * The
 * bias and Z are read, never written; C must not overlap them.  ep == NULL
 * is gemm_run.  With K == 0 or alpha == 0 the product is zero and the
 * epilogue still applies to beta*C.  Errors: GEMM_ERR_INVALID_VALUE for an
 * unknown activation, a bias with DGELU, DGELU without Z or with
 * ld_aux < N; GEMM_ERR_MISALIGNED for a bias or Z not 4-byte aligned; the
 * other checks are gemm_run's. */
gemm_status_t gemm_run_epilogue(gemm_handle_t h, int mode, int transA, int transB,
                                int64_t M, int64_t N, int64_t K, float alpha,
                                const void* A, int64_t lda, const void* B, int64_t ldb,
                                float beta, float* C, int64_t ldc,
                                const gemm_epilogue_t* ep, void* stream);

/* The argument checks gemm_run performs, without a handle or a device.
 * Returns GEMM_OK or the status gemm_run would return for these arguments
 * (A and B are checked only when K > 0 and alpha != 0, since only then are
 * they read). */
gemm_status_t gemm_validate(int mode, int transA, int transB,
                            int64_t M, int64_t N, int64_t K, float alpha,
                            const void* A, int64_t lda, const void* B, int64_t ldb,
                            const float* C, int64_t ldc);

/* Set a planner option (gemm_option_t) for later calls on this handle. */
gemm_status_t gemm_set_option(gemm_handle_t h, int option, int64_t value);

/* Copy the plan of the last successful gemm_run into *out. */
gemm_status_t gemm_get_plan(gemm_handle_t h, gemm_plan_t* out);

/* Synchronize `stream`, then read and clear the handle's device status word.
 * Returns GEMM_ERR_DEVICE_TIMEOUT if a kernel abandoned a bounded wait since
 * the last check (its output is then undefined), GEMM_ERR_CUDA if the stream
 * reports an error, GEMM_OK otherwise. */
gemm_status_t gemm_check_device(gemm_handle_t h, void* stream);

/* Launch, on `stream`, an empty kernel with the launch configuration of the
 * main kernel of this handle's last successful gemm_run (its grid, block,
 * dynamic shared memory, cluster size and programmatic dependent launch;
 * not the transposes, re-packs or reductions around it).  It reads and
 * writes no memory.  Timed like the GEMM, it gives the cost of launching,
 * placing and retiring that configuration: the floor under the call's time
 * (the "identity null" that the "gpu kernels" write-up on devpost times
 * beside every shape, section "How we know the numbers are real").  GEMM_ERR_INVALID_VALUE when the last
 * call launched no GEMM kernel (M, N or K zero, alpha zero) or none was made;
 * GEMM_ERR_CUDA when the launch fails. */
gemm_status_t gemm_launch_null(gemm_handle_t h, void* stream);

/* A calibration kernel, not a GEMM (the source pages have no counterpart):
 * the FP32 fused multiply-add rate of this part, against which the FP32
 * mode is measured.  Launches, on `stream`, `grid` CTAs of 256 threads that
 * each run 16 independent FMA chains of `iters` steps in registers --
 * packed == 0: scalar fma.rn.f32; packed == 1: eight fma.rn.f32x2 pairs --
 * and store one float per thread to `out` (grid * 256 floats of device
 * memory, 4-byte aligned, owned by the caller).  FLOPs per launch =
 * grid * 256 * iters * 32; timed with events it gives the FP32 roof.
 * GEMM_ERR_INVALID_VALUE for grid outside [1, 2^20], iters < 1, a null
 * `out` or packed not 0/1; GEMM_ERR_CUDA when the launch fails. */
gemm_status_t gemm_launch_fma_peak(int packed, int64_t grid, int64_t iters, float* out, void* stream);

/* Bytes of the fixed device array that gemm_run_small_m_noalloc uses as its
 * only scratch memory (one array per device, held until the process exits). */
#define GEMM_NOALLOC_SCRATCH_BYTES (8u << 20)

/* The small-M product of gemm_run (M <= 16: a few token rows against a weight
 * matrix, as in one decode step) for callers that cannot allocate device
 * memory.  The source pages have no counterpart to this call; it exists for
 * code that runs where cudaMalloc is unavailable or forbidden -- an inference
 * runtime that owns every allocation through its own pool, a plug-in inside
 * another program's CUDA context, a loop that must never enter the allocator.
 * gemm_run cannot serve such callers because its handle allocates a status
 * word when created and a workspace when first used.
 *
 * The same product as gemm_run, within the mode's tolerance, but not the same
 * kernels: this call runs the persistent tcgen05 kernel in its swapped form
 * plus a separate kernel that sums the split-K partials, where gemm_run uses
 * the cluster kernel that sums its K slices in distributed shared memory.
 * A is stored M x K (transA is always 0), B is K x N (transB == 0) or N x K
 * (transB == 1), mode is GEMM_MODE_BF16 or GEMM_MODE_TF32 (TF32 needs
 * transB == 1), C is M x N fp32.  The caller passes inputs and outputs; the only scratch is a
 * fixed device array of GEMM_NOALLOC_SCRATCH_BYTES inside the library (the
 * device status word and the split-K partial sums).  The call makes no
 * cudaMalloc, no cudaFree and no allocating library call.
 *
 * Limits and errors: M > 16 gives GEMM_ERR_TOO_LARGE (the K-slice count is
 * lowered until the partial sums fit the array; one slice needs none); an
 * operand the
 * TMA unit cannot read in place (base not 16-byte aligned, row pitch not a
 * multiple of 16 bytes) gives GEMM_ERR_MISALIGNED; FP32 or FP8 mode, or TF32
 * with transB == 0, gives GEMM_ERR_NOT_SUPPORTED; the other checks are
 * gemm_run's.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  Every
 * call on a device shares the one array and leaves its contents behind: the
 * call clears the status word itself, and calls whose kernels overlap on the
 * GPU (different streams, no ordering between them) race on the array and
 * give undefined results.  A device-side wait that times out is recorded in
 * the array's status word; this call returns before its kernels run and
 * cannot report it: gemm_noalloc_check_device does, and must be called
 * before the next call on the device clears the word. */
gemm_status_t gemm_run_small_m_noalloc(int mode, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                                       const void* A, int64_t lda, const void* B, int64_t ldb,
                                       float beta, float* C, int64_t ldc, void* stream);

/* The check of gemm_check_device for gemm_run_small_m_noalloc, which has no
 * handle (no counterpart on the source pages either): synchronize `stream`,
 * then read and clear the status word in the library's fixed scratch array
 * of the current device.  Returns GEMM_ERR_DEVICE_TIMEOUT if a kernel of an
 * earlier gemm_run_small_m_noalloc call gave up a bounded wait (that call's
 * C is then undefined), GEMM_ERR_CUDA if the stream reports an error,
 * GEMM_OK otherwise.  Allocates nothing.  The next gemm_run_small_m_noalloc
 * call on the device clears the word, so check before it. */
gemm_status_t gemm_noalloc_check_device(void* stream);

/* Block-scaled low-precision product: C = alpha * (A . SA) * (B . SB)^T +
 * beta * C, where every run of `bs` consecutive K elements of a row shares
 * one scale.  The "Low-Precision Kernels: INT4, INT8 and FP8 Matmuls,
 * Measured" summary (vidyal.ai) names the MX and NVFP4 formats; their
 * definitions are the OCP Microscaling specification's and NVIDIA's NVFP4:
 *   GEMM_MODE_MXFP8_E4M3 / _E5M2: 8-bit E4M3 / E5M2 codes, bs = 32, E8M0
 *     scales (2^(e - 127); 0xFF is NaN);
 *   GEMM_MODE_NVFP4: E2M1 codes packed two per byte (the even element of a
 *     pair in the low nibble), bs = 16, UE4M3 scales (the E4M3 magnitude;
 *     the sign bit is ignored).  A per-tensor factor goes into alpha.
 * A is stored M x K and B N x K (K contiguous in both, the weights of a
 * linear layer as usually kept), lda / ldb in elements (NVFP4: K, lda and
 * ldb even; a row is lda / 2 bytes); C is M x N fp32, ldc >= N.  SA and SB
 * are the scales of A (M x ceil(K / bs)) and B (N x ceil(K / bs)) in the
 * tiled layout gemm_block_scales_tile writes.  A partial last block is
 * allowed.  Served for the decode shape, M <= 16, by the small-M kernels (K
 * split across a thread-block cluster, or the persistent swapped form for
 * wide weights), and for M > 16 by the persistent kernel on 128 x 128
 * tiles; the scale atoms of every pipeline stage are copied into tensor
 * memory with tcgen05.cp.
 * Errors: GEMM_ERR_INVALID_VALUE for another mode, negative sizes, a null
 * pointer, lda or ldb < K, an odd K / lda / ldb in NVFP4;
 * GEMM_ERR_MISALIGNED when A, B, SA or SB is not 16-byte aligned
 * or a row of A or B is not a multiple of 16 bytes.  M == 0 or N == 0 is a
 * no-op; K == 0 or alpha == 0 gives C = beta * C.  Asynchronous on `stream`. */
gemm_status_t gemm_run_block_scaled(gemm_handle_t h, int mode, int64_t M, int64_t N, int64_t K, float alpha,
                                    const void* A, int64_t lda, const void* SA, const void* B, int64_t ldb,
                                    const void* SB, float beta, float* C, int64_t ldc, void* stream);

/* Bytes of the tiled scale layout for a rows x blocks scale matrix:
 * ceil(rows / 128) * 4 * ceil(blocks / 16) * 512; -1 for negative sizes.
 * Host only (no device needed). */
int64_t gemm_block_scales_tiled_bytes(int64_t rows, int64_t blocks);

/* Rewrite block scales S (rows x blocks bytes, row-major, leading dimension
 * lds >= blocks) into T (gemm_block_scales_tiled_bytes bytes, 16-byte
 * aligned, device memory) in the layout the tensor cores read them in: for
 * each tile of 128 rows, groups of four blocks as 512-byte atoms, row r of
 * the tile and block j of the group at byte 16 * (r % 32) + 4 * (r / 32) +
 * j, atoms ordered by group, tiles one after another, 4 * ceil(blocks / 16)
 * atoms per tile; every byte past the matrix is 0.  No counterpart on the
 * source pages (a layout of this library's kernels).  Asynchronous on
 * `stream`. */
gemm_status_t gemm_block_scales_tile(int64_t rows, int64_t blocks, const void* S, int64_t lds, void* T,
                                     void* stream);

/* Scaled dot-product attention, forward, fused: for each of `problems`
 * independent problems (a batch element and a head) and each query row i,
 *     O[i] = sum_j softmax_j(scale * q_i . k_j) v_j
 * over the keys j that row i sees (j <= i when causal = 1, every j < T when
 * causal = 0).  "bare-metal-bard" (third paragraph) reports such a fused,
 * FlashAttention-style kernel for its GPT's causal self-attention: the score
 * matrix is never written out; a running maximum and sum are carried from
 * one block of keys to the next, so memory grows linearly with T.  Here the
 * scores of 128 queries x 128 keys live in tensor memory (tcgen05), the
 * probabilities are rounded to bf16 for the P V product, and the row sums
 * are kept in fp32.
 * Q, K, V: bfloat16, [problems][T][Dh] contiguous (row i of problem p at
 * element (p * T + i) * Dh); O: float32 of the same shape.  All device
 * memory owned by the caller, 16-byte aligned.  Dh must be 64 (the GPT's
 * head size); scale is usually 1 / sqrt(Dh).
 * Errors: GEMM_ERR_INVALID_VALUE for a null handle or pointer, negative
 * sizes, causal not 0/1, a non-finite scale or more than 2^31 - 1 query
 * tiles; GEMM_ERR_NOT_SUPPORTED for Dh != 64; GEMM_ERR_MISALIGNED for a
 * pointer not 16-byte aligned.  problems == 0 or T == 0 is a no-op.
 * Asynchronous on `stream`; the handle's device status word records a
 * bounded wait that gave up (gemm_check_device).  gemm_get_plan reports
 * family GEMM_FAMILY_ATTENTION and the grid. */
gemm_status_t gemm_attention_forward(gemm_handle_t h, int64_t problems, int64_t T, int64_t Dh, int causal,
                                     float scale, const void* Q, const void* K, const void* V, float* O,
                                     void* stream);

/* A static string naming a status code. */
const char* gemm_status_string(gemm_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_GB300_GEMM_H */
