/*
 * rg.h - activation-gradient OUT_PROD through a resident quantized or
 * half-precision weight, for NVIDIA GB300 (sm_103a).
 *
 * The operation.  The llama.cpp fork's PR "cuda: out_prod accepts a quantized
 * src0" (commit message and section "What") gives the backward of
 * mul_mat(W, x) with respect to x as out_prod(W, grad^T), taken over every
 * quantized, F16 and BF16 src0 with F32 src1/dst.  With W stored as N rows of
 * K values (blocks run along K) and the incoming gradient dY of shape [T, N]:
 *
 *     dX[t, k] = beta * dX[t, k] + sum_{n < N} dY[t, n] * deq(W)[n, k]
 *
 * deq() is the block decode of the weight's storage type (rg_dequant).  The
 * PR's route copies deq(W) to a dense F32 pool buffer and runs SGEMM on it;
 * the Retrograd page "CUDA status", section "Limitations", adds a budgeted,
 * sliced version of that copy and an in-place decoder for small outputs.
 * This library instead decodes the packed blocks inside the GEMM, straight
 * into tensor-core operand tiles, so no dense copy of W ever exists.
 *
 * Conventions for every call below.
 *  - Pointers to data are DEVICE pointers (cudaMalloc / PyTorch storage) and
 *    stay owned by the caller; the library never frees or retains them.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Work is enqueued asynchronously; nothing here synchronizes
 *    except rg_check and the blocking variants named as such.
 *  - Arguments are validated on the host before anything is enqueued; on any
 *    error status nothing has been launched and outputs are untouched.
 *  - Layouts: W is N rows of rg_row_bytes(wtype, K) bytes each, rows
 *    contiguous; dY is [T, N] row-major F32; dX and `out` are [T, K] and
 *    [N, K] row-major F32.  W, dY, dX and out must be 16-byte aligned.
 *  - Sizes: 0 <= T, N, K <= 2^31 - 1.  T == 0 or K == 0 is an empty output
 *    (RG_OK, nothing launched, pointers may be NULL).  N == 0 is an empty
 *    contraction: dX = beta * dX (dX = 0 when beta == 0).
 *  - K must be a multiple of 256 for the quantized types (whole 256-value
 *    tiles of every block type) and a multiple of 8 for F32, F16 and BF16
 *    (16-byte rows); otherwise RG_ERR_SHAPE.  On the tensor-core and small-T
 *    variants Q6_K and Q3_K also need K % 2048 == 0 and Q2_K K % 1024 == 0
 *    (16-byte aligned rows).
 *  - Every device-side wait is bounded (about 2 s); a wait that gives up
 *    records RG_ERR_TIMEOUT in a per-device status word that rg_check reads.
 *    The outputs of a call whose kernels gave up are undefined (partly
 *    written); the context stays usable.
 */
#ifndef RG_H
#define RG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight storage types (ggml's GGUF block types of the same names). */
typedef enum {
    RG_F16 = 1,   /* IEEE binary16, 2 B per value                                   */
    RG_BF16 = 2,  /* bfloat16, 2 B per value                                         */
    RG_Q8_0 = 3,  /* 34 B / 32 values: fp16 d, int8 q[32]; value d*q                 */
    RG_Q4_0 = 4,  /* 18 B / 32 values: fp16 d, 16 B nibbles (lo = j, hi = j+16);
                     value d*(q-8)                                                   */
    RG_Q4_K = 5,  /* 144 B / 256 values: fp16 d, fp16 dmin, 12 B of 6-bit (sc, m)
                     for 8 sub-blocks of 32, 128 B nibbles; value d*sc*q - dmin*m    */
    RG_Q4_1 = 6,  /* 20 B / 32 values: fp16 d, fp16 m, 16 B nibbles as Q4_0;
                     value d*q + m                                                   */
    RG_Q5_0 = 7,  /* 22 B / 32 values: fp16 d, 4 B qh (bit i of the little-endian
                     word = fifth bit of value i), 16 B nibbles; value d*(q-16)      */
    RG_Q5_1 = 8,  /* 24 B / 32 values: fp16 d, fp16 m, 4 B qh, 16 B nibbles;
                     value d*q + m                                                   */
    RG_Q5_K = 9,  /* 176 B / 256 values: the Q4_K header, 32 B qh (bit 2c / 2c+1 of
                     qh[l] = fifth bit of value 64c+l / 64c+32+l), 128 B nibbles;
                     value d*sc*q - dmin*m                                           */
    RG_Q6_K = 10, /* 210 B / 256 values: ql[128] low nibbles, qh[64] bit pairs,
                     int8 scales[16], fp16 d; value d*sc[v/16]*(q-32).  Rows of
                     210*K/256 bytes are 16-byte aligned only when K % 2048 == 0,
                     which the tensor-core and small-T variants need (else
                     RG_ERR_SHAPE; RG_VARIANT_AUTO then runs the SIMT variant)   */
    RG_F32 = 11,  /* IEEE binary32, 4 B per value.  The tensor-core variants round W
                     and dY to bf16 (F32 range, relative error at most 2^-9 each)
                     in the workspace; the other variants use the F32 values    */
    RG_Q2_K = 12, /* 84 B / 256 values: scales[16] (lo nibble sc, hi nibble m),
                     qs[64], fp16 d, fp16 dmin.  Value 128h+32j+16s+l: bits 2j..2j+1
                     of qs[32h+16s+l], scales byte 8h+2j+s; value d*sc*q - dmin*m.
                     Rows 16-byte aligned only when K % 1024 == 0 (as Q6_K)     */
    RG_Q3_K = 13, /* 110 B / 256 values: hmask[32], qs[64], 12 B of sixteen 6-bit
                     scales, fp16 d.  Value 128h+32j+16s+l: low bits as Q2_K, minus
                     4 unless bit 4h+j of hmask[16s+l] is set; value d*(sc-32)*q.
                     Rows 16-byte aligned only when K % 2048 == 0 (as Q6_K)     */
    RG_MXFP4 = 14,/* 17 B / 32 values: E8M0 scale byte e, 16 B nibbles as Q4_0, each
                     an E2M1 code (OCP microscaling: bit 3 sign, 2 exponent bits,
                     1 mantissa bit: 0, 0.5, 1, 1.5, 2, 3, 4, 6); value
                     E2M1(q) * 2^(e-127) (e = 255: NaN).  Rows 16-byte aligned
                     only when K % 512 == 0, which the tensor-core and small-T
                     variants need.  The tensor-core variants round the values
                     to fp16: block scales outside 2^-24..2^15 lose them       */
    RG_NVFP4 = 15 /* 36 B / 64 values: four FP8 E4M3 scale bytes d[s] (sign, 4
                     exponent bits with bias 7, 3 mantissa bits; 0x7f NaN), one
                     per 16 values, then 32 B of E2M1 codes (as MXFP4): the 16
                     values of d[s] in bytes 4+8s .. 11+8s, value 16s+j (j < 8)
                     the low nibble of byte 4+8s+j, 16s+j+8 its high nibble;
                     value E2M1(q) * E4M3(d[s]).  NVIDIA's second-level,
                     tensor-wide F32 scale is not part of the block (fold it
                     into dY or the result).  Every value is exact in fp16
                     (2^-10 .. 2688), so the tensor-core operands are too    */
} rg_wtype;

typedef enum {
    RG_OK = 0,
    RG_ERR_ARG = -1,     /* NULL pointer where data is needed, negative or too large size */
    RG_ERR_TYPE = -2,    /* unknown wtype, or unknown variant                              */
    RG_ERR_SHAPE = -3,   /* K not a multiple of 256 (quantized) or 8 (F32/F16/BF16); Q6_K or
                            Q3_K with K % 2048 != 0, Q2_K with K % 1024 != 0, MXFP4 with
                            K % 512 != 0, on a tensor-core or small-T variant                */
    RG_ERR_ALIGN = -4,   /* W, dY, dX or out not 16-byte aligned                           */
    RG_ERR_CUDA = -5,    /* a CUDA runtime/driver call or a launch failed                  */
    RG_ERR_TIMEOUT = -6, /* a bounded device-side wait gave up (reported by rg_check)      */
    RG_ERR_RANGE = -7    /* a finite dY value lay outside the 16-bit operand kind's range
                            (fp16: |dY| >= 65520) and became inf in the tensor-core
                            operand copy: the call's dX holds inf or NaN (reported by
                            rg_check; rerun with RG_VARIANT_SIMT32 or a scaled dY)       */
} rg_status;

/* Kernel variants of rg_out_prod_variant. */
typedef enum {
    RG_VARIANT_AUTO = 0,   /* the shape dispatcher's choice (what rg_out_prod runs)        */
    RG_VARIANT_TC = 1,     /* fused decode + tcgen05 tensor-core GEMM, fp16/bf16 operands,
                              F32 accumulation in tensor memory                             */
    RG_VARIANT_SMALLT = 2, /* small-T, weight-bandwidth-bound: TMA streams row stages
                              of W; exact F32 decode and F32 FMA with up to 8 dY rows
                              (Q4_K, Q8_0: the weight integers as exact fp16 operands of
                              warp-level MMAs, dY*scale rounded to fp16 once, F32
                              accumulation); rows
                              split over many CTAs, partial sums added in a fixed order
                              by a second kernel (N <= 256: one kernel writes dX)     */
    RG_VARIANT_SIMT32 = 3, /* exact F32 decode and F32 FMA with blocked accumulation: the
                              full-precision variant (slow; a correctness reference)        */
    RG_VARIANT_TC_SINGLE = 4, /* RG_VARIANT_TC with one-CTA 128 x 128 tiles                */
    RG_VARIANT_TC_PAIR = 5    /* RG_VARIANT_TC with two-CTA (cta_group::2) 256 x 256 tiles  */
} rg_variant;

/*
 * dX = beta * dX + dY . deq(W)   (see the top of this file).
 *
 * wtype: rg_wtype.  W: N * rg_row_bytes(wtype, K) bytes.  dY: [T, N] F32.
 * dX: [T, K] F32, read only when beta != 0 (with beta == 0 its old contents,
 * NaN included, are ignored).  The variant is chosen from (wtype, T, N, K);
 * the environment variable RG_VARIANT=auto|tc|tc1|tc2|smallt|simt32, read
 * once per process, overrides that choice.  Asynchronous on `stream`.
 *
 * Scratch: the tensor-core variant converts dY once to fp16/bf16, and the
 * small-T variant writes per-CTA partial sums, in a device workspace of
 * rg_workspace_bytes() bytes.  rg_out_prod takes it
 * stream-ordered from a per-device memory pool owned by the library
 * (cudaMallocFromPoolAsync / cudaFreeAsync on `stream`); the pool keeps its
 * memory, so only the first call of a given size reaches the driver.  Use
 * rg_out_prod_ws to supply the workspace and allocate nothing at all.
 */
int rg_out_prod(int wtype, const void* W, int64_t N, int64_t K,
                const float* dY, int64_t T, float* dX, float beta, void* stream);

/* rg_out_prod with an explicit variant (rg_variant; RG_VARIANT_AUTO = dispatch;
 * RG_VARIANT_TC picks its tile shape from the problem, TC_SINGLE / TC_PAIR
 * force one).  RG_VARIANT ignored.  Same contract as rg_out_prod. */
int rg_out_prod_variant(int variant, int wtype, const void* W, int64_t N, int64_t K,
                        const float* dY, int64_t T, float* dX, float beta, void* stream);

/* Device workspace bytes that rg_out_prod_ws needs for this call (0 if none). */
size_t rg_workspace_bytes(int variant, int wtype, int64_t N, int64_t K, int64_t T);

/* rg_out_prod_variant with a caller-owned device workspace of at least
 * rg_workspace_bytes(variant, wtype, N, K, T) bytes, 256-byte aligned
 * (RG_ERR_ARG if smaller, RG_ERR_ALIGN if misaligned).  Allocates nothing and
 * does not synchronize.  Calls that share a workspace must be ordered on
 * one stream. */
int rg_out_prod_ws(int variant, int wtype, const void* W, int64_t N, int64_t K,
                   const float* dY, int64_t T, float* dX, float beta,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of the fixed device scratch behind rg_out_prod_noalloc. */
#define RG_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * rg_out_prod for callers that cannot allocate device memory.  (This entry
 * point has no counterpart in the pages this library follows; it is a
 * convenience of this implementation.)
 *
 * Who needs it: code that must not call cudaMalloc or a memory pool at all,
 * e.g. a runtime that owns every byte of device memory through its own
 * allocator and forbids others, a callback or real-time path that cannot
 * afford the allocator's locking or implicit device synchronization, or an
 * embedding that runs under an allocation guard.  rg_out_prod takes its dY
 * workspace from a memory pool; rg_out_prod_ws needs a buffer the caller
 * allocated.  This call needs neither: the tensor-core path converts dY into
 * a fixed scratch array compiled into the library (RG_NOALLOC_SCRATCH_BYTES,
 * 32 MiB), which every GPU that loads the library keeps until the process
 * exits.  It calls no cudaMalloc, cudaFree or pool routine.
 *
 * Same arguments, layouts and results as rg_out_prod (same kernels, same
 * variant choice), except that its tensor-core plans never share the last
 * tiles' contraction over all units (stream-K): those partial slabs would
 * not fit the scratch.  Where rg_out_prod would, the two results differ in
 * summation order only, both within the same error bound.  Limits: when the
 * chosen variant is a tensor-core one, the 16-bit copy of dY, T * (N rounded
 * up to 8) * 2 bytes (plus any split partial sums), must fit the scratch,
 * else RG_ERR_ARG and nothing is launched (e.g. T = 2048 allows N <= 8192).
 * The scratch is shared by every call on a device and keeps the last call's
 * contents (each call overwrites what it reads; nothing needs clearing), so
 * calls that may overlap on the GPU (different streams, or different host
 * threads) race on it: order them on one stream.  The first call on a device
 * looks up the scratch's device address (a runtime query, no allocation);
 * make that first call before any stream capture.
 */
int rg_out_prod_noalloc(int wtype, const void* W, int64_t N, int64_t K,
                        const float* dY, int64_t T, float* dX, float beta, void* stream);

/*
 * The general form: `batch` independent products with their own strides.
 * For b < batch,
 *     dX_b[t, k] = beta * dX_b[t, k] + sum_n dY_b[t, n] * deq(W_b)[n, k]
 * with W_b = W + b * w_batch_bytes (0: one W shared by every batch),
 * dY_b[t, n] = dY[b * dy_batch + t * dy_t + n * dy_n] and
 * dX_b[t, k] = dX[b * dx_batch + t * dx_t + k]   (strides in elements).
 * dY may come transposed (dy_t = 1, dy_n = T), as ggml's out_prod(W, grad^T)
 * receives grad^T as a strided view: the llama.cpp fork's PR "cuda: out_prod
 * accepts a quantized src0" runs ggml's OUT_PROD paths for a plain or
 * transposed src1 and its batch dimensions on the dense copy ("What",
 * "Measured").  Rules: dy_t, dy_n >= 1; dx_t >= K and a multiple of 4;
 * w_batch_bytes a multiple of 16 and dx_batch of 4; dY 16-byte aligned when
 * its rows are contiguous (dy_n == 1, dy_t == N), else 4-byte aligned; every
 * batch's W and dX 16-byte aligned (else RG_ERR_ALIGN / RG_ERR_ARG, checked
 * for every batch before anything is launched).  Batches that stack into
 * one taller dY and dX under a shared W run as one call; others run one
 * after another on `stream`.  The batches' dX regions must not overlap.
 * `variant` as for rg_out_prod_variant; batch == 0 is RG_OK.
 */
int rg_out_prod_ex(int variant, int wtype, const void* W, int64_t N, int64_t K,
                   int64_t w_batch_bytes, const float* dY, int64_t T, int64_t dy_t, int64_t dy_n,
                   int64_t dy_batch, float* dX, int64_t dx_t, int64_t dx_batch, int64_t batch,
                   float beta, void* stream);

/*
 * ggml's full OUT_PROD surface: two batch dimensions, and fewer weights than
 * batches, each weight serving a run of consecutive batches (the broadcast a
 * grouped projection needs, e.g. grouped-query attention's shared k/v
 * weights).  For i3 < n3, i2 < n2:
 *     dX_b[t, k] = beta * dX_b[t, k] + sum_n dY_b[t, n] * deq(W_b)[n, k],
 *     W_b = W + (i2 / (n2 / w_n2)) * w_s2 + (i3 / (n3 / w_n3)) * w_s3   (bytes),
 *     dY_b[t, n] = dY[i2 * dy_s2 + i3 * dy_s3 + t * dy_t + n * dy_n],
 *     dX_b[t, k] = dX[i2 * dx_s2 + i3 * dx_s3 + t * dx_t + k]            (elements).
 * This is the broadcast rule of ggml's out_prod (a weight batch count that
 * divides the gradient's, per dimension), whose CUDA route the llama.cpp
 * fork's PR "cuda: out_prod accepts a quantized src0" runs on the dense copy
 * and whose broadcasting cases its "Measured" section reports skipped.
 * Rules: w_n2, w_n3 >= 1 dividing n2, n3 (else RG_ERR_SHAPE); strides >= 0;
 * w_s2, w_s3 multiples of 16 and dx_s2, dx_s3 of 4 (else RG_ERR_ALIGN); the
 * row rules of rg_out_prod_ex for every batch, all checked before anything
 * is launched.  Consecutive batches (i2 fastest) that read the same weight
 * and whose dY and dX rows continue one another's run as one call with
 * more rows; the others in turn on `stream`.  The batches' dX regions must
 * not overlap.  n2 == 0 or n3 == 0 is RG_OK.
 */
int rg_out_prod_batched(int variant, int wtype, const void* W, int64_t N, int64_t K, int64_t w_n2,
                        int64_t w_n3, int64_t w_s2, int64_t w_s3, const float* dY, int64_t T,
                        int64_t dy_t, int64_t dy_n, int64_t dy_s2, int64_t dy_s3, float* dX,
                        int64_t dx_t, int64_t dx_s2, int64_t dx_s3, int64_t n2, int64_t n3,
                        float beta, void* stream);

/*
 * The forward mul_mat(W, x) through the same resident weight (the op whose
 * backward rg_out_prod is; llama.cpp fork PR "cuda: out_prod accepts a
 * quantized src0", commit message):
 *
 *     Y[t, n] = beta * Y[t, n] + sum_{k < K} X[t, k] * deq(W)[n, k]
 *
 * X: [T, K] F32, Y: [T, N] F32 (read only when beta != 0), both row-major
 * and 16-byte aligned; W as for rg_out_prod.  N must be a multiple of 8
 * (RG_ERR_SHAPE).  Two routes, chosen by the shape:
 *   - one or two rows of X with 16-byte aligned rows of W (see below): W
 *     is streamed once, each row's values decoded exactly to F32 and
 *     multiplied with X in F32 (|err| far below the bound that follows);
 *     one launch, no workspace;
 *   - otherwise X is rounded once to a 16-bit copy (fp16; bf16 for F32 and
 *     BF16 W) and the tensor-core kernel decodes W's blocks straight into
 *     its operand tiles, now contracting over the K values of each row, with
 *     F32 accumulation: |err| <= 5e-3 * sum_k |X||deq W| + 1e-7; no copy of
 *     deq(W) exists (F32 W: a bf16 copy of W, as rg_out_prod makes).  Rows
 *     that are not 16-byte aligned (Q6_K and Q3_K with K % 2048 != 0, Q2_K
 *     with K % 1024 != 0, MXFP4 with K % 512 != 0) instead decode deq(W)^T
 *     once per call into a transient 16-bit [K, N] copy (2*N*K bytes).
 * Workspace from the library's stream-ordered pool
 * (rg_mul_mat_workspace_bytes).  T == 0 or N == 0: nothing to do; K == 0:
 * Y = beta * Y.
 */
int rg_mul_mat(int wtype, const void* W, int64_t N, int64_t K, const float* X, int64_t T, float* Y,
               float beta, void* stream);

/* rg_mul_mat with its route named: RG_VARIANT_AUTO (rg_mul_mat's choice),
 * RG_VARIANT_TC (the tensor-core kernel, any T) or RG_VARIANT_SMALLT (W
 * streamed once per four rows of X, up to 262140 rows; RG_ERR_SHAPE beyond
 * that and for rows that are not 16-byte aligned).  Other variants:
 * RG_ERR_TYPE. */
int rg_mul_mat_variant(int variant, int wtype, const void* W, int64_t N, int64_t K, const float* X,
                       int64_t T, float* Y, float beta, void* stream);

/* Device workspace bytes one rg_mul_mat call of this shape takes from the
 * pool on the current device (0 for an invalid or empty shape, and for the
 * one-or-two-row route, which takes none). */
size_t rg_mul_mat_workspace_bytes(int wtype, int64_t N, int64_t K, int64_t T);

/*
 * The input gradient through the resident weight AND a low-rank adapter
 * (LoRA) trained beside it (llama.cpp fork PR "cuda: out_prod accepts a
 * quantized src0", commit message: a LoRA training on a resident quantized
 * base).  For the forward y = x deq(W)^T + scale * (x A^T) B^T:
 *
 *     dX = beta * dX + dY . deq(W) + scale * (dY . B) . A
 *
 * lora_a: A [rank, K] F32 row-major (the adapter's down projection);
 * lora_b: B [N, rank] F32 row-major (its up projection); both 16-byte aligned
 * (RG_ERR_ALIGN), read only; rank in [0, 1024] (RG_ERR_ARG below 0,
 * RG_ERR_SHAPE above).  W, dY, dX, T, beta and the variant as for
 * rg_out_prod_variant (contiguous dY [T, N] and dX [T, K]).  rank == 0 is
 * rg_out_prod_variant; N == 0 leaves dX = beta * dX.
 *
 * Tensor-core variants: U = dY . B is itself an OUT_PROD over B's 16-bit
 * copy, and the base product's kernel takes U's columns and scale * A's rows
 * (16-bit, the kind the base operands use) as extra contraction chunks, so
 * the adapter term lands in the same F32 accumulator as dY . deq(W).  Its
 * error: |err| <= 5e-3 * sum_n |dY||deq W| + 1e-2 * |scale| *
 * sum_j (sum_n |dY||B|)|A| + 1e-7 (dY, B, U and A each rounded to 16 bits).
 * fp16 kinds (quantized and F16 W) need U and scale * A within the fp16
 * range, like dY.  Other variants: the base product as they compute it, then
 * U and scale * U . A in F32 (about 1e-5 relative to the same sums).
 * Workspace from the library's stream-ordered pool, as rg_out_prod.
 */
int rg_out_prod_lora(int variant, int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                     int64_t T, float* dX, float beta, const float* lora_a, const float* lora_b,
                     int64_t rank, float scale, void* stream);

/* The variant RG_VARIANT_AUTO picks for this shape (ignores RG_VARIANT). */
int rg_select_variant(int wtype, int64_t N, int64_t K, int64_t T);

/* How one OUT_PROD call of a shape runs on the current device: a report for
 * measurement (the redundant-decode count the method trades for not storing
 * an F32 copy of W), filled in without launching or allocating anything. */
typedef struct rg_plan_info {
  int32_t variant;          /* the variant that runs (never RG_VARIANT_AUTO) */
  int32_t cta_group;        /* tensor-core variants: CTAs per MMA (1 or 2); else 0 */
  int32_t tile_k;           /* output tile: values along K ... */
  int32_t tile_t;           /* ... by rows along T (dY rows one pass over W serves) */
  int32_t n_splits;         /* contraction over N split into this many partial sums (1: none) */
  int32_t grid;             /* CTAs of the main kernel (tensor-core: before the residency cap) */
  int32_t launches;         /* kernels one call enqueues, for beta 0 and row-contiguous dY (a
                               contraction split in two then adds both halves into dX; with
                               beta != 0 or strided dY it adds a reduction kernel) */
  int32_t stream_k;         /* tensor-core variants: 1 when the last tiles' contraction is
                               shared evenly over all units (stream-K), else 0 */
  int64_t decode_ops;       /* weight values decoded per call: ceil(T / tile_t) * N * K */
  int64_t workspace_bytes;  /* what rg_out_prod_ws needs for this variant */
} rg_plan_info;

/* Fills *out for `variant` (RG_VARIANT_AUTO: the shape's choice) and returns
 * RG_OK; RG_ERR_TYPE, RG_ERR_ARG (out NULL, negative or too large sizes) or
 * RG_ERR_SHAPE as rg_out_prod validates them; RG_ERR_CUDA without a current
 * CUDA device (the plan depends on its SM count).  T == 0 or K == 0: nothing
 * runs (launches 0); N == 0: one kernel scales dX by beta. */
int rg_plan(int variant, int wtype, int64_t N, int64_t K, int64_t T, rg_plan_info* out);

/* Kernels this library has enqueued in this process (all devices and entry
 * points, successful launches only): a measurement aid, read before and after
 * a region to count its launches. */
uint64_t rg_launch_count(void);

/*
 * out[n, k] = deq(W)[n, k] as F32, bit-exact: every decoded value is an exact
 * F32 (Q8_0: 11-bit x 8-bit product; Q4_0: 11-bit x 4-bit; F16/BF16: widened)
 * except Q4_K, whose (d*sc)*q - dmin*m is rounded once, to nearest even.
 * Signed zeros are kept (d < 0 times a zero code is -0.0).  This is the role
 * of the PR's ggml_get_to_fp32_cuda converters.  Enqueued on the legacy
 * default stream; out: [N, K] F32, 16-byte aligned.
 */
int rg_dequant(int wtype, const void* W, int64_t N, int64_t K, float* out);

/* rg_dequant on `stream`. */
int rg_dequant_async(int wtype, const void* W, int64_t N, int64_t K, float* out, void* stream);

/* Stored bytes of one row of K values: K/32*34 (Q8_0), K/32*18 (Q4_0),
 * K/32*20 (Q4_1), K/32*22 (Q5_0), K/32*24 (Q5_1), K/256*144 (Q4_K),
 * K/256*176 (Q5_K), K/256*210 (Q6_K), K/256*84 (Q2_K), K/256*110 (Q3_K),
 * K/32*17 (MXFP4), K/64*36 (NVFP4), 2K (F16, BF16), 4K (F32); 0 for an
 * unknown type or a K that is not a whole number of blocks. */
size_t rg_row_bytes(int wtype, int64_t K);

/* Static, NUL-terminated description of a status code. */
const char* rg_strerror(int status);

/* Synchronizes `stream`, then reads and clears the current device's status
 * word.  Returns RG_ERR_TIMEOUT if a kernel gave up a bounded wait since the
 * last check, RG_ERR_RANGE if a dY value overflowed the tensor-core operand
 * kind since the last check (the conversion of dY checks every value; the
 * decoded weight values' fp16 range is a precondition of the quantized and
 * F16 types, not checked), RG_ERR_CUDA if the stream reports an error, else
 * RG_OK.  The first error recorded since the last check wins. */
int rg_check(void* stream);

/* Library version, (major << 16) | minor. */
int rg_version(void);

/* Measurement aid: the next tensor-core OUT_PROD call (rg_out_prod* choosing
 * a TC variant) made from this host thread records the CUDA event `before`
 * on its stream right before its GEMM kernel and `after` right after it
 * (cudaEvent_t handles passed as void*), so the kernel alone can be timed
 * inside a larger timed region; the dY conversion is outside the pair, the
 * partial-sum reduction of a split contraction inside it.  The
 * events are used once, then forgotten.  NULL, NULL clears.  Returns RG_OK. */
int rg_profile_next_gemm(void* before, void* after);

/* Test hook for failure detection: enqueues one kernel whose single wait can
 * never complete, so that it gives up after timeout_ms (1..60000; else
 * RG_ERR_ARG) and records RG_ERR_TIMEOUT for the next rg_check.  The context
 * stays usable. */
int rg_debug_wait_probe(int timeout_ms, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RG_H */
