/*
 * stage_gemm.h -- C ABI of the GB300 (sm_103a) tensor-core GEMM
 *
 *     C = epilogue(A . B)
 *
 * A is M x K, B is K x N, C is M x N, all row-major with leading dimensions
 * (row pitches, in elements) lda >= K, ldb >= N, ldc >= N.  A and B are both
 * fp16, both bf16 or both FP8 E4M3; the product is accumulated in fp32; C is
 * fp32, fp16 or bf16.  The operation and its rules come from these pages:
 *
 *   - gizml:tile, "Tile.dot": the matrix product [M,K][K,N] -> [M,N] in F32,
 *     on matrix cores when both operands are F16 or both are BF16; "FP8" is
 *     the page's fourth storage type (E4M3), taken here as a third operand
 *     type of one kind for both operands (tcgen05 kind::f8f6f4).
 *   - gizml:tile, "Tile.run" (the fused example over 128 x 128 output tiles,
 *     storing acc.relu()), "Tile.relu" and "Tile.add": the epilogues.  The
 *     bias of SG_EPI_BIAS_RELU is one fp32 value per column, added to the
 *     fp32 accumulator before the ReLU, as the per-column accumulator seed of
 *     the Swin-layer epilogue notes (d4r, rrswin_enc2_epilogues.md).
 *   - gizml:tile, "Tile.to": the single rounding of the fp32 result into the
 *     output type is round-to-nearest-even; overflow gives +-infinity.
 *   - gizml:tile, "In.at": operand elements past the edge of A or B (row >= M,
 *     column >= N, k >= K, including any ld padding) are read as 0; they are
 *     never loaded from memory.  Tolk.Stage, "operands": a gate whose index
 *     is invalid copies 0.
 *   - gizml:tile, "Out.put": elements of C outside M x N (including the ldc
 *     padding columns) are not written.
 *   - gizml:tile, "Program.stages" and Tolk.Stage (two-stage pipeline,
 *     "depth"): `stages` blocks of operands in flight; 1 reads each trip's
 *     blocks in turn, 2 overlaps the next trip's copy with this trip's
 *     products, more hide longer latency.  Tolk.Stage, module overview:
 *     staging moves values and never rounds them, so every stage count gives
 *     bit-identical C.
 *   - gizml:tile, "Program.fold": an empty K range leaves the initial zeros,
 *     so K = 0 writes C = epilogue(0 [+ bias]).
 *   - Tolk.Uniform, "Precondition": parameters that are written do not
 *     overlap others; C must not overlap A, B or bias.
 *
 * Ownership: the caller owns A, B, C and bias (device memory, e.g. from
 * PyTorch).  The library never frees caller memory.  It allocates, once per
 * device, a 4-byte device status word and keeps host-side caches.  Where an
 * operand or residual has no TMA-legal layout (see Layouts below), a call
 * also takes one stream-ordered buffer for a copy of it with 16-byte row
 * pitches, released on the call's stream after the kernel.  sg_gemm_host
 * also creates, once per device, three streams and five events, and takes
 * one stream-ordered device buffer per call (released on the call's
 * stream).  Those buffers come from a memory pool the library creates on
 * each device on first use; freed blocks stay in it, so a later call maps
 * no new memory, and the pool keeps up to the largest amount used at once
 * until the process exits.  While `stream` is being captured into a graph
 * they come from the device's default pool instead.  sg_gemm_noalloc
 * allocates nothing.
 *
 * Execution: every call is asynchronous on `stream` (a cudaStream_t passed as
 * void*; NULL is the legacy default stream).  Argument checks run on the
 * host before any CUDA call.
 *
 * Errors: 0 on success, a negative SG_ERR_* code otherwise (sg_strerror gives
 * its text).  A device-side wait that gives up (see SG_ERR_TIMEOUT) is
 * reported asynchronously through sg_device_status.
 */
#ifndef STAGE_GEMM_H
#define STAGE_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage types. */
enum {
    SG_F32 = 0,  /* IEEE binary32 (output only) */
    SG_F16 = 1,  /* IEEE binary16 */
    SG_BF16 = 2, /* bfloat16 */
    SG_E4M3 = 3  /* OCP FP8 E4M3 (operands only; gizml:tile, "FP8") */
};

/* Epilogues applied to the fp32 accumulator before the output rounding. */
enum {
    SG_EPI_NONE = 0,      /* C = A.B */
    SG_EPI_RELU = 1,      /* C = max(A.B, 0) */
    SG_EPI_BIAS_RELU = 2  /* C = max(A.B + bias[col], 0) */
};

/* Return codes. */
enum {
    SG_OK = 0,
    SG_ERR_ARG = -1,     /* M, N or K < 0; ld < row length; null pointer; bias
                            missing for SG_EPI_BIAS_RELU or given otherwise;
                            a dimension or pitch beyond 2^31 - 1 */
    SG_ERR_DTYPE = -2,   /* in_dtype not fp16/bf16/e4m3, out_dtype not fp32/fp16/bf16,
                            or an unknown epilogue */
    SG_ERR_STAGES = -3,  /* stages < 0, > SG_MAX_STAGES, or does not fit in
                            shared memory for the chosen tile */
    SG_ERR_ALIAS = -4,   /* C overlaps A, B, R or bias */
    SG_ERR_ALIGN = -5,   /* a pointer not aligned to its own elements: A or B
                            (2 bytes for 16-bit operands), C or R (the output
                            type's size), bias or b_scale (4 bytes) */
    SG_ERR_ARCH = -6,    /* the current device is not sm_103 */
    SG_ERR_CUDA = -7,    /* a CUDA runtime/driver call or the launch failed */
    SG_ERR_TIMEOUT = -8, /* a device-side wait gave up (reported by
                            sg_device_status) */
    SG_ERR_CONFIG = -9   /* sg_gemm_ex / sg_plan_ex: an unknown field value,
                            or a tile width or kernel mode this problem
                            cannot take */
};

#define SG_MAX_STAGES 8
#define SG_VERSION 120 /* 1.2.0: sg_gemm_ex / sg_plan_ex with sg_config; C and bias alignment checked */

/*
 * sg_gemm -- C[i*ldc + j] = epilogue(sum_k A[i*lda + k] * B[k*ldb + j])
 * for 0 <= i < M, 0 <= j < N, rounded once into out_dtype.
 *
 *   M, N, K     problem size (>= 0).  M == 0 or N == 0 is a no-op.
 *   A, lda      device pointer to M x K row-major in_dtype elements; lda >= K.
 *   B, ldb      device pointer to K x N row-major in_dtype elements; ldb >= N.
 *   C, ldc      device pointer to M x N row-major out_dtype elements; ldc >= N.
 *   in_dtype    SG_F16, SG_BF16 or SG_E4M3 (both operands).
 *   out_dtype   SG_F32, SG_F16 or SG_BF16.
 *   epilogue    SG_EPI_NONE, SG_EPI_RELU or SG_EPI_BIAS_RELU.
 *   bias        device pointer to N fp32 values, required iff BIAS_RELU.
 *   stages      shared-memory operand slots in flight: 0 = the largest count
 *               that fits, else 1..SG_MAX_STAGES.
 *   stream      cudaStream_t (as void*) the work is queued on.
 *
 * Layouts: an operand whose base is 16-byte aligned and whose row pitch is
 * a multiple of 16 bytes (lda, ldb multiples of 8 elements, of 16 for FP8;
 * any pitch for a single row) is staged by TMA.  Any other operand (and any
 * such residual) is first copied on `stream` into a buffer with 16-byte row
 * pitches and staged from there by TMA; if that buffer cannot be had (and
 * always in sg_gemm_noalloc) it is staged by element loads of the producer
 * warp into the same shared-memory layout (slower; the kernel then runs one
 * CTA per tile).  The results are bit-identical either way.  Only
 * element alignment (2 bytes for 16-bit operands) is required, else
 * SG_ERR_ALIGN.  C must be aligned to its own elements (4 bytes for fp32, 2
 * for fp16 / bf16) and bias to 4 bytes, else SG_ERR_ALIGN; a C that is not
 * 16-byte aligned or whose pitch is not a multiple of 16 bytes is computed
 * into a buffer with 16-byte row pitches and its N columns copied into
 * place on `stream` (its padding is not written); without that buffer (and
 * in sg_gemm_noalloc) it is written row by row from the epilogue's staging
 * buffer with ordinary stores masked to M x N.  The same bits either way.
 */
int sg_gemm(int64_t M, int64_t N, int64_t K,
            const void* A, int64_t lda,
            const void* B, int64_t ldb,
            void* C, int64_t ldc,
            int in_dtype, int out_dtype, int epilogue,
            const float* bias, int stages, void* stream);

/*
 * sg_gemm_residual -- C = epilogue(A . B + R): the residual R (M x N,
 * row-major, pitch ldr >= N, of type out_dtype) is added to the fp32
 * accumulator before the bias and the ReLU, the fold starting from R
 * instead of zeros.  This is the back-projection of the Swin-layer MLP band
 * (d4r, rrswin_enc2_epilogues.md, "Shape of the whole MLP band": its MMA
 * takes the previous accumulator as its C input) and gizml:tile's
 * "Program.fold" with a non-zero init; K = 0 gives C = epilogue(R [+bias]).
 * R may be C itself (same pointer and ldr == ldc): every element is read
 * before it is written.  Any other overlap of R and C is SG_ERR_ALIAS; R
 * not aligned to its elements is SG_ERR_ALIGN; a NULL R is SG_ERR_ARG.  An
 * R whose base is 16-byte aligned and whose pitch is a multiple of 16 bytes
 * is loaded by TMA, any other by element loads.  Everything else is as for
 * sg_gemm.
 */
int sg_gemm_residual(int64_t M, int64_t N, int64_t K,
                     const void* A, int64_t lda,
                     const void* B, int64_t ldb,
                     const void* R, int64_t ldr,
                     void* C, int64_t ldc,
                     int in_dtype, int out_dtype, int epilogue,
                     const float* bias, int stages, void* stream);

/*
 * sg_gemm_qb -- C = epilogue(A . B) with an integer-coded B: Bq holds signed
 * 8-bit codes q (K x N row-major, pitch ldb >= N, single bytes, no alignment
 * rule) and b_scale one fp32 value s_j per column (device pointers), so
 * that b_kj = s_j * q_kj; A is fp16 or bf16 (in_dtype) as for sg_gemm.  The
 * pages' decoded panel (Tolk.Stage, "Decoded panels on the host": an operand
 * decoded from integer codes, as a quantised matrix's is, has the values of
 * its panel decoded once and read back by every trip of the other output
 * loops) is taken on the GPU: each CTA decodes all of B once into shared
 * memory as 16-bit values equal to the codes (exact), every row tile's MMAs
 * read that panel, and s_j multiplies column j of the fp32 accumulator
 * before the bias and the ReLU.  B must fit the resident panel: K <= 128
 * and N <= 512 (else SG_ERR_ARG).  A is staged by TMA: an A without a
 * TMA-legal layout (16-byte aligned base, pitch a multiple of 16 bytes) is
 * first copied to 16-byte pitches on `stream` (if that copy's buffer cannot
 * be had, SG_ERR_ARG), and a C likewise as for sg_gemm.  The scales must be
 * finite.  C must not overlap A, Bq, b_scale or bias (SG_ERR_ALIAS); a NULL
 * b_scale, or a NULL Bq with K > 0, is SG_ERR_ARG; a b_scale not aligned
 * to 4 bytes is SG_ERR_ALIGN; in_dtype other than
 * fp16/bf16 is SG_ERR_DTYPE.  Everything else is as for sg_gemm.
 */
int sg_gemm_qb(int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda,
               const int8_t* Bq, int64_t ldb, const float* b_scale,
               void* C, int64_t ldc,
               int in_dtype, int out_dtype, int epilogue,
               const float* bias, int stages, void* stream);

/*
 * sg_gemm_host -- the same product, C = epilogue(A . B [+ R]), on HOST
 * buffers: A, B, R (may be NULL: no residual), bias and C are host pointers
 * with the meanings, layouts and pitches of sg_gemm / sg_gemm_residual.
 * The pages define only the product; this call adds the transfers around
 * it.  It takes one device buffer (stream-ordered, from the library's pool
 * on `stream`, released with cudaFreeAsync on the same stream), copies bias
 * and B in, then copies A (and R) in row chunks on a library-owned stream
 * while each chunk's GEMM runs as soon as its rows have arrived (chunks
 * alternate between `stream` and a library-owned compute stream, so one
 * chunk's last wave overlaps the next chunk's first), and copies each chunk
 * of C back on another library-owned stream while later chunks compute.  A
 * host pitch that is a whole number of 16-byte units is kept on the device
 * and each chunk then moves as one contiguous span; other pitches move row
 * by row.  All of it is ordered after the work already on `stream`, and
 * `stream` waits for all of it: synchronise `stream` before reading C or
 * releasing the host buffers.  Page-locked host memory
 * lets the copies overlap the GEMMs; pageable memory works, with the copies
 * staged by the driver.  The chunks are GEMMs over row ranges of the same
 * operands, so every element of C has the same bits as from sg_gemm.
 * Concurrent calls on one device are serialised while they are queued (the
 * library's copy streams and events are shared).  The environment variable
 * STAGE_GEMM_HOST_CHUNKS (1..64) overrides the chunk count (tuning only).
 * Returns the codes of sg_gemm and sg_gemm_residual (host-side checks,
 * including the overlap rules, apply to the host ranges); SG_ERR_CUDA when
 * an allocation, copy or launch fails.
 */
int sg_gemm_host(int64_t M, int64_t N, int64_t K,
                 const void* A, int64_t lda,
                 const void* B, int64_t ldb,
                 const void* R, int64_t ldr,
                 void* C, int64_t ldc,
                 int in_dtype, int out_dtype, int epilogue,
                 const float* bias, int stages, void* stream);

/* The launch configuration sg_gemm would use for TMA-legal A and B (no GPU
 * work is queued).  Needs a current CUDA device; returns the same codes as
 * sg_gemm. */
typedef struct {
    int32_t block_m;       /* output tile rows (128) */
    int32_t block_n;       /* output tile columns */
    int32_t block_k;       /* K elements per stage (64, or 128 for FP8) */
    int32_t stages;        /* operand slots in the shared-memory ring */
    int32_t max_stages;    /* the largest count that fits for this tile */
    int32_t tiles;         /* output tiles */
    int32_t grid;          /* persistent CTAs launched */
    int32_t threads;       /* threads per CTA */
    int32_t smem_bytes;    /* dynamic shared memory per CTA (modes 4 and 5:
                              with a bias, the biases too) */
    int32_t tmem_columns;  /* tensor-memory columns allocated per CTA */
    int32_t tma_store;     /* 1: C written by TMA stores; 0: C has no
                              TMA-legal layout (sg_gemm computes it into a
                              16-byte-pitch buffer and copies it into place,
                              sg_gemm_noalloc writes it row by row) */
    int32_t cluster_m;     /* CTAs per cluster (1 or 2) */
    int32_t pair_mma;      /* 1: the cluster's two CTAs compute one 256-row tile
                              with the paired MMA, each CTA owning 128 rows of
                              it; 0: one CTA per 128-row tile */
    int32_t group_m;       /* cluster row blocks swept together by the tile raster */
    int32_t mode;          /* 1 single CTA, 3 paired MMA, 4 B resident in
                              shared memory, 5 integer-coded B decoded into
                              shared memory, 6 paired 256 x 512 tiles held as
                              two 256-column accumulators (2 is not used) */
    int32_t ring_group;    /* ring slots filled and consumed together on one
                              pair of barriers (2 when both operands arrive by
                              TMA and the ring has 6 or 8 slots, else 1) */
    int32_t tail_units;    /* half-width units the last tiles of the raster
                              were split into (0: none): when a last wave of
                              256-column tiles (16-bit operands, both by TMA)
                              would fill at most half of the clusters, each of
                              its tiles runs as two 128-column units */
} sg_plan_info;

int sg_plan(int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, int epilogue, int stages,
            int64_t ldc, const void* C, sg_plan_info* info);

/*
 * Launch configuration for sg_gemm_ex and sg_plan_ex.  A field left 0 is the
 * planner's choice; a non-zero field is honoured exactly or the call fails
 * with SG_ERR_CONFIG (never silently replaced).  Every configuration issues
 * the same MMAs in the same K order for each output element, so C has the
 * same bits whatever the configuration (gizml:tile, "tune": every
 * configuration computes the same result; Tolk.Stage: staging never rounds).
 *
 *   block_n     output tile columns: 128, 192, 256 or 512 (FP8 operands:
 *               128, 256 or 512, whole 128-byte B boxes); 512 is mode 6.
 *   mode        1: one CTA per 128 x block_n output tile.
 *               3: the two CTAs of a cluster compute one 256 x block_n tile
 *                  with the paired MMA (tcgen05 cta_group::2); each CTA owns
 *                  128 x block_n of it and stages its own A rows and half of
 *                  the B columns.  block_n must split into whole B boxes per
 *                  CTA (128 or 256 for 16-bit operands, 256 for FP8), and A
 *                  and B must be TMA-legal.
 *               4: B resident in shared memory (block_n 128; K at most two
 *                  128-byte stages of K, N at most 512; A and B TMA-legal);
 *                  with a bias, the biases are staged there too.
 *               6: as 3 over 256 x 512 tiles held as two 256-column
 *                  accumulators (block_n 512): each CTA stages its A rows
 *                  once for both, a quarter fewer operand bytes per product
 *                  than 256-column pairs; A and B must be TMA-legal.
 *   stages      operand ring depth, 1..SG_MAX_STAGES (0: the deepest that
 *               fits); a depth that does not fit is SG_ERR_STAGES.
 *   group_m     tile raster: cluster row blocks swept together, 1..64 (odd
 *               groups sweep the column blocks backwards).
 *   tail_split  1 or 0: split a short last wave of 256- or 512-column tiles
 *               into half-width units where it pays (the default); -1:
 *               never.
 *
 * The gizml:tile program's workgroup per 128 x 128 output tile is
 * {block_n = 128, mode = 1} (one CTA per tile) or {block_n = 128, mode = 3}
 * (each CTA of a pair owns one 128 x 128 tile and the pair shares B).
 */
typedef struct {
    int32_t block_n;
    int32_t mode;
    int32_t stages;
    int32_t group_m;
    int32_t tail_split;
} sg_config;

/*
 * sg_gemm_ex -- sg_gemm (R == NULL) or sg_gemm_residual (R != NULL, with its
 * rules for R and ldr) under an explicit launch configuration.  `config` may
 * be NULL or all zeros: then this is exactly sg_gemm / sg_gemm_residual
 * (including a configuration cached by sg_tune).  Returns sg_gemm's codes,
 * plus SG_ERR_CONFIG when a requested field cannot be honoured for this
 * problem (checked on the host before any GPU work is queued).
 */
int sg_gemm_ex(int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda,
               const void* B, int64_t ldb,
               const void* R, int64_t ldr,
               void* C, int64_t ldc,
               int in_dtype, int out_dtype, int epilogue,
               const float* bias, const sg_config* config, void* stream);

/* The launch configuration sg_gemm_ex would use for TMA-legal A and B under
 * `config` (NULL: sg_plan's), without queueing GPU work.  Needs a current
 * CUDA device; returns sg_gemm_ex's codes. */
int sg_plan_ex(int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, int epilogue,
               int64_t ldc, const void* C, const sg_config* config, sg_plan_info* info);

/*
 * sg_tune -- times every launch configuration that fits this problem (tile
 * width, kernel mode, ring depth, raster group) on the
 * caller's operands, on `stream`, and keeps the fastest for later sg_gemm
 * and sg_plan calls with the same key (device, M, N, K, types, epilogue, and
 * whether A, B and C are TMA-legal).  This is gizml:tile's "tune": each
 * configuration is measured once and the choice cached; every configuration
 * computes the same bits (the same products summed in the same K order), so
 * tuning never changes a result.  C is written several times (the kernel
 * never reads C); arguments are checked as by sg_gemm (stages is not an
 * argument: ring depth is tuned).  Blocks until the measurements finish.
 * `best` and `best_ms` (either may be NULL) receive the chosen plan and its
 * time per call.  An explicit `stages` in a later sg_gemm call still wins.
 */
int sg_tune(int64_t M, int64_t N, int64_t K,
            const void* A, int64_t lda,
            const void* B, int64_t ldb,
            void* C, int64_t ldc,
            int in_dtype, int out_dtype, int epilogue,
            const float* bias, void* stream,
            sg_plan_info* best, float* best_ms);

/* Forgets every tuned configuration; returns how many there were. */
int sg_tune_clear(void);

/* Tuned configurations currently cached. */
int sg_tune_count(void);

/* Waits for `stream`, then returns SG_ERR_TIMEOUT if any kernel of this
 * library on the current device gave up on a wait since the last call (and
 * clears that record), SG_ERR_CUDA if the stream reports an error, else 0. */
int sg_device_status(void* stream);

/* The bound on each device-side wait, in nanoseconds (default 2e9; the
 * environment variable STAGE_GEMM_WAIT_LIMIT_MS overrides it at load).
 * Applies to launches made after the call. */
void sg_set_wait_limit_ns(uint64_t ns);
uint64_t sg_get_wait_limit_ns(void);

/* Static text for a return code. */
const char* sg_strerror(int code);

/* SG_VERSION of the built library. */
int sg_version(void);

/*
 * sg_gemm_noalloc -- the same GEMM as sg_gemm, for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry
 * point; it exists for the library's users, not for the method.
 *
 * Who needs it: code that runs where cudaMalloc is not allowed or not
 * wanted -- inside a host memory-pool or allocator callback, under an
 * embedding runtime that owns every device allocation (and budgets it), or
 * in a process that must not grow its device footprint after start-up.
 * sg_gemm allocates a 4-byte device status word on its first call on each
 * device, and a buffer for a copy of any operand without a TMA-legal layout;
 * this entry point does neither (such an operand is staged by element
 * loads).
 *
 * Scratch: the kernel's only scratch memory is that status word (written by
 * a device-side wait that gives up).  Here it lives in a file-scope
 * static __device__ array of SG_NOALLOC_SCRATCH_BYTES (256) bytes, which
 * every GPU that loads the library holds until the process exits.  This
 * kernel needs 4 bytes of it whatever M, N and K are; a need above the
 * array's size would be rejected with SG_ERR_ARG.
 *
 * Set-up: the first call on a device (with that device current) looks up
 * the array's device address with cudaGetSymbolAddress and queries the
 * device's attributes; make that first call before any stream capture.
 * Later calls do no set-up.  No call allocates: no cudaMalloc, cudaFree or
 * allocating library routine.  The caller passes inputs and outputs exactly
 * as for sg_gemm; arguments, return codes and results are sg_gemm's.
 *
 * Sharing: every call uses the same array and leaves its contents behind.
 * Each call clears the status word on `stream` before its kernel runs, so
 * sg_gemm_noalloc_status reports the most recent call.  Calls whose kernels
 * overlap on the GPU (on different streams, or from different threads)
 * race on the status word: serialise them if the status matters.
 */
#define SG_NOALLOC_SCRATCH_BYTES 256
int sg_gemm_noalloc(int64_t M, int64_t N, int64_t K,
                    const void* A, int64_t lda,
                    const void* B, int64_t ldb,
                    void* C, int64_t ldc,
                    int in_dtype, int out_dtype, int epilogue,
                    const float* bias, int stages, void* stream);

/* Waits for `stream`, then returns SG_ERR_TIMEOUT if the last
 * sg_gemm_noalloc kernel on the current device gave up on a device-side
 * wait, SG_ERR_CUDA on a stream error, else 0.  Allocates nothing; reads the
 * status word with a plain device-to-host copy. */
int sg_gemm_noalloc_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* STAGE_GEMM_H */
