/*
 * stage_gemm_testing.h -- test-only entry points of libstage_gemm.so.
 *
 * Not part of the supported interface; the test suite uses them to exercise
 * the device-side failure path without faulting, trapping or hanging a GPU.
 */
#ifndef STAGE_GEMM_TESTING_H
#define STAGE_GEMM_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Failure injection for the bounded device waits (gizml:tile lists "fail" as
 * an effect of every call; the pages define no device-side failure
 * mechanism, so this hook has no counterpart there).  After this call, every
 * CTA of every later sg_gemm launch skips the TMA copy of its K chunk with
 * index `it` (counted over the CTA's tiles).  The MMA issuer's bounded wait
 * for that chunk then runs out, the kernel records a timeout in the device
 * status word, every role leaves its loop, drains its own copies and MMAs,
 * frees tensor memory and exits; sg_device_status returns SG_ERR_TIMEOUT.
 * C is left partly unwritten.  it < 0 switches the hook off.  Returns 0.
 */
int sg_test_set_skip_load(int64_t it);

/*
 * Forces the output tile width of later sg_gemm / sg_plan calls to `bn`
 * columns (128, 192 or 256; 0 restores the planner's choice).  Every width
 * issues the same MMAs in the same K order for each output element, so C
 * must be bit-identical across widths (gizml:tile, "tune": every
 * configuration computes the same result).  Returns 0, or SG_ERR_ARG for any
 * other width.  The environment variable STAGE_GEMM_TILE_N sets the initial
 * value when the library loads.
 */
int sg_test_set_tile_n(int bn);

/*
 * Forces the kernel mode of later sg_gemm / sg_plan calls: 1 (one CTA per
 * 128-row tile, copying its whole B tile), 3 (the two CTAs of a cluster
 * compute one 256-row tile with the paired MMA, each staging half of B) or
 * 4 (each CTA keeps all of B in shared memory and streams A; only where B
 * has at most 2 K chunks and 4 column blocks of 128, otherwise the
 * planner's choice stands); mode 3 needs a tile width of 128 or 256.  0 restores the planner's choice.  Every mode sums the same products in the same K order
 * for each output element, so C must be bit-identical.  Returns 0, or
 * SG_ERR_ARG.  The environment variable STAGE_GEMM_CLUSTER sets the initial
 * value at load.
 */
int sg_test_set_cluster(int mode);

/*
 * Whether later plans may split a short last wave of 256-column tiles into
 * 128-column units (1, the default) or never (0).  Every element is computed
 * by one unit either way, summing the same products in the same K order, so
 * C must be bit-identical.  Returns 0, or SG_ERR_ARG.  The environment
 * variable STAGE_GEMM_TAIL_SPLIT=0 sets the initial value at load.
 */
int sg_test_set_tail_split(int on);

/*
 * Whether later sg_gemm / sg_gemm_residual / sg_gemm_ex calls may copy an
 * operand or residual without a TMA-legal layout into a stream-ordered
 * buffer with 16-byte pitches (1, the default) or must stage it by element
 * loads (0, as sg_gemm_noalloc always does).  The copies move values only,
 * so C must be bit-identical either way.  Returns 0, or SG_ERR_ARG.
 */
int sg_test_set_repack(int on);

#ifdef __cplusplus
}
#endif

#endif /* STAGE_GEMM_TESTING_H */
