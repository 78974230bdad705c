/*
 * qgemm_testing.h -- test hooks of libqgemm.so, not part of the compute API.
 *
 * qg_test_bounded_wait -- runs the library's bounded pipeline wait on the GPU
 * in a kernel shaped like its pipelines (a producer warp and three consumer
 * warps waiting on one shared-memory stage barrier), so that a test can make
 * the wait give up without faulting, trapping or hanging the GPU.  The
 * source pages have no counterpart: every wait in this library's kernels is
 * bounded, and this is how that bound is exercised.
 *
 *   fill      0: the producer never fills the stage, so each consumer warp's
 *               wait runs out after `limit_us` and gives up: it records
 *               FAULT_WAIT_FULL (bit 1) in the device fault word (read it with
 *               qg_read_device_fault) and the warp ends;
 *             1: the producer fills the stage; every wait completes.
 *   limit_us  the bound of each wait, 1 .. 2000000 microseconds (the
 *             library's own kernels use 2 s).
 *   out_dev   device int[3]: per consumer warp, 1 if its wait completed, 0 if
 *             it gave up.
 * Returns QG_OK, QG_ERR_INVALID_ARG (null out_dev, limit out of range) or
 * QG_ERR_CUDA (launch error).  Enqueued on `stream` of the current device;
 * nothing is synchronised.
 */
/*
 * qg_test_gemv_plan -- the launch plan the 2-bit tensor-core GEMV takes on
 * the current device for a 2-bit, block-64 request of this shape, so that
 * tests can check that their shapes reach each variant.  Nothing is launched.
 *
 *   a_dtype, zp_mode  as in qgemm_nbits (0 fp32, 1 fp16, 2 bf16; 0 none,
 *                     1 tensor, 2 uniform)
 *   (fp32 activations with M > 4 run as one launch per group of four rows;
 *   where the B fragments of all rows leave no room for the ring, 3 or 4 rows
 *   of 16-bit activations run as two launches of two rows and 2 rows of fp32
 *   activations as two launches of one; the plan is that of a full group)
 *   out               host int[4]: weight rows per tile (32: block parameters
 *                     staged with the codes; 16: long K, block parameters
 *                     copied per span by the consumer warps), consumer warps,
 *                     CTAs launched, shared-memory ring stages.
 * Returns QG_OK, QG_ERR_INVALID_ARG (null out, M, N or K not positive) or
 * QG_ERR_UNSUPPORTED (the request does not take this GEMV: other paths serve it).
 */
#ifndef QGEMM_TESTING_H
#define QGEMM_TESTING_H

#include "qgemm.h"

#ifdef __cplusplus
extern "C" {
#endif

int qg_test_bounded_wait(int fill, unsigned int limit_us, int *out_dev, qg_stream_t stream);
int qg_test_gemv_plan(int M, int N, int K, int a_dtype, int zp_mode, int *out);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_TESTING_H */
