/*
 * gsfp8_test.h -- test hooks of libgsfp8 (not part of the computation).
 *
 * The kernel fed by TMA -- fp8_gemm_block_scaled -- waits on shared-memory
 * barriers for its loads, for the tensor cores and for the promotion warps.
 * Every such wait is bounded (about 2 s by %globaltimer); a kernel that gives
 * up records GS_ERR_TIMEOUT in the device status word (gs_device_status),
 * lets its own copies and MMAs in flight finish, frees its tensor memory and
 * returns, leaving the CUDA context usable.  This hook
 * lets a test exercise that path without a fault: no trap, no bad address,
 * no endless loop -- a barrier that nothing completes, waited on with its
 * limit.
 */
#ifndef GSFP8_TEST_H
#define GSFP8_TEST_H

#ifdef __cplusplus
extern "C" {
#endif

/* on != 0: launches made from now on by this process of the kernel named
 * above issue no TMA loads, so their first bounded wait runs out: the launch
 * takes about 2 s, writes nothing valid to its outputs and records
 * GS_ERR_TIMEOUT.  on == 0 restores normal operation.  Process-wide; set it
 * only while no other thread launches that kernel.  Returns GS_OK. */
int gs_test_set_stall(int on);

#ifdef __cplusplus
}
#endif
#endif /* GSFP8_TEST_H */
