/*
 * mla_decode_testing.h -- test hooks of the MLA decode library.  Not part of
 * the decode operation; for exercising its failure detection only.
 *
 * Every wait inside the tensor-core decode kernel is bounded (2 s).  When a
 * wait runs out, the kernel records MLA device error 1 (wait timeout, read
 * with mla_device_error), stops its other roles, drains what it has in
 * flight, frees its tensor memory and returns; the CUDA context stays usable.
 */
#ifndef MLA_DECODE_TESTING_H_
#define MLA_DECODE_TESTING_H_

#ifdef __cplusplus
extern "C" {
#endif

/* on != 0: every later tensor-core decode launch (from any thread, on any
 * device) issues no page copies, so each of its waits for a page runs out
 * after 2 s and the launch ends with device error 1; its outputs are
 * undefined.  on == 0 restores normal operation.  Returns the previous
 * setting.  Host-side only: nothing on the GPU faults, traps or hangs. */
int mla_test_stall_copies(int on);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_TESTING_H_ */
