/*
 * sv_probe.h -- streaming read probe used to calibrate the attainable HBM read bandwidth.
 *
 * This is a measurement aid for the roofline of the verify kernel; the pages define no such
 * operation. It reads `bytes` of device memory once with 128-bit loads spread over every SM
 * and adds a checksum of what it read into *out_checksum (device memory, one 64-bit word that
 * the caller zeroes), so the loads cannot be elided.
 *   buf           device pointer, 16-byte aligned.
 *   bytes         multiple of 16.
 *   out_checksum  device pointer to one unsigned 64-bit word.
 *   stream        cudaStream_t; the call is asynchronous.
 * Returns SV_ERR_INVALID_ARG for a null or misaligned pointer or a bad size, SV_ERR_CUDA if
 * the launch fails.
 */
#ifndef SV_PROBE_H
#define SV_PROBE_H

#include <stddef.h>

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

sv_status sv_hbm_read_probe(const void* buf, size_t bytes, unsigned long long* out_checksum,
                            void* stream);

/*
 * Failure-detection check of the bounded waits, with no GPU fault: one thread waits on an
 * mbarrier that nothing ever arrives at, using the same bounded wait as the verify, row and
 * LM-head kernels, for about budget_us microseconds of SM clock (1 .. 1000000), then raises the
 * error word of `stream`'s workspace and returns, as a kernel whose copy or peer never came
 * does. spec_verify_device_error(stream) then reports SV_ERR_DEVICE_TIMEOUT once and clears it;
 * the context stays usable. Asynchronous on `stream`.
 */
sv_status sv_wait_probe(unsigned int budget_us, void* stream);

/*
 * The same bounded wait, raising the error word of another workspace, so that the reports of
 * the entry points with their own workspaces can be checked: target SV_PROBE_NOALLOC raises the
 * fixed array of spec_verify_noalloc on the current device (looked up on first use, like that
 * entry point's first call; `workspace` is ignored), and spec_verify_device_error then reports
 * it once; target SV_PROBE_WORKSPACE raises the word of `workspace`, a caller-owned workspace
 * of spec_verify_ws (device memory, 16-byte aligned), and spec_verify_workspace_error reports
 * it once. SV_ERR_INVALID_ARG for another target, a budget outside 1 .. 1000000 us, or a null or
 * misaligned caller workspace. Asynchronous on `stream`.
 */
enum { SV_PROBE_NOALLOC = 1, SV_PROBE_WORKSPACE = 2 };
sv_status sv_wait_probe_at(unsigned int budget_us, int target, void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SV_PROBE_H */
