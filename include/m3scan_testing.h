/*
 * m3scan_testing.h -- test hooks of libm3scan.so.
 *
 * Not part of the scan: the pages describe nothing like it.  These calls
 * let the library's own tests (1) check which prefill schedule a call
 * took, and (2) make a bounded device wait run out on purpose -- a planted
 * fault on the host side of a handover, never a trap or a bad address --
 * to see the library report M3_ERR_TIMEOUT and stay usable.  They change
 * process-wide settings of the library: a program that is not a test
 * leaves them alone.
 */
#ifndef M3SCAN_TESTING_H
#define M3SCAN_TESTING_H

#include "m3scan.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The prefill kernel a call launched. */
typedef enum m3_test_kernel {
  M3_TEST_KERNEL_NONE = 0,
  M3_TEST_KERNEL_CHUNKED = 1,          /* tensor-core kernel, one CTA per (sequence, head) unit */
  M3_TEST_KERNEL_CHUNKED_BALANCED = 2, /* tensor-core kernel, balanced schedule (handover scratch) */
  M3_TEST_KERNEL_RECURRENT = 3,        /* token-serial kernel */
  M3_TEST_KERNEL_CHUNKED_SPLIT = 4     /* tensor-core kernel, split schedule (few units: segments of each unit
                                          in parallel, a state-only pass first) */
} m3_test_kernel;

/* Planted faults (m3_test_set_fault). */
typedef enum m3_test_fault {
  M3_TEST_FAULT_NONE = 0,
  /* In a balanced-schedule prefill, the CTAs that write handover slots
     do not publish them: each CTA that reads a slot waits until its
     bounded wait runs out, gives up (the rest of the unit it was to
     finish stays unwritten), and the call's status word reads
     M3_ERR_TIMEOUT.  The units that no CTA cut complete. */
  M3_TEST_FAULT_SKIP_HANDOVER_RELEASE = 1
} m3_test_fault;

/* What the last prefill launched (from any host thread). */
typedef struct m3_launch_info {
  int32_t kernel;        /* m3_test_kernel */
  int32_t grid;          /* CTAs launched (per pass) */
  int64_t scratch_bytes; /* handover scratch the launch used (balanced or split schedule), else 0 */
} m3_launch_info;

/*
 * Plant `fault` (m3_test_fault) in the prefill launches that follow, and
 * set their bounded-wait limit to wait_limit_ns (0: the default, 200 ms).
 * m3_test_set_fault(M3_TEST_FAULT_NONE, 0) restores normal operation.
 * Errors: M3_ERR_INVALID_ARG (unknown fault, negative limit).
 */
M3_API m3_status m3_test_set_fault(int32_t fault, int64_t wait_limit_ns);

/* Fill *out with what the last prefill launched.  M3_ERR_INVALID_ARG for NULL. */
M3_API m3_status m3_test_last_launch(m3_launch_info* out);

#ifdef __cplusplus
}
#endif

#endif /* M3SCAN_TESTING_H */
