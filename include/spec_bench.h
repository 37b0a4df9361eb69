/*
 * spec_bench.h -- helpers around the method, not part of it: a read-only
 * streaming probe whose bandwidth serves as the HBM read reference beside the
 * copy bandwidth the roofline divides by, and a self-test of the bounded
 * device waits that report a stalled kernel.
 */
#ifndef SPEC_BENCH_H
#define SPEC_BENCH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Read `bytes` of device memory at `buf` once with 16-byte loads (streaming,
 * evict-first) on `stream` and write one 32-bit word per CTA to `sink` so
 * the loads are kept.  `buf` must be 16-byte aligned and `bytes` a multiple
 * of 16; `sink` must hold spec_bench_read_sink_words() words.  Returns
 * SPEC_OK (0) once launched, SPEC_EINVAL (1) for bad arguments, SPEC_ECUDA
 * (2) for a failed launch.
 */
int32_t spec_bench_read(const void *buf, size_t bytes, uint32_t *sink, void *stream);

/* Words `sink` must hold (one per CTA of the probe's grid on this device). */
int32_t spec_bench_read_sink_words(void);

/*
 * Self-test of the kernels' failure detection: launches one thread that waits
 * on a shared-memory mbarrier nothing ever arrives at, with the same bounded
 * wait the verification and sampling rings use but a limit of `limit_ns`
 * nanoseconds (1 .. 1e8), after which it writes SPEC_DEV_WAIT_TIMEOUT into
 * the status word of `workspace` (a spec_verify or spec_sample workspace,
 * 16-byte aligned) and returns.  Read the result with spec_verify_read_status.
 * No fault and no hang: the wait always ends, and nothing else is in flight.
 * Returns SPEC_OK once launched, SPEC_EINVAL for bad arguments.
 */
int32_t spec_selftest_wait_timeout(void *workspace, uint64_t limit_ns, void *stream);

/*
 * The same self-test on the scratch array of spec_verify_noalloc (on the
 * current device): the timed-out wait writes SPEC_DEV_WAIT_TIMEOUT into that
 * scratch's status word, which spec_verify_noalloc_read_status reports.
 * Returns SPEC_OK once launched, SPEC_EINVAL for a bad limit, SPEC_ECUDA if the
 * scratch's address cannot be looked up.
 */
int32_t spec_selftest_wait_timeout_noalloc(uint64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_BENCH_H */
