/*
 * spec_bench.h -- a measurement helper of the benchmark, not part of the
 * method: a read-only streaming probe whose bandwidth serves as the HBM read
 * reference beside the copy bandwidth the roofline divides by.
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

#ifdef __cplusplus
}
#endif

#endif /* SPEC_BENCH_H */
