// internal.h -- host functions one translation unit of the library calls in
// another.  Not part of the C ABI (hidden symbols).
#ifndef SPEC_INTERNAL_H
#define SPEC_INTERNAL_H

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#define SPEC_HIDDEN __attribute__((visibility("hidden")))

namespace spec_internal {

// Records per row of the sampler's chunk kernel: one per 4 KB of the row.
SPEC_HIDDEN size_t chunk_count(int32_t V, int32_t dtype);

// Launch the sampler's chunk kernel alone on R rows of V logits: one float2
// record per 4 KB chunk of each row into rec[R][chunk_count], (chunk max,
// sum 2^((x - max) log2(e) / T)) for a sampled row.  Row r's temperature is
// temperature[r / rows_per_temp]; rows with an invalid temperature, or at
// T = 0, are not read.  The kernel lets the next kernel on the stream start
// early (programmatic dependent launch); that kernel must wait for this
// grid before it reads the records.  Returns a SPEC_* status.
SPEC_HIDDEN int chunk_records(const void *logits, const float *temperature, int32_t rows_per_temp,
                              float2 *rec, void *hdr, int32_t R, int32_t V, int32_t dtype,
                              cudaStream_t stream);

// The device address of spec_verify_noalloc's scratch array on the current
// device (looked up once per device and kept).  Returns a SPEC_* status.
SPEC_HIDDEN int noalloc_scratch(void **addr);

}  // namespace spec_internal

#endif
