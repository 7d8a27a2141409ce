/* icpnn_probe.h -- measurement helper of libicpnn; not part of the
 * registration path and not described by the pages.
 *
 * icpnn_probe_l2_read -- read a device buffer `repeats` times in one launch
 * with loads that bypass L1 (each SM's blocks stride over the whole buffer),
 * so that for a buffer that fits in L2 the achieved rate approaches the L2
 * read bandwidth: the ceiling of a search whose tree stays L2-resident.
 *   buf      device buffer of `bytes` bytes, 16-byte aligned, bytes a
 *            multiple of 16; only read.
 *   repeats  passes over the buffer, >= 1.
 *   sink     one device uint32 that the kernel may write (keeps the loads).
 *   stream   cudaStream_t (NULL = legacy default stream); not synchronised.
 * Time it with events on `stream`; bytes read = bytes * repeats.
 * Errors: INVALID_ARG, CUDA. */
#ifndef ICPNN_PROBE_H
#define ICPNN_PROBE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int icpnn_probe_l2_read(const void* buf, int64_t bytes, int32_t repeats, uint32_t* sink, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ICPNN_PROBE_H */
