/*
 * nspack_probe.h -- a measurement helper of the GB300 packing library.
 *
 * The pages have no counterpart to this entry point: it measures the
 * arithmetic ceiling of one kernel.  The held-out hash adds, for every token
 * of a document, SplitMix64((i << 32) | token) (i its index in the document;
 * NeuronSpark-Trainer README, Concepts: held out by a hash of the document's
 * text), and on this GPU it is bound by the integer pipe, not by memory.
 * This call runs that term in a loop that reads no memory, so that a
 * benchmark can time it and report the hash kernel's rate as a fraction of
 * it.
 */
#ifndef NSPACK_PROBE_H
#define NSPACK_PROBE_H

#include <stdint.h>

#include "nspack.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Launch `blocks` blocks of 256 threads on cuda_stream (NULL: the legacy
 * default stream), asynchronously; thread g (g = block * 256 + thread)
 * computes terms_per_thread terms, the t-th with index (g mod 1024) + t and
 * token (g * 2654435761 mod 2^32) xor t, and adds its wrapping sum of them to
 * *sum_dev (device, 8-byte aligned, not cleared here).  The terms computed
 * are blocks * 256 * terms_per_thread.  Errors: INVALID_ARG (NULL or
 * misaligned sum_dev, blocks 0 or above 2^20), CUDA. */
int ns_pack_probe_hash_terms(uint32_t blocks, uint32_t terms_per_thread, uint64_t *sum_dev,
                             void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* NSPACK_PROBE_H */
