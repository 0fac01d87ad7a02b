/*
 * attn_pdump.h -- test build of the library only (libpa_gb300_pdump.so, built
 * from the same sources with PA_PDUMP defined). The timed library does not
 * export this call and its kernels carry none of the code behind it.
 *
 * Where several results are correct, a parity test has to see which one the
 * device chose. A probability lying within fp32 rounding of an E4M3 rounding
 * boundary has two faithful codes ("Fused attention kernel", 8-bit forward
 * pass: P is cast to e4m3 before the P V product; the device evaluates the
 * scores in its own fp32 summation order and 2^x with an approximation), so
 * the test build writes every probability code it hands to the P V MMA to a
 * caller buffer, and the test checks each code against the oracle's tie band
 * before it uses them.
 */
#ifndef PA_GB300_ATTN_PDUMP_H
#define PA_GB300_ATTN_PDUMP_H

#include <stdint.h>

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Every FP8 forward call made after this one writes its E4M3 probability codes
 * to `buf` (device, 16-byte aligned, caller-owned; NULL stops the writes):
 * byte [(h * T + t) * key_stride + k] receives the code that row t of head h
 * gave the document-local key k, for every key tile the row's work item
 * visits (keys the row does not see get code 0); rows and keys outside are
 * left untouched. key_stride: a multiple of 128 at least 128 x the key tiles
 * of the longest document, else ATTN_ERR_INVALID_ARG. Host-only, process-wide;
 * returns ATTN_OK. */
attn_status attn_pdump_set(void* buf, int64_t key_stride);

#ifdef __cplusplus
}
#endif
#endif
