/*
 * pagedkv_testing.h -- test hooks of the paged KV-cache library.  They are
 * not part of the method and have no counterpart on the pages: they exist
 * so that tests can reach error paths that correct inputs never take,
 * without faulting, trapping or hanging a GPU.  Never set them in a
 * program that serves requests.
 */
#ifndef PAGEDKV_TESTING_H
#define PAGEDKV_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* From the next call of paged_attention_decode (and of the decode pass of
 * paged_attention_decode_cascade) on, every warp that works on sequence
 * `sequence` stops after its first 16-token block as if its bounded wait for
 * the next block had run out: it records PKV_ERR_TIMEOUT with that sequence
 * as the detail (read by pkv_check), lets the copies it already issued land
 * (the drain waits keep their normal limit) and contributes nothing more to
 * the output.  No wait is shortened.  A negative value switches the hook
 * off (the default).  Process-wide; host-only. */
void pkv_testing_fail_decode_sequence(int32_t sequence);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_TESTING_H */
