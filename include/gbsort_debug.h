/*
 * gbsort test hooks.  Not part of the sorting API: these exist so that the
 * test suite can exercise the device-side bounded waits and count launches.
 * None of them is needed to sort; none changes results unless set.
 */
#ifndef GBSORT_DEBUG_H
#define GBSORT_DEBUG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Makes tile `tile` of digit pass `pass` of every later radix call skip
 * publishing its look-back status (pass < 0 switches the fault off), and
 * sets the number of polls after which a waiting tile gives up, records
 * GBS_ERR_TIMEOUT in the work buffer and carries on (0 restores the
 * default, about a second of waiting).  A call run with the fault on
 * returns wrong data and gbs_get_status reports GBS_ERR_TIMEOUT; the CUDA
 * context stays usable.  Process-wide setting; not thread-safe.
 */
void gbs_debug_set_lookback_fault(int pass, uint32_t tile, uint32_t spin_limit);

/*
 * Kernel timing hook.  With events != NULL, every later sorting call made by
 * the calling thread records events[0] on its stream right before its first
 * kernel and events[i] right after its i-th kernel (i < count), so that
 * cudaEventElapsedTime(events[i-1], events[i]) is the device time of kernel
 * i.  The events are cudaEvent_t handles created by the caller.  Pass NULL to
 * switch the hook off.  Calls with more kernels than count - 1 leave the rest
 * unrecorded.
 */
void gbs_debug_set_timing_events(void **events, int count);

/*
 * Digit width of the radix sort's later keys-only calls with fewer than 2^29
 * keys: 8 (the library's path, the default) or 11, a measured prototype with
 * 2048 digit values per pass (3 passes for 32-bit keys, 6 for 64-bit keys
 * instead of 4 and 8).  Same results; pairs and larger sorts keep 8-bit
 * digits.  Any other value restores 8.  Process-wide; not thread-safe.
 */
void gbs_debug_set_radix_bits(int bits);

/* Number of kernels the calling thread's last sorting call launched. */
int gbs_debug_last_launch_count(void);

/* Keys per tile of the radix pass kernel for a key width (4 or 8 bytes) and
 * a value width (0: keys only; 8: 64-bit values; any other non-zero: 32-bit
 * values). */
size_t gbs_debug_radix_tile_keys(int key_bytes, int value_bytes);

#ifdef __cplusplus
}
#endif

#endif /* GBSORT_DEBUG_H */
