/*
 * gbsort — device-wide sorting of fixed-length keys on NVIDIA GB300 (sm_103a).
 *
 * C ABI of the CUDA library.  Every entry point takes plain pointers and
 * sizes; device pointers are CUDA global-memory addresses on the current
 * device, and `stream` is a cudaStream_t (CUstream) handle, NULL meaning the
 * legacy default stream.  All work is enqueued on `stream`; no entry point
 * synchronises the stream except gbs_get_status.
 *
 * Method (web pages, cited by title and section):
 *  - LSD radix sort with 8-bit digits: per digit a histogram, an exclusive
 *    prefix over the buckets and a STABLE scatter, lowest digit first
 *    (kwkr.cn practice notes on bitonic sort vs LSD radix sort, §3.1-3.2;
 *    "GPU基数排序：从CUB工程实现到性能调优", §3).
 *  - Order-preserving key maps for signed integers and IEEE-754 floats
 *    (kwkr.cn notes §3.3; "GPU基数排序", §5.2-5.3).
 *  - Half-open bit ranges [begin_bit, end_bit), a size query with a NULL
 *    work buffer, a reusable caller-owned work buffer, in-place calls
 *    ("GPU基数排序", §2 and §6).
 *  - Bitonic compare-exchange network, partner i^j, direction from the
 *    segment bit (i & k), padding to a power of two with a maximal sentinel
 *    ("并行排序：从归并网络到 GPU 双调排序", §3.3-3.5 and §4.2-4.3;
 *    kwkr.cn notes §2.2-2.4 and §5.1).
 *
 * Ownership: the caller allocates and frees every buffer, including the work
 * buffer `d_temp`.  The library allocates no memory on any sort call.
 *
 * Work-buffer protocol: call once with d_temp == NULL; *temp_bytes receives
 * the size needed for these arguments and nothing is launched.  Then call
 * with a device buffer of at least that many bytes (256-byte aligned) and
 * *temp_bytes set to its size.  A buffer may be reused by later calls on the
 * same stream; calls that share one buffer must not run concurrently.
 *
 * Errors: arguments are checked on the host before anything is launched and
 * the call returns a status other than GBS_OK without touching memory.
 * A CUDA launch failure returns GBS_ERR_CUDA.  Faults found on the device
 * (a bounded wait that ran out) are recorded in the work buffer and
 * reported by gbs_get_status.
 */
#ifndef GBSORT_H
#define GBSORT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GBS_OK = 0,
    GBS_ERR_INVALID_ARG = 1,    /* null pointer, bad bit range, bad key type, ... */
    GBS_ERR_TEMP_TOO_SMALL = 2, /* *temp_bytes below the queried size */
    GBS_ERR_UNSUPPORTED = 3,    /* size beyond the library's limits */
    GBS_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
    GBS_ERR_TIMEOUT = 5         /* a device-side bounded wait ran out */
} gbs_status;

typedef enum {
    GBS_U32 = 0, /* uint32_t, sorted as unsigned */
    GBS_I32 = 1, /* int32_t, two's complement; code = x ^ 0x80000000 */
    GBS_F32 = 2, /* IEEE-754 binary32; code = b ^ (sign ? 0xFFFFFFFF : 0x80000000).
                    -0.0 sorts before +0.0; -inf and +inf are the extremes;
                    a NaN sorts by its bits (+NaN after +inf, -NaN before -inf). */
    GBS_U64 = 3, /* uint64_t, sorted as unsigned */
    GBS_I64 = 4, /* int64_t, two's complement; code = x ^ 0x8000000000000000 */
    GBS_F64 = 5  /* IEEE-754 binary64; code = b ^ (sign ? all ones : 0x8000000000000000),
                    the f32 map over 64 bits ("GPU基数排序" §5.3): -0.0 before +0.0,
                    infinities at the extremes, a NaN by its bits */
} gbs_key_type;

/* Largest number of keys a radix sort call accepts: keys, positions and
 * per-digit counts are 32-bit.  Sorts of 2^29 keys or more keep their
 * look-back status in 64-bit words (about 2 KiB per 8192-key tile instead of
 * 1 KiB, which the work-buffer size query includes). */
#define GBS_MAX_RADIX_KEYS ((size_t)0xFFFFFFFFu)
/* Longest segment that one CTA's bitonic network sorts on chip; longer
 * segments take the radix path. */
#define GBS_MAX_SEGMENT_LEN ((size_t)16384)

/*
 * gbs_sort_keys — sort n keys by the bits [begin_bit, end_bit) of their code
 * (the key itself for unsigned types, the order-preserving map above for i32
 * and f32).  Equal codes keep their input order (stable; LSD radix sort:
 * kwkr.cn notes §3.1, "GPU基数排序" §3).  Descending order (descending != 0)
 * is the stable ascending order of the complemented code: keys
 * non-increasing, equal keys in input order.  Output keys are the full
 * original keys, bit for bit.
 *   d_keys_in   device array of n keys (not modified unless equal to d_keys_out)
 *   d_keys_out  device array of n keys; may equal d_keys_in (in place);
 *               partial overlap is not allowed
 *   n           number of keys, at most GBS_MAX_RADIX_KEYS
 *   begin_bit, end_bit  0 <= begin_bit <= end_bit <= key width in bits;
 *               begin_bit == end_bit copies the keys
 * Small full-width calls (n <= GBS_MAX_SEGMENT_LEN, begin_bit == 0,
 * end_bit == key width) run the one-CTA bitonic sorter; ties there are
 * bit-identical keys, so the result equals the stable one.
 */
gbs_status gbs_sort_keys(void *d_temp, size_t *temp_bytes, gbs_key_type key_type,
                         const void *d_keys_in, void *d_keys_out, size_t n,
                         int begin_bit, int end_bit, int descending, void *stream);

/*
 * gbs_sort_keys_host — gbs_sort_keys (same key types, bit range, order and
 * result) on keys in HOST memory: enqueues on `stream` a copy of the n keys
 * to the device, the sort, and a copy of the sorted keys back to h_keys_out.
 * The web pages sort device-resident arrays; this entry point adds the two
 * transfers around that sort for callers whose data lives on the host.
 *   h_keys_in   host array of n keys (not modified unless equal to h_keys_out)
 *   h_keys_out  host array of n keys; may equal h_keys_in
 *   d_temp      device work buffer (same protocol as gbs_sort_keys: query the
 *               size with d_temp == NULL); it holds the sort's own work buffer
 *               followed by the keys' device copy (about n * key size more)
 * Page-locked host buffers (cudaHostAlloc, cudaHostRegister) make both copies
 * asynchronous; with pageable buffers the call blocks during the copies.
 * The call returns once everything is enqueued: synchronise `stream` (or call
 * gbs_get_status, which does) before reading h_keys_out.  The transfers run
 * at the host link's rate, which bounds the call's throughput.
 */
gbs_status gbs_sort_keys_host(void *d_temp, size_t *temp_bytes, gbs_key_type key_type, const void *h_keys_in,
                              void *h_keys_out, size_t n, int begin_bit, int end_bit, int descending, void *stream);

/*
 * gbs_sort_keys_host_batch — gbs_sort_keys_host on `count` independent host
 * arrays (same key type, bit range and order for all), with the transfers of
 * neighbouring arrays overlapped: while array i is sorted on `stream`, array
 * i + 1 is copied to the device and array i - 1 copied back, on two streams
 * of the library's own (created for the call with their events and released
 * when it returns; no memory is allocated).  The two directions of the host
 * link then run at the same time.  Each array's result equals
 * gbs_sort_keys_host's.
 *   h_keys_in[i], h_keys_out[i]  host arrays of n[i] keys.  h_keys_out[i]
 *               may equal h_keys_in[i] (in place) but must not overlap any
 *               other entry's input; inputs may repeat, and so may outputs
 *               (the copies back run in batch order: a repeated output ends
 *               holding the result of its last entry)
 *   n           host array of the count sizes, each at most GBS_MAX_RADIX_KEYS
 *   count       number of arrays (0: only the status header is cleared)
 *   d_temp      device work buffer (query with d_temp == NULL): one sort work
 *               buffer for the largest n[i], then three device key buffers of
 *               that size (an array's buffer is reused by array i + 3 once its
 *               copy back has finished)
 * The sorts run one after another on `stream`; the copies start after the
 * work enqueued on `stream` before the call, and everything the call enqueues
 * has finished when `stream` reaches the call's end, so the caller
 * synchronises `stream` alone.  Page-locked host buffers are needed for the
 * overlap.  gbs_get_status(d_temp, ...) reports the first device-side error
 * of any sort in the batch.  Errors: GBS_ERR_INVALID_ARG (a NULL array with
 * count > 0, a NULL pointer for an array with n[i] > 0, a bad bit range),
 * GBS_ERR_UNSUPPORTED (an n[i] above GBS_MAX_RADIX_KEYS), GBS_ERR_CUDA (a
 * failed enqueue: the work enqueued before it still joins `stream`).
 */
gbs_status gbs_sort_keys_host_batch(void *d_temp, size_t *temp_bytes, gbs_key_type key_type,
                                    const void *const *h_keys_in, void *const *h_keys_out, const size_t *n,
                                    size_t count, int begin_bit, int end_bit, int descending, void *stream);

/*
 * gbs_sort_pairs — like gbs_sort_keys, moving one uint32_t value with each
 * key.  Stable: pairs with equal codes keep their input order.
 *   d_vals_in / d_vals_out  device arrays of n uint32_t; may be equal
 */
gbs_status gbs_sort_pairs(void *d_temp, size_t *temp_bytes, gbs_key_type key_type,
                          const void *d_keys_in, void *d_keys_out,
                          const uint32_t *d_vals_in, uint32_t *d_vals_out, size_t n,
                          int begin_bit, int end_bit, int descending, void *stream);

/*
 * gbs_sort_pairs64 — gbs_sort_pairs with one uint64_t value per key (for
 * payloads such as 64-bit indices or pointers).  Stable.
 *   d_vals_in / d_vals_out  device arrays of n uint64_t; may be equal
 */
gbs_status gbs_sort_pairs64(void *d_temp, size_t *temp_bytes, gbs_key_type key_type,
                            const void *d_keys_in, void *d_keys_out,
                            const uint64_t *d_vals_in, uint64_t *d_vals_out, size_t n,
                            int begin_bit, int end_bit, int descending, void *stream);

/*
 * gbs_segmented_sort — sort each of num_segments consecutive segments of
 * segment_len keys independently, over the full key width.  Segments of up
 * to GBS_MAX_SEGMENT_LEN keys run the bitonic network, one segment per CTA
 * (or warp), padded on chip with a sentinel that sorts after every key when
 * the length is not a power of two ("并行排序" §3.3-3.5, §4.2-4.3).  Longer
 * segments run the radix sort, one segment after another in one radix work
 * area (the bitonic network of one CTA holds at most 2^14 keys).
 *   segment_len  1 .. GBS_MAX_RADIX_KEYS (0 segments or length 0: no work)
 *   d_keys_out may equal d_keys_in.
 *   d_temp       work buffer: a status header, plus a radix work area for
 *                segment_len keys when segment_len > GBS_MAX_SEGMENT_LEN
 * Device-side timeouts of the radix part are reported by gbs_get_status on
 * d_temp (the first one wins).
 */
gbs_status gbs_segmented_sort(void *d_temp, size_t *temp_bytes, gbs_key_type key_type,
                              const void *d_keys_in, void *d_keys_out,
                              size_t num_segments, size_t segment_len,
                              int descending, void *stream);

/*
 * gbs_segmented_sort_offsets — sort each of num_segments segments of any
 * length independently, over the full key width: segment s is the keys
 * [h_offsets[s], h_offsets[s+1]) of d_keys_in, sorted into the same places
 * of d_keys_out.  Segments of up to GBS_MAX_SEGMENT_LEN keys run the bitonic
 * network, each padded only to its own power of two (the pages advise
 * against padding every segment to one common size: kwkr.cn notes §5.3);
 * longer segments run the radix sort one after another.
 *   h_offsets   HOST array of num_segments + 1 non-decreasing 64-bit offsets,
 *               read during the call (the size query needs them too); each
 *               segment at most GBS_MAX_RADIX_KEYS keys; every offset must lie
 *               within both key arrays (not checked: the arrays' sizes are not
 *               passed)
 *   d_keys_out  may equal d_keys_in; keys outside the segments are not written
 *   d_temp      work buffer (query its size with d_temp == NULL and the same
 *               offsets): the offsets and a segment list by length class, plus
 *               a radix work area for the longest segment above 2^14 keys
 * Decreasing offsets return GBS_ERR_INVALID_ARG.  Device-side timeouts of the
 * radix part are reported by gbs_get_status on d_temp (the first one wins).
 */
gbs_status gbs_segmented_sort_offsets(void *d_temp, size_t *temp_bytes, gbs_key_type key_type, const void *d_keys_in,
                                      void *d_keys_out, size_t num_segments, const uint64_t *h_offsets,
                                      int descending, void *stream);

/*
 * gbs_sort_keys_msd_bitonic — gbs_sort_keys over the full key width (same
 * key types, order and result) by the pages' hybrid: most-significant-digit
 * radix passes group the keys by the top 16 bits of their code into 65536
 * buckets, then the bitonic network sorts every bucket on chip, each padded
 * only to its own power of two (kwkr.cn notes §5.3: bucket by the high bits,
 * bitonic-sort each bucket; §3.4 and §5.2 on cutting radix passes).  Keys
 * only, full width; buckets above GBS_MAX_SEGMENT_LEN keys take the radix
 * path.  A measured alternative to gbs_sort_keys, not its replacement.
 * Unlike the other entry points it synchronises `stream` once (the bucket
 * plan is made on the host).  Same work-buffer protocol; device-side
 * timeouts are reported by the return value or by gbs_get_status.
 */
gbs_status gbs_sort_keys_msd_bitonic(void *d_temp, size_t *temp_bytes, gbs_key_type key_type,
                                     const void *d_keys_in, void *d_keys_out, size_t n,
                                     int descending, void *stream);

/*
 * gbs_digit_histograms — the upfront digit histograms of a radix sort on
 * their own: hist[p*256 + d] = number of keys whose digit p (bits
 * [begin_bit + 8p, min(begin_bit + 8p + 8, end_bit)) of the code,
 * complemented when descending) equals d (kwkr.cn notes §3.2, two-level
 * counting).  d_hist receives ceil((end_bit - begin_bit) / 8) * 256 uint32_t.
 * Same work-buffer protocol as gbs_sort_keys.
 */
gbs_status gbs_digit_histograms(void *d_temp, size_t *temp_bytes, gbs_key_type key_type,
                                const void *d_keys, size_t n, int begin_bit, int end_bit,
                                int descending, uint32_t *d_hist, void *stream);

/*
 * gbs_sort_keys_noalloc — gbs_sort_keys (same key types, bit range, order
 * and result) for callers that cannot allocate device memory: plug-ins
 * inside an application that owns every allocation, real-time loops that
 * cannot afford cudaMalloc's latency and implicit synchronisation, or
 * processes whose memory pool is fixed up front.  The web pages have no
 * counterpart to this entry point.
 *
 * The caller passes only its keys; the work buffer is one array of about
 * 8.4 MiB in the library's own device memory, which every GPU that loads the
 * library holds until the process exits.  No cudaMalloc, cudaFree or other
 * allocating call is made.
 *   n  at most GBS_NOALLOC_MAX_KEYS; larger n returns GBS_ERR_UNSUPPORTED
 *      and launches nothing.
 * Every call asks the runtime for the array's device address on the current
 * device (cudaGetSymbolAddress); the first call on a device also loads the
 * library's device code there, so make that first call before any stream
 * capture.  Every call, on every stream, shares the one array: calls whose
 * work overlaps on the GPU race and corrupt each other's results, so
 * serialise them (one stream, or events).  The array keeps the last call's
 * contents; each call clears what it needs to start at zero.  A device-side
 * timeout is recorded in the array's header; gbs_get_status_noalloc reports
 * it.
 */
#define GBS_NOALLOC_MAX_KEYS ((size_t)1 << 20)
gbs_status gbs_sort_keys_noalloc(gbs_key_type key_type, const void *d_keys_in, void *d_keys_out, size_t n,
                                 int begin_bit, int end_bit, int descending, void *stream);

/*
 * gbs_get_status_noalloc — gbs_get_status for gbs_sort_keys_noalloc, whose
 * work buffer is the library's own array on the current device: synchronises
 * `stream`, then returns GBS_ERR_TIMEOUT if the last call on this device
 * recorded a device-side timeout, else GBS_OK (GBS_ERR_CUDA if the stream or
 * the read reports an error).  Allocates nothing.  The web pages have no
 * counterpart.
 */
gbs_status gbs_get_status_noalloc(void *stream);

/*
 * gbs_get_status — synchronises `stream`, then reports GBS_ERR_TIMEOUT if the
 * last call that used this work buffer recorded a device-side timeout, else
 * GBS_OK (GBS_ERR_CUDA if the stream reports an error).  temp_bytes is the
 * size of d_temp.
 */
gbs_status gbs_get_status(const void *d_temp, size_t temp_bytes, void *stream);

/* Human-readable name of a status code (static storage). */
const char *gbs_status_string(gbs_status status);

/* Library version, e.g. "0.1.0" (static storage). */
const char *gbs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBSORT_H */
