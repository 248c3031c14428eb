/*
 * Sorting oracle: plain, slow, single-threaded CPU reference for the LSD radix
 * sort and the bitonic network.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA library: the key encodings, digit
 * extraction, counting sort and bitonic network are written out again here
 * from the pages' descriptions.
 *
 * Sources (web pages, cited by title and section):
 *  - "并行排序：从归并网络到 GPU 双调排序" (parallel sort, quant67):
 *      §1.1 comparator definition, §1.2 0-1 principle, §3.2 bitonic split,
 *      §3.3 recursive bitonic sort (compare_swap / bitonic_merge /
 *      bitonic_sort), §3.4 depth and size, §3.5 padding with +infinity,
 *      §11.3 stability.
 *  - kwkr.cn practice notes on bitonic sort vs LSD radix sort: §2.2 bitonic
 *      worked example, §3.1 serial LSD with 8-bit digits (count, exclusive
 *      prefix, stable placement, ping-pong), §3.3 float/int bit maps,
 *      §5.1 sentinel pitfalls.
 *  - "GPU基数排序：从CUB工程实现到性能调优" (bjdmk, GPU radix): §2 half-open
 *      [begin_bit, end_bit) bit range and per-byte pass order, §5.2 signed
 *      integer sign flip, §5.3 float map, §5.4 composite keys.
 *
 * Key kinds: 0 = u32, 1 = i32, 2 = f32 (raw IEEE-754 bits), 3 = u64,
 * 4 = i64, 5 = f64 (raw IEEE-754 bits).
 * Arrays are host memory owned by the caller.  Functions return 0 on success
 * and a negative number on a bad argument.
 */
#ifndef SORT_ORACLE_H
#define SORT_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_U32 = 0, ORC_I32 = 1, ORC_F32 = 2, ORC_U64 = 3, ORC_I64 = 4, ORC_F64 = 5 };

/* Width in bits of a key kind (32 or 64); 0 for an unknown kind. */
int orc_key_bits(int kind);

/* Order-preserving map of a raw key bit pattern to an unsigned integer whose
 * unsigned order is the key order; descending complements it. */
uint64_t orc_key_transform(int kind, uint64_t raw, int descending);
/* Inverse of orc_key_transform. */
uint64_t orc_key_inverse(int kind, uint64_t t, int descending);

/* Element-wise orc_key_transform / orc_key_inverse over n keys (codes are
 * always returned as uint64). */
int orc_key_transform_array(int kind, const void *raw, size_t n, int descending,
                            uint64_t *codes);
int orc_key_inverse_array(int kind, const uint64_t *codes, size_t n, int descending,
                          void *raw);

/* Number of 8-bit digit passes over [begin_bit, end_bit). */
int orc_num_passes(int begin_bit, int end_bit);

/* Digit histograms: hist[p*256 + d] = number of keys whose digit p (bits
 * [begin+8p, min(begin+8p+8, end)) of the transformed key) equals d.
 * hist must hold orc_num_passes(...)*256 entries. */
int orc_digit_histograms(int kind, const void *keys, size_t n, int begin_bit,
                         int end_bit, int descending, uint64_t *hist);

/* Stable LSD radix sort (8-bit digits from begin_bit upward).  Sorts by the
 * bits [begin_bit, end_bit) of the transformed key; outputs the full original
 * keys.  vals_in/vals_out may both be NULL (keys only).  keys_out may equal
 * keys_in, and vals_out may equal vals_in. */
int orc_lsd_radix_sort(int kind, const void *keys_in, const uint32_t *vals_in,
                       size_t n, int begin_bit, int end_bit, int descending,
                       void *keys_out, uint32_t *vals_out);

/* Recursive bitonic sort of one array of len keys (any len >= 0), padded to
 * the next power of two with a sentinel that sorts after every real key.
 * comparators/depth (may be NULL) receive the number of compare-exchange
 * operations executed and the number of comparator layers of the network. */
int orc_bitonic_sort(int kind, const void *keys_in, size_t len, int descending,
                     void *keys_out, uint64_t *comparators, uint64_t *depth);

/* Bitonic sort of num_segments consecutive segments of seg_len keys each. */
int orc_segmented_sort(int kind, const void *keys_in, size_t num_segments,
                       size_t seg_len, int descending, void *keys_out);

/* One bitonic split (half-cleaner) of a[0..cnt) in place: compare-exchange
 * (i, i + cnt/2) for i < cnt/2 in direction up (1 ascending, 0 descending).
 * cnt must be a power of two.  Operates on plain unsigned 32-bit values. */
int orc_bitonic_split_u32(uint32_t *a, size_t cnt, int up);

/* Bitonic merge of a bitonic sequence a[0..cnt) (power of two) in place. */
int orc_bitonic_merge_u32(uint32_t *a, size_t cnt, int up);

#ifdef __cplusplus
}
#endif

#endif
