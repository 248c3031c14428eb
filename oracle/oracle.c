/*
 * Sorting oracle (see oracle.h).  TEST INFRASTRUCTURE ONLY: plain, slow,
 * single-threaded C, written from the pages' descriptions and sharing nothing
 * with the CUDA library.
 *
 * Page names used below:
 *   [kwkr]    kwkr.cn "bitonic sort vs LSD radix sort" practice notes
 *   [quant67] "并行排序：从归并网络到 GPU 双调排序"
 *   [bjdmk]   "GPU基数排序：从CUB工程实现到性能调优"
 */
#include "oracle.h"

#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Key encodings                                                             */
/* ------------------------------------------------------------------------ */

int orc_key_bits(int kind) {
    switch (kind) {
    case ORC_U32:
    case ORC_I32:
    case ORC_F32: return 32;
    case ORC_U64:
    case ORC_I64:
    case ORC_F64: return 64;
    default: return 0;
    }
}

static uint64_t width_mask(int kind) {
    return orc_key_bits(kind) == 64 ? ~(uint64_t)0 : (uint64_t)0xFFFFFFFFu;
}

/*
 * [bjdmk] §5.1: unsigned integers are sorted as they are.
 * [bjdmk] §5.2: a signed 32-bit integer is sorted as (x XOR 0x80000000), which
 *   sends INT_MIN to 0 and INT_MAX to 0xFFFFFFFF.  ([kwkr] §3.3 says the
 *   negatives should be inverted as well; for two's complement that reverses
 *   their order, so the [bjdmk] form is the one used.)
 * [kwkr] §3.3 and [bjdmk] §5.3: an IEEE-754 float with the sign bit set has all
 *   its bits inverted, otherwise only the sign bit is flipped.
 * [bjdmk] §5.3: a double takes the same treatment over 64 bits; a signed
 *   64-bit integer flips its sign bit as the 32-bit one does (§5.2).
 * Descending order is the ascending order of the complemented code.
 */
uint64_t orc_key_transform(int kind, uint64_t raw, int descending) {
    uint64_t t;
    switch (kind) {
    case ORC_U32:
        t = raw & 0xFFFFFFFFu;
        break;
    case ORC_I32:
        t = (raw & 0xFFFFFFFFu) ^ 0x80000000u;
        break;
    case ORC_F32: {
        uint32_t b = (uint32_t)raw;
        if (b & 0x80000000u)
            b = b ^ 0xFFFFFFFFu;
        else
            b = b ^ 0x80000000u;
        t = b;
        break;
    }
    case ORC_U64:
        t = raw;
        break;
    case ORC_I64:
        t = raw ^ ((uint64_t)1 << 63);
        break;
    case ORC_F64:
        if (raw >> 63)
            t = ~raw;
        else
            t = raw ^ ((uint64_t)1 << 63);
        break;
    default:
        return 0;
    }
    if (descending) t = ~t & width_mask(kind);
    return t;
}

uint64_t orc_key_inverse(int kind, uint64_t t, int descending) {
    if (descending) t = ~t & width_mask(kind);
    switch (kind) {
    case ORC_U32: return t & 0xFFFFFFFFu;
    case ORC_I32: return (t & 0xFFFFFFFFu) ^ 0x80000000u;
    case ORC_F32: {
        uint32_t b = (uint32_t)t;
        /* A code with the top bit set came from a non-negative float. */
        if (b & 0x80000000u)
            b = b ^ 0x80000000u;
        else
            b = b ^ 0xFFFFFFFFu;
        return b;
    }
    case ORC_U64: return t;
    case ORC_I64: return t ^ ((uint64_t)1 << 63);
    case ORC_F64:
        /* A code with the top bit set came from a non-negative double. */
        return (t >> 63) ? t ^ ((uint64_t)1 << 63) : ~t;
    default: return 0;
    }
}

static uint64_t load_raw(int kind, const void *keys, size_t i) {
    if (orc_key_bits(kind) == 64) return ((const uint64_t *)keys)[i];
    return ((const uint32_t *)keys)[i];
}

static void store_raw(int kind, void *keys, size_t i, uint64_t v) {
    if (orc_key_bits(kind) == 64)
        ((uint64_t *)keys)[i] = v;
    else
        ((uint32_t *)keys)[i] = (uint32_t)v;
}

int orc_key_transform_array(int kind, const void *raw, size_t n, int descending,
                            uint64_t *codes) {
    if (orc_key_bits(kind) == 0) return -1;
    for (size_t i = 0; i < n; ++i) codes[i] = orc_key_transform(kind, load_raw(kind, raw, i), descending);
    return 0;
}

int orc_key_inverse_array(int kind, const uint64_t *codes, size_t n, int descending,
                          void *raw) {
    if (orc_key_bits(kind) == 0) return -1;
    for (size_t i = 0; i < n; ++i) store_raw(kind, raw, i, orc_key_inverse(kind, codes[i], descending));
    return 0;
}

static int check_range(int kind, int begin_bit, int end_bit) {
    int w = orc_key_bits(kind);
    if (w == 0) return -1;
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > w) return -2;
    return 0;
}

int orc_num_passes(int begin_bit, int end_bit) {
    if (end_bit <= begin_bit) return 0;
    return (end_bit - begin_bit + 7) / 8;
}

/* Digit p: bits [begin + 8p, min(begin + 8p + 8, end)) of the code t.
 * [bjdmk] §2: bit ranges are half-open and the passes walk up one byte at a
 * time from begin_bit; a narrower last digit sits at the top. */
static unsigned digit_of(uint64_t t, int begin_bit, int end_bit, int p) {
    int shift = begin_bit + 8 * p;
    int width = end_bit - shift;
    if (width > 8) width = 8;
    return (unsigned)((t >> shift) & (((uint64_t)1 << width) - 1));
}

int orc_digit_histograms(int kind, const void *keys, size_t n, int begin_bit,
                         int end_bit, int descending, uint64_t *hist) {
    int rc = check_range(kind, begin_bit, end_bit);
    if (rc) return rc;
    int passes = orc_num_passes(begin_bit, end_bit);
    memset(hist, 0, sizeof(uint64_t) * 256 * (size_t)passes);
    for (size_t i = 0; i < n; ++i) {
        uint64_t t = orc_key_transform(kind, load_raw(kind, keys, i), descending);
        for (int p = 0; p < passes; ++p)
            hist[(size_t)p * 256 + digit_of(t, begin_bit, end_bit, p)] += 1;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* LSD radix sort                                                            */
/* ------------------------------------------------------------------------ */

/*
 * [kwkr] §3.1, the serial LSD radix sort: for every 8-bit digit from the low
 * end, (1) count how many keys fall in each of the 256 buckets, (2) turn the
 * counts into an exclusive prefix sum, (3) walk the keys in their current
 * order and place each at its bucket's cursor, advancing the cursor, then
 * swap the roles of the two buffers.  Step (3) visits keys in order, which is
 * what makes each pass stable ([bjdmk] §3 and §6 on why LSD needs a stable
 * scatter).  Values ride along with their keys.
 */
int orc_lsd_radix_sort(int kind, const void *keys_in, const uint32_t *vals_in,
                       size_t n, int begin_bit, int end_bit, int descending,
                       void *keys_out, uint32_t *vals_out) {
    int rc = check_range(kind, begin_bit, end_bit);
    if (rc) return rc;
    if ((vals_in == NULL) != (vals_out == NULL)) return -3;
    int passes = orc_num_passes(begin_bit, end_bit);

    uint64_t *data = (uint64_t *)malloc(sizeof(uint64_t) * (n ? n : 1));
    uint64_t *out = (uint64_t *)malloc(sizeof(uint64_t) * (n ? n : 1));
    uint32_t *vdata = NULL, *vout = NULL;
    if (vals_in) {
        vdata = (uint32_t *)malloc(sizeof(uint32_t) * (n ? n : 1));
        vout = (uint32_t *)malloc(sizeof(uint32_t) * (n ? n : 1));
    }
    if (!data || !out || (vals_in && (!vdata || !vout))) {
        free(data); free(out); free(vdata); free(vout);
        return -4;
    }
    for (size_t i = 0; i < n; ++i) {
        data[i] = orc_key_transform(kind, load_raw(kind, keys_in, i), descending);
        if (vdata) vdata[i] = vals_in[i];
    }

    for (int p = 0; p < passes; ++p) {
        size_t count[256];
        for (int d = 0; d < 256; ++d) count[d] = 0;
        for (size_t i = 0; i < n; ++i) count[digit_of(data[i], begin_bit, end_bit, p)] += 1;
        size_t total = 0;
        for (int d = 0; d < 256; ++d) {
            size_t c = count[d];
            count[d] = total;
            total += c;
        }
        for (size_t i = 0; i < n; ++i) {
            unsigned d = digit_of(data[i], begin_bit, end_bit, p);
            size_t pos = count[d]++;
            out[pos] = data[i];
            if (vdata) vout[pos] = vdata[i];
        }
        uint64_t *tk = data; data = out; out = tk;
        uint32_t *tv = vdata; vdata = vout; vout = tv;
    }

    for (size_t i = 0; i < n; ++i) {
        store_raw(kind, keys_out, i, orc_key_inverse(kind, data[i], descending));
        if (vals_out) vals_out[i] = vdata[i];
    }
    free(data); free(out); free(vdata); free(vout);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Bitonic network                                                           */
/* ------------------------------------------------------------------------ */

/* State of one run of the network: the array, comparator count and, per
 * wire, the layer of the last comparator that touched it (for the depth). */
typedef struct {
    uint64_t *a;
    uint64_t comparators;
    uint64_t *layer;
    uint64_t depth;
} net_t;

/* [quant67] §1.1 / §3.3 compare_swap: with dir = 1 the smaller value ends on
 * wire i, with dir = 0 the larger one does. */
static void compare_swap(net_t *s, size_t i, size_t j, int dir) {
    s->comparators += 1;
    if (s->layer) {
        uint64_t l = (s->layer[i] > s->layer[j] ? s->layer[i] : s->layer[j]) + 1;
        s->layer[i] = s->layer[j] = l;
        if (l > s->depth) s->depth = l;
    }
    if (dir == (s->a[i] > s->a[j])) {
        uint64_t tmp = s->a[i];
        s->a[i] = s->a[j];
        s->a[j] = tmp;
    }
}

/* [quant67] §3.3 bitonic_merge: split (compare lo+i with lo+i+cnt/2), then
 * merge both halves recursively in the same direction. */
static void bitonic_merge(net_t *s, size_t lo, size_t cnt, int dir) {
    if (cnt <= 1) return;
    size_t k = cnt / 2;
    for (size_t i = lo; i < lo + k; ++i) compare_swap(s, i, i + k, dir);
    bitonic_merge(s, lo, k, dir);
    bitonic_merge(s, lo + k, k, dir);
}

/* [quant67] §3.3 bitonic_sort: left half ascending, right half descending,
 * which makes the whole a bitonic sequence, then merge in direction dir.
 * ([kwkr] §2.2 gives the same recursion.) */
static void bitonic_sort_rec(net_t *s, size_t lo, size_t cnt, int dir) {
    if (cnt <= 1) return;
    size_t k = cnt / 2;
    bitonic_sort_rec(s, lo, k, 1);
    bitonic_sort_rec(s, lo + k, k, 0);
    bitonic_merge(s, lo, cnt, dir);
}

static size_t next_pow2(size_t n) {
    size_t p = 1;
    while (p < n) p <<= 1;
    return p;
}

/*
 * Sorts the codes of one array.  Non-power-of-two lengths are padded
 * ([quant67] §3.5 method 1, [kwkr] §5.1): the pad must land after every real
 * key, so it is the all-ones code when sorting up and the all-zeros code when
 * sorting down.  Descending uses the network's own direction flag on the
 * plain (uncomplemented) codes.
 */
int orc_bitonic_sort(int kind, const void *keys_in, size_t len, int descending,
                     void *keys_out, uint64_t *comparators, uint64_t *depth) {
    if (orc_key_bits(kind) == 0) return -1;
    size_t m = next_pow2(len ? len : 1);
    net_t s;
    s.a = (uint64_t *)malloc(sizeof(uint64_t) * m);
    s.layer = (depth != NULL) ? (uint64_t *)calloc(m, sizeof(uint64_t)) : NULL;
    if (!s.a || (depth && !s.layer)) {
        free(s.a); free(s.layer);
        return -4;
    }
    s.comparators = 0;
    s.depth = 0;
    int up = descending ? 0 : 1;
    uint64_t pad = up ? width_mask(kind) : 0;
    for (size_t i = 0; i < m; ++i)
        s.a[i] = i < len ? orc_key_transform(kind, load_raw(kind, keys_in, i), 0) : pad;
    bitonic_sort_rec(&s, 0, m, up);
    for (size_t i = 0; i < len; ++i) store_raw(kind, keys_out, i, orc_key_inverse(kind, s.a[i], 0));
    if (comparators) *comparators = s.comparators;
    if (depth) *depth = s.depth;
    free(s.a);
    free(s.layer);
    return 0;
}

int orc_segmented_sort(int kind, const void *keys_in, size_t num_segments,
                       size_t seg_len, int descending, void *keys_out) {
    if (orc_key_bits(kind) == 0) return -1;
    size_t w = (size_t)orc_key_bits(kind) / 8;
    for (size_t s = 0; s < num_segments; ++s) {
        const char *src = (const char *)keys_in + s * seg_len * w;
        char *dst = (char *)keys_out + s * seg_len * w;
        int rc = orc_bitonic_sort(kind, src, seg_len, descending, dst, NULL, NULL);
        if (rc) return rc;
    }
    return 0;
}

static int is_pow2(size_t n) { return n != 0 && (n & (n - 1)) == 0; }

int orc_bitonic_split_u32(uint32_t *a, size_t cnt, int up) {
    if (!is_pow2(cnt)) return -1;
    net_t s;
    s.a = (uint64_t *)malloc(sizeof(uint64_t) * cnt);
    if (!s.a) return -4;
    s.layer = NULL;
    s.comparators = 0;
    s.depth = 0;
    for (size_t i = 0; i < cnt; ++i) s.a[i] = a[i];
    size_t k = cnt / 2;
    for (size_t i = 0; i < k; ++i) compare_swap(&s, i, i + k, up ? 1 : 0);
    for (size_t i = 0; i < cnt; ++i) a[i] = (uint32_t)s.a[i];
    free(s.a);
    return 0;
}

int orc_bitonic_merge_u32(uint32_t *a, size_t cnt, int up) {
    if (!is_pow2(cnt)) return -1;
    net_t s;
    s.a = (uint64_t *)malloc(sizeof(uint64_t) * cnt);
    if (!s.a) return -4;
    s.layer = NULL;
    s.comparators = 0;
    s.depth = 0;
    for (size_t i = 0; i < cnt; ++i) s.a[i] = a[i];
    bitonic_merge(&s, 0, cnt, up ? 1 : 0);
    for (size_t i = 0; i < cnt; ++i) a[i] = (uint32_t)s.a[i];
    free(s.a);
    return 0;
}
