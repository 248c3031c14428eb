// C ABI of the gbsort library: argument checks, work-buffer layout, dispatch
// between the radix path and the bitonic tile sorter, status reporting.
#include <algorithm>
#include <cstring>
#include <vector>

#include "../../include/gbsort.h"
#include "../../include/gbsort_debug.h"
#include "launch.h"

namespace {

using gbs::Header;

constexpr size_t ALIGN = 256;
constexpr uint32_t DEFAULT_SPIN_LIMIT = 1u << 22;

size_t round_up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }

int key_bytes_of(gbs_key_type kt) {
    switch (kt) {
    case GBS_U32:
    case GBS_I32:
    case GBS_F32: return 4;
    case GBS_U64:
    case GBS_I64:
    case GBS_F64: return 8;
    default: return 0;
    }
}

// test hooks (process-wide)
int g_fault_pass = -1;
uint32_t g_fault_tile = 0;
uint32_t g_spin_limit = DEFAULT_SPIN_LIMIT;
int g_radix_bits = 8;  // 11: keys-only sorts of fewer than 2^29 keys take the 11-bit-digit prototype
thread_local int t_launches = 0;
thread_local void **t_events = nullptr;
thread_local int t_event_count = 0;
thread_local int t_event_next = 0;

// Records events[0] before a call's first kernel (see gbs_debug_set_timing_events).
void timing_start(cudaStream_t s) {
    t_event_next = 0;
    if (t_events && t_event_count > 0 &&
        cudaEventRecord(reinterpret_cast<cudaEvent_t>(t_events[t_event_next++]), s) != cudaSuccess)
        (void)cudaGetLastError();  // a bad caller event must not be reported as a launch failure
}

// Work-buffer layout of a radix call.
struct Layout {
    size_t hist, digit_base, status, keys_alt, vals_alt, total;
    uint32_t num_tiles;
};

// The 11-bit-digit prototype serves this call (test hook; keys only, < 2^29 keys).
bool use_radix11(int val_bytes, size_t n) { return g_radix_bits == 11 && val_bytes == 0 && n < gbs::WIDE_STATUS_MIN_KEYS; }

Layout radix_layout(int key_bytes, int val_bytes, size_t n) {
    Layout l;
    const bool r11 = use_radix11(val_bytes, n);
    const uint32_t tile = r11 ? gbs::radix11_tile_keys(key_bytes) : gbs::radix_tile_keys(key_bytes, val_bytes);
    const size_t digits = r11 ? 2048 : 256;  // histogram and status words per digit position / tile
    l.num_tiles = (uint32_t)((n + tile - 1) / tile);
    size_t off = sizeof(Header);
    l.hist = off;
    off += round_up(sizeof(uint32_t) * gbs::MAX_PASSES * digits);
    l.digit_base = off;
    off += round_up(sizeof(uint32_t) * gbs::MAX_PASSES * digits);
    l.status = off;
    off += round_up(r11 ? sizeof(uint32_t) * digits * l.num_tiles : gbs::status_bytes(n, l.num_tiles));
    l.keys_alt = off;
    off += round_up((size_t)key_bytes * n);
    l.vals_alt = off;
    off += round_up((size_t)val_bytes * n);
    l.total = off;
    return l;
}

gbs_status check_temp(void *d_temp, size_t *temp_bytes, size_t need, bool *query) {
    *query = false;
    if (temp_bytes == nullptr) return GBS_ERR_INVALID_ARG;
    if (d_temp == nullptr) {
        *temp_bytes = need;
        *query = true;
        return GBS_OK;
    }
    if ((reinterpret_cast<uintptr_t>(d_temp) % ALIGN) != 0) return GBS_ERR_INVALID_ARG;
    if (*temp_bytes < need) return GBS_ERR_TEMP_TOO_SMALL;
    return GBS_OK;
}

gbs_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GBS_OK : GBS_ERR_CUDA; }

cudaError_t copy_if_needed(const void *src, void *dst, size_t bytes, cudaStream_t s) {
    if (src == dst || bytes == 0) return cudaSuccess;
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
}

// keep_error: leave the header's error words as they are (a call made of
// several sorts reports the first error of any of them).
// val_bytes: 0 (keys only), 4 or 8 bytes per value.
gbs_status radix_common(void *d_temp, size_t *temp_bytes, gbs_key_type kt, const void *keys_in, void *keys_out,
                        const void *vals_in, void *vals_out, int val_bytes, size_t n, int begin_bit, int end_bit,
                        int descending, void *stream, bool keep_error = false) {
    const bool pairs = val_bytes != 0;
    if (!keep_error) t_launches = 0;
    const int kb = key_bytes_of(kt);
    if (kb == 0) return GBS_ERR_INVALID_ARG;
    if (temp_bytes == nullptr) return GBS_ERR_INVALID_ARG;
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > 8 * kb) return GBS_ERR_INVALID_ARG;
    if (n > GBS_MAX_RADIX_KEYS) return GBS_ERR_UNSUPPORTED;
    const Layout lay = radix_layout(kb, val_bytes, n);
    bool query = false;
    gbs_status st = check_temp(d_temp, temp_bytes, lay.total, &query);
    if (st != GBS_OK || query) return st;
    if (n > 0 && (keys_in == nullptr || keys_out == nullptr)) return GBS_ERR_INVALID_ARG;
    if (pairs && n > 0 && (vals_in == nullptr || vals_out == nullptr)) return GBS_ERR_INVALID_ARG;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *tb = reinterpret_cast<unsigned char *>(d_temp);
    const size_t keep = keep_error ? 2 * sizeof(uint32_t) : 0;  // error, error_detail
    cudaError_t e = cudaMemsetAsync(tb + keep, 0, lay.digit_base - keep, s);  // header + histograms
    if (e != cudaSuccess) return GBS_ERR_CUDA;

    const bool r11 = use_radix11(val_bytes, n);
    const int passes = r11 ? (end_bit - begin_bit + 10) / 11 : (end_bit - begin_bit + 7) / 8;
    if (n <= 1 || passes == 0) {
        e = copy_if_needed(keys_in, keys_out, n * kb, s);
        if (e == cudaSuccess && pairs) e = copy_if_needed(vals_in, vals_out, n * (size_t)val_bytes, s);
        return from_cuda(e);
    }
    timing_start(s);
    // small full-width key sorts: one CTA of the bitonic sorter
    if (!pairs && n <= GBS_MAX_SEGMENT_LEN && begin_bit == 0 && end_bit == 8 * kb) {
        e = gbs::launch_segmented_bitonic((int)kt, kb, keys_in, keys_out, 1, n, descending != 0, s, &t_launches);
        return from_cuda(e);
    }

    gbs::RadixJob job;
    job.kind = (int)kt;
    job.key_bytes = kb;
    job.val_bytes = val_bytes;
    job.keys_in = keys_in;
    job.keys_out = keys_out;
    job.keys_alt = tb + lay.keys_alt;
    job.vals_in = vals_in;
    job.vals_out = vals_out;
    job.vals_alt = pairs ? static_cast<void *>(tb + lay.vals_alt) : nullptr;
    job.n = n;
    job.begin_bit = begin_bit;
    job.end_bit = end_bit;
    job.num_passes = passes;
    job.descending = descending != 0;
    job.in_place = (keys_in == keys_out) || (pairs && vals_in == vals_out);
    job.hdr = reinterpret_cast<Header *>(tb);
    job.hist = reinterpret_cast<uint32_t *>(tb + lay.hist);
    job.digit_base = reinterpret_cast<uint32_t *>(tb + lay.digit_base);
    job.status = tb + lay.status;
    job.wide_status = n >= gbs::WIDE_STATUS_MIN_KEYS;
    job.num_tiles = lay.num_tiles;
    job.spin_limit = g_spin_limit;
    job.fault_pass = g_fault_pass;
    job.fault_tile = g_fault_tile;
    if (r11) return from_cuda(gbs::launch_radix11_sort(job, s, &t_launches));
    return from_cuda(gbs::launch_radix_sort(job, s, &t_launches));
}

}  // namespace

namespace gbs {
void debug_fault_settings(int *fault_pass, uint32_t *fault_tile, uint32_t *spin_limit) {
    *fault_pass = g_fault_pass;
    *fault_tile = g_fault_tile;
    *spin_limit = g_spin_limit;
}

void timing_mark(cudaStream_t s) {
    if (t_events && t_event_next > 0 && t_event_next < t_event_count &&
        cudaEventRecord(reinterpret_cast<cudaEvent_t>(t_events[t_event_next++]), s) != cudaSuccess)
        (void)cudaGetLastError();
}
}  // namespace gbs

static_assert(GBS_MAX_RADIX_KEYS <= gbs::StatusWord<uint64_t>::MAX_KEYS, "key limit must fit the status words");
static_assert((int)GBS_U32 == gbs::KIND_U32 && (int)GBS_I32 == gbs::KIND_I32 && (int)GBS_F32 == gbs::KIND_F32 &&
                  (int)GBS_U64 == gbs::KIND_U64 && (int)GBS_I64 == gbs::KIND_I64 && (int)GBS_F64 == gbs::KIND_F64,
              "the ABI's key types are the kernels' key kinds");

namespace {
// Streams and events of one batch call, released when the call returns (work
// still pending on them completes first: the runtime defers the release).
struct BatchStreams {
    static constexpr int SLOTS = 3;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, in_done[SLOTS] = {}, sorted[SLOTS] = {}, out_done[SLOTS] = {};
    cudaEvent_t in_end = nullptr, out_end = nullptr;
    cudaError_t create() {
        cudaError_t e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking);
        cudaEvent_t *all[] = {&start, &in_end, &out_end};
        for (cudaEvent_t *ev : all)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        for (int j = 0; j < SLOTS && e == cudaSuccess; ++j) {
            e = cudaEventCreateWithFlags(&in_done[j], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sorted[j], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&out_done[j], cudaEventDisableTiming);
        }
        return e;
    }
    ~BatchStreams() {
        cudaEvent_t evs[] = {start, in_end, out_end, in_done[0], in_done[1], in_done[2], sorted[0], sorted[1],
                             sorted[2], out_done[0], out_done[1], out_done[2]};
        for (cudaEvent_t ev : evs)
            if (ev) cudaEventDestroy(ev);
        if (in) cudaStreamDestroy(in);
        if (out) cudaStreamDestroy(out);
    }
};
}  // namespace

extern "C" {

gbs_status gbs_sort_keys(void *d_temp, size_t *temp_bytes, gbs_key_type key_type, const void *d_keys_in,
                         void *d_keys_out, size_t n, int begin_bit, int end_bit, int descending, void *stream) {
    return radix_common(d_temp, temp_bytes, key_type, d_keys_in, d_keys_out, nullptr, nullptr, 0, n, begin_bit,
                        end_bit, descending, stream);
}

gbs_status gbs_sort_keys_host(void *d_temp, size_t *temp_bytes, gbs_key_type key_type, const void *h_keys_in,
                              void *h_keys_out, size_t n, int begin_bit, int end_bit, int descending, void *stream) {
    const int kb = key_bytes_of(key_type);
    if (kb == 0 || temp_bytes == nullptr) return GBS_ERR_INVALID_ARG;
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > 8 * kb) return GBS_ERR_INVALID_ARG;
    if (n > GBS_MAX_RADIX_KEYS) return GBS_ERR_UNSUPPORTED;
    // work buffer: the in-place device sort's own work buffer first (so that
    // gbs_get_status finds its header at d_temp), then the keys' device copy
    size_t sort_bytes = 0;
    gbs_status st = radix_common(nullptr, &sort_bytes, key_type, nullptr, nullptr, nullptr, nullptr, 0, n,
                                 begin_bit, end_bit, descending, stream);
    if (st != GBS_OK) return st;
    const size_t keys_off = round_up(sort_bytes);
    bool query = false;
    st = check_temp(d_temp, temp_bytes, keys_off + round_up((size_t)kb * n), &query);
    if (st != GBS_OK || query) return st;
    if (n > 0 && (h_keys_in == nullptr || h_keys_out == nullptr)) return GBS_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *d_keys = reinterpret_cast<unsigned char *>(d_temp) + keys_off;
    if (n > 0 && cudaMemcpyAsync(d_keys, h_keys_in, n * kb, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return GBS_ERR_CUDA;
    size_t inner = keys_off;  // also clears the status header when n == 0
    st = radix_common(d_temp, &inner, key_type, d_keys, d_keys, nullptr, nullptr, 0, n, begin_bit, end_bit,
                      descending, stream);
    if (st != GBS_OK || n == 0) return st;
    return from_cuda(cudaMemcpyAsync(h_keys_out, d_keys, n * kb, cudaMemcpyDeviceToHost, s));
}


gbs_status gbs_sort_keys_host_batch(void *d_temp, size_t *temp_bytes, gbs_key_type key_type,
                                    const void *const *h_keys_in, void *const *h_keys_out, const size_t *n,
                                    size_t count, int begin_bit, int end_bit, int descending, void *stream) {
    constexpr int SLOTS = BatchStreams::SLOTS;
    const int kb = key_bytes_of(key_type);
    if (kb == 0 || temp_bytes == nullptr) return GBS_ERR_INVALID_ARG;
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > 8 * kb) return GBS_ERR_INVALID_ARG;
    if (count > 0 && (n == nullptr || h_keys_in == nullptr || h_keys_out == nullptr)) return GBS_ERR_INVALID_ARG;
    size_t max_n = 0;
    for (size_t i = 0; i < count; ++i) {
        if (n[i] > GBS_MAX_RADIX_KEYS) return GBS_ERR_UNSUPPORTED;
        max_n = std::max(max_n, n[i]);
    }
    // work buffer: one sort work buffer for the largest array (a smaller
    // array's layout fits inside it), then SLOTS device key buffers
    size_t sort_bytes = 0;
    gbs_status st = radix_common(nullptr, &sort_bytes, key_type, nullptr, nullptr, nullptr, nullptr, 0, max_n,
                                 begin_bit, end_bit, descending, stream);
    if (st != GBS_OK) return st;
    const size_t keys_off = round_up(sort_bytes), slot_bytes = round_up((size_t)kb * max_n);
    bool query = false;
    st = check_temp(d_temp, temp_bytes, keys_off + SLOTS * slot_bytes, &query);
    if (st != GBS_OK || query) return st;
    for (size_t i = 0; i < count; ++i)
        if (n[i] > 0 && (h_keys_in[i] == nullptr || h_keys_out[i] == nullptr)) return GBS_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    size_t inner = keys_off;
    if (count == 0)  // clears the status header, as a sort of no keys does
        return radix_common(d_temp, &inner, key_type, nullptr, nullptr, nullptr, nullptr, 0, 0, begin_bit, end_bit,
                            descending, stream);

    BatchStreams bs;
    if (bs.create() != cudaSuccess) return GBS_ERR_CUDA;
    // the copies follow the work enqueued on `stream` before the call
    cudaError_t e = cudaEventRecord(bs.start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(bs.in, bs.start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(bs.out, bs.start, 0);
    if (e != cudaSuccess) return GBS_ERR_CUDA;
    unsigned char *slots = reinterpret_cast<unsigned char *>(d_temp) + keys_off;
    for (size_t i = 0; i < count && st == GBS_OK; ++i) {
        const int j = (int)(i % SLOTS);
        void *d_keys = slots + j * slot_bytes;
        const size_t bytes = n[i] * kb;
        // array i - SLOTS used this buffer: its copy back must have finished
        if (i >= (size_t)SLOTS) e = cudaStreamWaitEvent(bs.in, bs.out_done[j], 0);
        if (e == cudaSuccess && bytes) e = cudaMemcpyAsync(d_keys, h_keys_in[i], bytes, cudaMemcpyHostToDevice, bs.in);
        if (e == cudaSuccess) e = cudaEventRecord(bs.in_done[j], bs.in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, bs.in_done[j], 0);
        if (e != cudaSuccess) {
            st = GBS_ERR_CUDA;
            break;
        }
        // the first sort clears the header's error word, the others keep it
        st = radix_common(d_temp, &inner, key_type, d_keys, d_keys, nullptr, nullptr, 0, n[i], begin_bit, end_bit,
                          descending, stream, i > 0);
        if (st != GBS_OK) break;
        e = cudaEventRecord(bs.sorted[j], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(bs.out, bs.sorted[j], 0);
        if (e == cudaSuccess && bytes) e = cudaMemcpyAsync(h_keys_out[i], d_keys, bytes, cudaMemcpyDeviceToHost, bs.out);
        if (e == cudaSuccess) e = cudaEventRecord(bs.out_done[j], bs.out);
        if (e != cudaSuccess) st = GBS_ERR_CUDA;
    }
    // join: `stream` passes the call's end only after both side streams' work
    e = cudaEventRecord(bs.in_end, bs.in);
    if (e == cudaSuccess) e = cudaEventRecord(bs.out_end, bs.out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, bs.in_end, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, bs.out_end, 0);
    if (st == GBS_OK && e != cudaSuccess) st = GBS_ERR_CUDA;
    return st;
}

gbs_status gbs_sort_pairs(void *d_temp, size_t *temp_bytes, gbs_key_type key_type, const void *d_keys_in,
                          void *d_keys_out, const uint32_t *d_vals_in, uint32_t *d_vals_out, size_t n,
                          int begin_bit, int end_bit, int descending, void *stream) {
    return radix_common(d_temp, temp_bytes, key_type, d_keys_in, d_keys_out, d_vals_in, d_vals_out, 4, n,
                        begin_bit, end_bit, descending, stream);
}

gbs_status gbs_sort_pairs64(void *d_temp, size_t *temp_bytes, gbs_key_type key_type, const void *d_keys_in,
                            void *d_keys_out, const uint64_t *d_vals_in, uint64_t *d_vals_out, size_t n,
                            int begin_bit, int end_bit, int descending, void *stream) {
    return radix_common(d_temp, temp_bytes, key_type, d_keys_in, d_keys_out, d_vals_in, d_vals_out, 8, n,
                        begin_bit, end_bit, descending, stream);
}

gbs_status gbs_segmented_sort(void *d_temp, size_t *temp_bytes, gbs_key_type key_type, const void *d_keys_in,
                              void *d_keys_out, size_t num_segments, size_t segment_len, int descending,
                              void *stream) {
    t_launches = 0;
    const int kb = key_bytes_of(key_type);
    if (kb == 0 || temp_bytes == nullptr) return GBS_ERR_INVALID_ARG;
    if (segment_len > GBS_MAX_RADIX_KEYS) return GBS_ERR_UNSUPPORTED;
    if (num_segments != 0 && segment_len != 0 && num_segments > (size_t)-1 / segment_len / 8)
        return GBS_ERR_INVALID_ARG;
    // segments longer than one CTA's network: the radix sort, one segment after another in a
    // shared radix work area (as gbs_segmented_sort_offsets does for its long segments)
    const bool radix = segment_len > GBS_MAX_SEGMENT_LEN;
    size_t need = sizeof(Header);
    if (radix) {
        gbs_status st = radix_common(nullptr, &need, key_type, nullptr, nullptr, nullptr, nullptr, 0, segment_len, 0,
                                     8 * kb, descending, stream);
        if (st != GBS_OK) return st;
    }
    bool query = false;
    gbs_status st = check_temp(d_temp, temp_bytes, need, &query);
    if (st != GBS_OK || query) return st;
    const size_t total = num_segments * segment_len;
    if (total > 0 && (d_keys_in == nullptr || d_keys_out == nullptr)) return GBS_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(d_temp, 0, sizeof(Header), s);
    if (e != cudaSuccess) return GBS_ERR_CUDA;
    if (total == 0) return GBS_OK;
    if (segment_len == 1) return from_cuda(copy_if_needed(d_keys_in, d_keys_out, total * kb, s));
    if (radix) {  // the launch count accumulates over the segments' sorts
        for (size_t i = 0; i < num_segments; ++i) {
            const size_t lo = i * segment_len * kb;
            size_t have = need;
            st = radix_common(d_temp, &have, key_type, static_cast<const unsigned char *>(d_keys_in) + lo,
                              static_cast<unsigned char *>(d_keys_out) + lo, nullptr, nullptr, 0, segment_len, 0,
                              8 * kb, descending, stream, /*keep_error=*/true);
            if (st != GBS_OK) return st;
        }
        return GBS_OK;
    }
    timing_start(s);
    return from_cuda(gbs::launch_segmented_bitonic((int)key_type, kb, d_keys_in, d_keys_out, num_segments,
                                                   segment_len, descending != 0, s, &t_launches));
}

gbs_status gbs_segmented_sort_offsets(void *d_temp, size_t *temp_bytes, gbs_key_type key_type, const void *d_keys_in,
                                      void *d_keys_out, size_t num_segments, const uint64_t *h_offsets,
                                      int descending, void *stream) {
    t_launches = 0;
    const int kb = key_bytes_of(key_type);
    if (kb == 0 || temp_bytes == nullptr) return GBS_ERR_INVALID_ARG;
    if (num_segments > 0xFFFFFFFFull) return GBS_ERR_UNSUPPORTED;  // 32-bit segment ids
    if (num_segments > 0 && h_offsets == nullptr) return GBS_ERR_INVALID_ARG;
    // bin the segments: class l in 1..14 holds lengths (2^(l-1), 2^l] (and 1 in class 1); longer
    // segments take the radix path one by one, sharing one radix work area
    constexpr int CLASSES = 15;
    size_t count[CLASSES] = {};
    size_t longest = 0;
    for (size_t i = 0; i < num_segments; ++i) {
        if (h_offsets[i + 1] < h_offsets[i]) return GBS_ERR_INVALID_ARG;
        const uint64_t len = h_offsets[i + 1] - h_offsets[i];
        if (len > GBS_MAX_RADIX_KEYS) return GBS_ERR_UNSUPPORTED;
        if (len == 0) continue;
        if (len > GBS_MAX_SEGMENT_LEN) {
            longest = std::max<size_t>(longest, len);
            continue;
        }
        int l = 1;
        while ((uint64_t(1) << l) < len) ++l;
        ++count[l];
    }
    // work buffer: [radix work area, or just the status header][offsets][segment ids by class]
    size_t radix_bytes = sizeof(Header);
    if (longest > 0) {
        gbs_status st = radix_common(nullptr, &radix_bytes, key_type, nullptr, nullptr, nullptr, nullptr, 0,
                                     longest, 0, 8 * kb, descending, stream);
        if (st != GBS_OK) return st;
    }
    const size_t off_offsets = round_up(radix_bytes);
    const size_t off_ids = off_offsets + round_up(sizeof(uint64_t) * (num_segments + 1));
    const size_t need = off_ids + round_up(sizeof(uint32_t) * std::max<size_t>(num_segments, 1));
    bool query = false;
    gbs_status st = check_temp(d_temp, temp_bytes, need, &query);
    if (st != GBS_OK || query) return st;
    if (num_segments > 0 && h_offsets[num_segments] > h_offsets[0] && (d_keys_in == nullptr || d_keys_out == nullptr))
        return GBS_ERR_INVALID_ARG;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *tb = reinterpret_cast<unsigned char *>(d_temp);
    if (cudaMemsetAsync(tb, 0, sizeof(Header), s) != cudaSuccess) return GBS_ERR_CUDA;
    if (num_segments == 0) return GBS_OK;
    // host staging of one copy: the offsets, then the segment ids grouped by class
    std::vector<unsigned char> staging(off_ids - off_offsets + sizeof(uint32_t) * num_segments);
    std::memcpy(staging.data(), h_offsets, sizeof(uint64_t) * (num_segments + 1));
    uint32_t *ids = reinterpret_cast<uint32_t *>(staging.data() + (off_ids - off_offsets));
    size_t start[CLASSES + 1] = {};
    for (int c = 1; c < CLASSES; ++c) start[c + 1] = start[c] + count[c];
    std::vector<uint32_t> long_ids;
    {
        size_t fill[CLASSES];
        std::copy(start, start + CLASSES, fill);
        for (size_t i = 0; i < num_segments; ++i) {
            const uint64_t len = h_offsets[i + 1] - h_offsets[i];
            if (len == 0) continue;
            if (len > GBS_MAX_SEGMENT_LEN) {
                long_ids.push_back((uint32_t)i);
                continue;
            }
            int l = 1;
            while ((uint64_t(1) << l) < len) ++l;
            ids[fill[l]++] = (uint32_t)i;
        }
    }
    uint64_t *d_offsets = reinterpret_cast<uint64_t *>(tb + off_offsets);
    uint32_t *d_ids = reinterpret_cast<uint32_t *>(tb + off_ids);
    // pageable source: the copy is staged before this call returns
    if (cudaMemcpyAsync(d_offsets, staging.data(), staging.size(), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return GBS_ERR_CUDA;
    timing_start(s);
    for (int c = 1; c < CLASSES; ++c) {
        if (count[c] == 0) continue;
        const cudaError_t e = gbs::launch_listed_bitonic((int)key_type, kb, d_keys_in, d_keys_out, d_ids + start[c],
                                                         count[c], d_offsets, c, descending != 0, s, &t_launches);
        if (e != cudaSuccess) return GBS_ERR_CUDA;
    }
    for (const uint32_t id : long_ids) {
        const size_t lo = h_offsets[id], len = h_offsets[id + 1] - lo;
        size_t have = radix_bytes;
        st = radix_common(d_temp, &have, key_type, static_cast<const unsigned char *>(d_keys_in) + lo * kb,
                          static_cast<unsigned char *>(d_keys_out) + lo * kb, nullptr, nullptr, 0, len, 0,
                          8 * kb, descending, stream, /*keep_error=*/true);
        if (st != GBS_OK) return st;
    }
    return GBS_OK;
}

gbs_status gbs_sort_keys_msd_bitonic(void *d_temp, size_t *temp_bytes, gbs_key_type key_type, const void *d_keys_in,
                                     void *d_keys_out, size_t n, int descending, void *stream) {
    const int kb = key_bytes_of(key_type);
    if (kb == 0 || temp_bytes == nullptr) return GBS_ERR_INVALID_ARG;
    if (n > GBS_MAX_RADIX_KEYS) return GBS_ERR_UNSUPPORTED;
    constexpr size_t BUCKETS = 65536;
    // work buffer: [radix sort of n keys | the segment sort's own work area] [bucket bounds]; the
    // segment sort needs at most a radix area for its longest segment (<= n keys), its offsets
    // and its segment list
    size_t radix_bytes = 0;
    gbs_status st = radix_common(nullptr, &radix_bytes, key_type, nullptr, nullptr, nullptr, nullptr, 0, n, 0, 8 * kb,
                                 descending, stream);
    if (st != GBS_OK) return st;
    const size_t seg_bytes = round_up(radix_bytes) + round_up(sizeof(uint64_t) * (BUCKETS + 1)) +
                             round_up(sizeof(uint32_t) * BUCKETS);
    const size_t off_bounds = round_up(seg_bytes);
    bool query = false;
    st = check_temp(d_temp, temp_bytes, off_bounds + round_up(sizeof(uint64_t) * (BUCKETS + 1)), &query);
    if (st != GBS_OK || query) return st;
    if (n > 0 && (d_keys_in == nullptr || d_keys_out == nullptr)) return GBS_ERR_INVALID_ARG;
    if (n <= GBS_MAX_SEGMENT_LEN)  // one segment: the regular entry point (one bitonic CTA)
        return gbs_sort_keys(d_temp, temp_bytes, key_type, d_keys_in, d_keys_out, n, 0, 8 * kb, descending, stream);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // 1. MSD: stable radix passes over the top 16 bits of the code (two 8-bit digits)
    size_t have = radix_bytes;
    st = radix_common(d_temp, &have, key_type, d_keys_in, d_keys_out, nullptr, nullptr, 0, n, 8 * kb - 16, 8 * kb,
                      descending, stream);
    if (st != GBS_OK) return st;
    int launches = t_launches;
    // 2. bucket boundaries, copied to the host for the per-bucket plan (this synchronises)
    uint64_t *d_bounds = reinterpret_cast<uint64_t *>(static_cast<unsigned char *>(d_temp) + off_bounds);
    if (gbs::launch_bucket_bounds((int)key_type, kb, d_keys_out, n, descending != 0, d_bounds, s, &launches) !=
        cudaSuccess)
        return GBS_ERR_CUDA;
    std::vector<uint64_t> bounds(BUCKETS + 1);
    if (cudaMemcpyAsync(bounds.data(), d_bounds, sizeof(uint64_t) * (BUCKETS + 1), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return GBS_ERR_CUDA;
    uint32_t err = 0;  // a timeout of the MSD passes is reported like the sort's own
    if (cudaMemcpy(&err, d_temp, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) return GBS_ERR_CUDA;
    if (err) return GBS_ERR_TIMEOUT;
    // 3. every bucket sorted in place by the bitonic network, padded to its own power of two
    //    (buckets above 2^14 keys: the radix path)
    have = seg_bytes;
    st = gbs_segmented_sort_offsets(d_temp, &have, key_type, d_keys_out, d_keys_out, BUCKETS, bounds.data(),
                                    descending, stream);
    t_launches += launches;
    return st;
}

gbs_status gbs_digit_histograms(void *d_temp, size_t *temp_bytes, gbs_key_type key_type, const void *d_keys,
                                size_t n, int begin_bit, int end_bit, int descending, uint32_t *d_hist,
                                void *stream) {
    t_launches = 0;
    const int kb = key_bytes_of(key_type);
    if (kb == 0 || temp_bytes == nullptr) return GBS_ERR_INVALID_ARG;
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > 8 * kb) return GBS_ERR_INVALID_ARG;
    if (n > GBS_MAX_RADIX_KEYS) return GBS_ERR_UNSUPPORTED;
    bool query = false;
    gbs_status st = check_temp(d_temp, temp_bytes, sizeof(Header), &query);
    if (st != GBS_OK || query) return st;
    const int passes = (end_bit - begin_bit + 7) / 8;
    if (passes == 0) return GBS_OK;
    if (d_hist == nullptr || (n > 0 && d_keys == nullptr)) return GBS_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(d_temp, 0, sizeof(Header), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_hist, 0, sizeof(uint32_t) * 256 * passes, s);
    if (e != cudaSuccess) return GBS_ERR_CUDA;
    if (n == 0) return GBS_OK;
    gbs::RadixJob job;
    std::memset(&job, 0, sizeof(job));
    job.kind = (int)key_type;
    job.key_bytes = kb;
    job.keys_in = d_keys;
    job.n = n;
    job.begin_bit = begin_bit;
    job.end_bit = end_bit;
    job.num_passes = passes;
    job.descending = descending != 0;
    job.hdr = reinterpret_cast<Header *>(d_temp);
    job.hist = d_hist;
    job.fault_pass = -1;
    timing_start(s);
    return from_cuda(gbs::launch_histograms(job, s, &t_launches));
}

gbs_status gbs_get_status(const void *d_temp, size_t temp_bytes, void *stream) {
    if (d_temp == nullptr || temp_bytes < sizeof(Header)) return GBS_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GBS_ERR_CUDA;
    uint32_t err = 0;
    if (cudaMemcpy(&err, d_temp, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) return GBS_ERR_CUDA;
    return err ? GBS_ERR_TIMEOUT : GBS_OK;
}

const char *gbs_status_string(gbs_status status) {
    switch (status) {
    case GBS_OK: return "GBS_OK";
    case GBS_ERR_INVALID_ARG: return "GBS_ERR_INVALID_ARG";
    case GBS_ERR_TEMP_TOO_SMALL: return "GBS_ERR_TEMP_TOO_SMALL";
    case GBS_ERR_UNSUPPORTED: return "GBS_ERR_UNSUPPORTED";
    case GBS_ERR_CUDA: return "GBS_ERR_CUDA";
    case GBS_ERR_TIMEOUT: return "GBS_ERR_TIMEOUT";
    default: return "GBS_ERR_UNKNOWN";
    }
}

const char *gbs_version(void) { return "0.1.0"; }

void gbs_debug_set_lookback_fault(int pass, uint32_t tile, uint32_t spin_limit) {
    g_fault_pass = pass;
    g_fault_tile = tile;
    g_spin_limit = spin_limit ? spin_limit : DEFAULT_SPIN_LIMIT;
}

int gbs_debug_last_launch_count(void) { return t_launches; }

void gbs_debug_set_timing_events(void **events, int count) {
    t_events = events;
    t_event_count = events ? count : 0;
}

void gbs_debug_set_radix_bits(int bits) { g_radix_bits = bits == 11 ? 11 : 8; }

size_t gbs_debug_radix_tile_keys(int key_bytes, int value_bytes) {
    return gbs::radix_tile_keys(key_bytes, value_bytes == 8 ? 8 : value_bytes ? 4 : 0);
}

}  // extern "C"
