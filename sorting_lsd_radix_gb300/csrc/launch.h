// Host-side interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace gbs {
// Sorts of at least this many keys use 64-bit look-back status words.
constexpr size_t WIDE_STATUS_MIN_KEYS = (size_t)StatusWord<uint32_t>::MAX_KEYS + 1;
// Bytes of look-back status words of a sort of n keys in num_tiles tiles.
constexpr size_t status_bytes(size_t n, size_t num_tiles) {
    return num_tiles * 256 * (n >= WIDE_STATUS_MIN_KEYS ? sizeof(uint64_t) : sizeof(uint32_t));
}
// Boundaries of the 65536 buckets of the top 16 code bits in keys sorted by
// them: bounds[c] = first position of bucket c or a later one (65537 words).
cudaError_t launch_bucket_bounds(int kind, int key_bytes, const void *keys, size_t n, bool descending,
                                 uint64_t *bounds, cudaStream_t stream, int *launches);

}  // namespace gbs

namespace gbs {

// One-time set-up of a kernel (its shared-memory attribute), done once per
// device: the first launch on each device runs `setup`; a set-up that fails
// is tried again on the next launch.  Devices 0..63 are remembered, others set
// up on every launch.  Two threads may both run a set-up; it is idempotent.
class PerDeviceOnce {
  public:
    template <typename F> cudaError_t run(F &&setup) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return setup();
        const uint64_t bit = uint64_t(1) << dev;
        if (done_.load(std::memory_order_acquire) & bit) return cudaSuccess;
        const cudaError_t e = setup();
        if (e == cudaSuccess) done_.fetch_or(bit, std::memory_order_acq_rel);
        return e;
    }

  private:
    std::atomic<uint64_t> done_{0};
};


// Everything one radix sort call needs on the device.
struct RadixJob {
    int kind;             // KeyKind
    int key_bytes;        // 4 or 8
    int val_bytes;        // 0 (keys only), 4 or 8
    const void *keys_in;
    void *keys_out;
    void *keys_alt;       // n keys of scratch in the work buffer
    const void *vals_in;  // values of val_bytes each
    void *vals_out;
    void *vals_alt;       // n values of scratch (pairs only)
    size_t n;
    int begin_bit, end_bit, num_passes;
    bool descending;
    bool in_place;        // keys_in == keys_out or vals_in == vals_out
    Header *hdr;
    uint32_t *hist;        // [MAX_PASSES][256]
    uint32_t *digit_base;  // [MAX_PASSES][256]
    void *status;          // [num_tiles][256] status words
    bool wide_status;      // 64-bit status words (sorts of 2^29 keys or more), else 32-bit
    uint32_t num_tiles;
    uint32_t spin_limit;   // bounded look-back wait (polls)
    int fault_pass;        // test hook: tile fault_tile of pass fault_pass never publishes (-1: off)
    uint32_t fault_tile;
};

// The test hooks' look-back fault and bounded-wait limit (see
// gbs_debug_set_lookback_fault); the defaults when the hook is off.
void debug_fault_settings(int *fault_pass, uint32_t *fault_tile, uint32_t *spin_limit);

// Kernel timing hook (see gbs_debug_set_timing_events): records the next
// caller-provided event on the stream after a launch, if the hook is set.
void timing_mark(cudaStream_t stream);

// Tile (keys per CTA) of the one-sweep pass kernel for a key width and a
// value width (0: keys only).
uint32_t radix_tile_keys(int key_bytes, int val_bytes);

// The 11-bit-digit prototype (radix11.cu): keys only, fewer than 2^29 keys;
// hist / digit_base hold [passes][2048] words and status [tiles][2048] words.
uint32_t radix11_tile_keys(int key_bytes);
cudaError_t launch_radix11_sort(const RadixJob &job, cudaStream_t stream, int *launches);

// The digit passes of a job with 64-bit look-back status words (radix_wide.cu).
cudaError_t launch_passes_wide(const RadixJob &job, cudaStream_t stream, int *launches);

// Histogram + plan, then every digit pass (and the final copy when needed).
cudaError_t launch_radix_sort(const RadixJob &job, cudaStream_t stream, int *launches);

// Only the upfront histogram kernel (hist left in job.hist).
cudaError_t launch_histograms(const RadixJob &job, cudaStream_t stream, int *launches);

// Segmented bitonic sort; segment_len in 1..16384.
cudaError_t launch_segmented_bitonic(int kind, int key_bytes, const void *keys_in, void *keys_out,
                                     size_t num_segments, size_t segment_len, bool descending,
                                     cudaStream_t stream, int *launches);
// The segments seg_ids[0 .. count) (segment id = keys [offsets[id],
// offsets[id + 1]), at most 2^len_log keys each), one bitonic network each.
cudaError_t launch_listed_bitonic(int kind, int key_bytes, const void *keys_in, void *keys_out,
                                  const uint32_t *seg_ids, size_t count, const uint64_t *offsets, int len_log,
                                  bool descending, cudaStream_t stream, int *launches);

// Boundaries of the 65536 buckets of the top 16 code bits in keys sorted by
// them: bounds[c] = first position of bucket c or a later one (65537 words).
cudaError_t launch_bucket_bounds(int kind, int key_bytes, const void *keys, size_t n, bool descending,
                                 uint64_t *bounds, cudaStream_t stream, int *launches);

}  // namespace gbs
