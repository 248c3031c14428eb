// Host-side interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace gbs {

// Everything one radix sort call needs on the device.
struct RadixJob {
    int kind;             // KeyKind
    int key_bytes;        // 4 or 8
    bool pairs;
    const void *keys_in;
    void *keys_out;
    void *keys_alt;       // n keys of scratch in the work buffer
    const uint32_t *vals_in;
    uint32_t *vals_out;
    uint32_t *vals_alt;   // n values of scratch (pairs only)
    size_t n;
    int begin_bit, end_bit, num_passes;
    bool descending;
    bool in_place;        // keys_in == keys_out or vals_in == vals_out
    Header *hdr;
    uint32_t *hist;        // [MAX_PASSES][256]
    uint32_t *digit_base;  // [MAX_PASSES][256]
    uint32_t *status;      // [num_tiles][256]
    uint32_t num_tiles;
    uint32_t spin_limit;   // bounded look-back wait (polls)
    int fault_pass;        // test hook: tile fault_tile of pass fault_pass never publishes (-1: off)
    uint32_t fault_tile;
};

// Kernel timing hook (see gbs_debug_set_timing_events): records the next
// caller-provided event on the stream after a launch, if the hook is set.
void timing_mark(cudaStream_t stream);

// Tile (keys per CTA) of the one-sweep pass kernel for a key width / pairs.
uint32_t radix_tile_keys(int key_bytes, bool pairs);

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

}  // namespace gbs
