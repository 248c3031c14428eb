// LSD radix sort: the exported launch functions of the upfront histogram,
// the digit passes (32-bit look-back status words; sorts of 2^29 keys or
// more take radix_wide.cu's 64-bit form) and the final copy.  The kernels are
// in radix_impl.cuh.
#include "radix_impl.cuh"

namespace gbs {

// Keys per tile of each launch shape (the pass kernel's tuning macros).
template <typename K, int VB> constexpr uint32_t shape_tile() {
    return (uint32_t)PassShape<K, VB>::THREADS * PassShape<K, VB>::ITEMS;
}

uint32_t radix_tile_keys(int key_bytes, int val_bytes) {
    if (key_bytes == 8)
        return val_bytes == 8 ? shape_tile<uint64_t, 8>() : val_bytes ? shape_tile<uint64_t, 4>() : shape_tile<uint64_t, 0>();
    return val_bytes == 8 ? shape_tile<uint32_t, 8>() : val_bytes ? shape_tile<uint32_t, 4>() : shape_tile<uint32_t, 0>();
}

cudaError_t launch_histograms(const RadixJob &job, cudaStream_t stream, int *launches) {
    if (job.key_bytes == 8) return launch_hist<uint64_t>(job, stream, false, launches);
    return launch_hist<uint32_t>(job, stream, false, launches);
}

cudaError_t launch_radix_sort(const RadixJob &job, cudaStream_t stream, int *launches) {
    cudaError_t e = job.key_bytes == 8 ? launch_hist<uint64_t>(job, stream, true, launches)
                                       : launch_hist<uint32_t>(job, stream, true, launches);
    if (e != cudaSuccess) return e;
    // sorts of 2^29 keys or more: 64-bit status words (radix_wide.cu)
    e = job.wide_status ? launch_passes_wide(job, stream, launches)
                        : launch_all_passes<uint32_t>(job, stream, launches);
    if (e != cudaSuccess) return e;
    if (job.in_place) {
        CopyParams cp;
        cp.keys_in = job.keys_in;
        cp.keys_out = job.keys_out;
        cp.keys_alt = job.keys_alt;
        cp.vals_in = job.vals_in;
        cp.vals_out = job.val_bytes ? job.vals_out : nullptr;
        cp.vals_alt = job.vals_alt;
        cp.key_bytes_total = job.n * (size_t)job.key_bytes;
        cp.val_bytes_total = job.n * (size_t)job.val_bytes;
        cp.hdr = job.hdr;
        const size_t blocks = std::min<size_t>((cp.key_bytes_total / 16 + 511) / 512 + 1, (size_t)device_sms() * 4);
        finish_copy_kernel<<<(unsigned)blocks, 512, 0, stream>>>(cp);
        ++*launches;
        timing_mark(stream);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace gbs
