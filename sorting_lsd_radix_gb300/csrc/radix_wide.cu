// The digit passes of radix sorts of 2^29 keys or more, whose look-back
// status words are 64-bit (their counts pass the 29-bit field of the 32-bit
// words).  A translation unit of its own so that it compiles in parallel with
// radix.cu.
#include "radix_impl.cuh"

namespace gbs {

cudaError_t launch_passes_wide(const RadixJob &job, cudaStream_t stream, int *launches) {
    return launch_all_passes<uint64_t>(job, stream, launches);
}

}  // namespace gbs
