// gbs_sort_keys_noalloc: the radix sort of gbs_sort_keys for callers that
// cannot allocate device memory.  Its work buffer is a fixed array in the
// library's own device memory instead of a caller-provided one.
//
// Who needs this: code that must not call cudaMalloc at all — for example a
// plug-in running inside a host application that owns every allocation, a
// real-time loop where an allocation's unbounded latency (and its implicit
// device synchronisation) is not acceptable, or an environment whose memory
// pool is fixed up front.  Such callers still own their keys; only the
// scratch space (header, histograms, look-back status words and the
// alternate key buffer) comes from here.
#include "../../include/gbsort.h"
#include "launch.h"

namespace {

// Scratch for up to GBS_NOALLOC_MAX_KEYS keys of at most 8 bytes:
//   [0, 256)            header (error word, pass plan, tile tickets)
//   [256, 8448)         digit histograms, 8 x 256 x u32
//   [8448, 16640)       digit bases, 8 x 256 x u32
//   [16640, +status)    look-back status words, 1 KiB per tile
//   [.., +8 MiB)        alternate key buffer
constexpr size_t kAlign = 256;
constexpr size_t kHeader = 256;
constexpr size_t kHist = 8 * 256 * 4;
constexpr size_t kMinTileKeys = 4096;  // smallest radix tile of any key width
constexpr size_t kMaxTiles = (GBS_NOALLOC_MAX_KEYS + kMinTileKeys - 1) / kMinTileKeys;
constexpr size_t kStatus = kMaxTiles * 256 * 4;
constexpr size_t kKeys = (size_t)GBS_NOALLOC_MAX_KEYS * 8;
constexpr size_t kScratchBytes = kHeader + 2 * kHist + kStatus + kKeys;

static_assert(kStatus == gbs::status_bytes(GBS_NOALLOC_MAX_KEYS, kMaxTiles),
              "scratch must hold the look-back status of its largest sort");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, never a device address, so
// every call asks the runtime for the address on the device that is current
// now.  The first call on a device also loads the library's device code there
// (the array is created with it); later calls are a table lookup.  Asking
// each time, instead of caching the pointer, keeps the address right after a
// cudaDeviceReset, which destroys the array and makes a new one at the next
// call.
gbs_status scratch_for_current_device(unsigned char **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return GBS_ERR_CUDA;
    *out = reinterpret_cast<unsigned char *>(p);
    return GBS_OK;
}

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

}  // namespace

extern "C" gbs_status gbs_sort_keys_noalloc(gbs_key_type key_type, const void *d_keys_in, void *d_keys_out,
                                            size_t n, int begin_bit, int end_bit, int descending, void *stream) {
    const int kb = (key_type == GBS_U64 || key_type == GBS_I64 || key_type == GBS_F64)   ? 8
                   : (key_type == GBS_U32 || key_type == GBS_I32 || key_type == GBS_F32) ? 4
                                                                                          : 0;
    if (kb == 0) return GBS_ERR_INVALID_ARG;
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > 8 * kb) return GBS_ERR_INVALID_ARG;
    if (n > GBS_NOALLOC_MAX_KEYS) return GBS_ERR_UNSUPPORTED;
    if (n > 0 && (d_keys_in == nullptr || d_keys_out == nullptr)) return GBS_ERR_INVALID_ARG;

    unsigned char *scratch = nullptr;
    gbs_status st = scratch_for_current_device(&scratch);
    if (st != GBS_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    const uint32_t tile = gbs::radix_tile_keys(kb, 0);
    const uint32_t tiles = (uint32_t)((n + tile - 1) / tile);
    const size_t off_hist = kHeader, off_base = off_hist + kHist, off_status = off_base + kHist;
    const size_t off_keys = off_status + up(gbs::status_bytes(n, tiles));
    if (off_keys + (size_t)kb * n > kScratchBytes) return GBS_ERR_UNSUPPORTED;

    // the header and histograms must start at zero on every call (the
    // look-back status words are cleared by the histogram kernel)
    if (cudaMemsetAsync(scratch, 0, off_base, s) != cudaSuccess) return GBS_ERR_CUDA;
    const int passes = (end_bit - begin_bit + 7) / 8;
    if (n <= 1 || passes == 0) {
        if (n == 0 || d_keys_in == d_keys_out) return GBS_OK;
        return cudaMemcpyAsync(d_keys_out, d_keys_in, n * kb, cudaMemcpyDeviceToDevice, s) == cudaSuccess
                   ? GBS_OK
                   : GBS_ERR_CUDA;
    }

    gbs::RadixJob job;
    job.kind = (int)key_type;
    job.key_bytes = kb;
    job.val_bytes = 0;
    job.keys_in = d_keys_in;
    job.keys_out = d_keys_out;
    job.keys_alt = scratch + off_keys;
    job.vals_in = nullptr;
    job.vals_out = nullptr;
    job.vals_alt = nullptr;
    job.n = n;
    job.begin_bit = begin_bit;
    job.end_bit = end_bit;
    job.num_passes = passes;
    job.descending = descending != 0;
    job.in_place = (d_keys_in == d_keys_out);
    job.hdr = reinterpret_cast<gbs::Header *>(scratch);
    job.hist = reinterpret_cast<uint32_t *>(scratch + off_hist);
    job.digit_base = reinterpret_cast<uint32_t *>(scratch + off_base);
    job.status = scratch + off_status;
    job.wide_status = false;  // n <= GBS_NOALLOC_MAX_KEYS, far below the 64-bit status threshold
    job.num_tiles = tiles;
    gbs::debug_fault_settings(&job.fault_pass, &job.fault_tile, &job.spin_limit);
    int launches = 0;
    return gbs::launch_radix_sort(job, s, &launches) == cudaSuccess ? GBS_OK : GBS_ERR_CUDA;
}

extern "C" gbs_status gbs_get_status_noalloc(void *stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return GBS_ERR_CUDA;
    unsigned char *scratch = nullptr;
    const gbs_status st = scratch_for_current_device(&scratch);
    if (st != GBS_OK) return st;
    uint32_t err = 0;  // first word of the header: the first device-side error of the last call
    if (cudaMemcpy(&err, scratch, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) return GBS_ERR_CUDA;
    return err ? GBS_ERR_TIMEOUT : GBS_OK;
}
