// LSD radix sort kernels (8-bit digits): the upfront digit histograms with
// the device-side pass plan, the one-sweep digit pass (tile load, stable
// warp-match rank, chained scan with decoupled look-back, shared-memory
// staged scatter) and the final copy.
//
// Method: kwkr.cn notes on bitonic vs LSD radix sort §3.1-3.2 (count, exclusive
// prefix, stable placement; block-local counts plus a global base instead of
// global atomics) and §3.4 (skip passes whose digit is constant);
// "GPU基数排序：从CUB工程实现到性能调优" §3 (histogram -> scan -> scatter per
// pass, a stable in-block rank instead of an atomic cursor) and §4 (8-bit
// digits, 16-byte vector loads); "并行排序：从归并网络到 GPU 双调排序" §8.1
// (warp-level histograms, block-local sort before the global write).
#include <algorithm>

#include "launch.h"

namespace gbs {
namespace {

constexpr uint32_t FULL = 0xFFFFFFFFu;

// ---------------------------------------------------------------------------
// Block-wide exclusive scan of one value per thread for threads 0..255; all
// threads of the block must call it.  wsum: 8 words of shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t excl_scan_256(uint32_t v, uint32_t *wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t x = v;
    if (tid < 256) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(FULL, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
    }
    __syncthreads();
    uint32_t base = 0;
    if (tid < 256) {
        for (int w = 0; w < warp; ++w) base += wsum[w];
    }
    __syncthreads();  // wsum may be reused right after
    return base + x - v;
}

// ---------------------------------------------------------------------------
// Upfront histogram of all digit passes (one read of the keys)
// ---------------------------------------------------------------------------

constexpr int HIST_THREADS = 512;
constexpr int HIST_UNROLL = 4;

template <typename K> struct HistCfg;
template <> struct HistCfg<uint32_t> {
    static constexpr int PASSES = 4, COPIES = 8, PER_VEC = 4;
};
template <> struct HistCfg<uint64_t> {
    static constexpr int PASSES = 8, COPIES = 4, PER_VEC = 2;
};

struct HistParams {
    const void *keys;
    uint32_t n;
    int kind, begin_bit, end_bit, num_passes;
    uint64_t flip;
    uint32_t *hist;
    uint32_t *digit_base;
    Header *hdr;
    uint4 *zero_ptr;  // look-back status words to clear
    size_t zero_vec;  // ... as 16-byte vectors
    int plan;         // compute the pass plan in the last CTA
};

template <typename K>
__global__ void __launch_bounds__(HIST_THREADS) upfront_histogram_kernel(const HistParams prm) {
    using C = HistCfg<K>;
    __shared__ uint32_t sh[C::COPIES * C::PASSES * 256];
    __shared__ uint32_t wsum[8];
    __shared__ uint32_t s_last;
    const int tid = threadIdx.x;

    for (int i = tid; i < C::COPIES * C::PASSES * 256; i += HIST_THREADS) sh[i] = 0;
    __syncthreads();

    // privatised copy: warps take turns so that one copy serves few warps
    uint32_t *my = sh + ((tid >> 5) % C::COPIES) * (C::PASSES * 256);
    const int P = prm.num_passes;
    int shift[C::PASSES];
    uint32_t mask[C::PASSES];
#pragma unroll
    for (int p = 0; p < C::PASSES; ++p) {
        shift[p] = prm.begin_bit + 8 * p;
        const int bits = min(8, prm.end_bit - shift[p]);
        mask[p] = (p < P) ? ((1u << bits) - 1u) : 0u;
        if (p >= P) shift[p] = 0;
    }
    const K flip = (K)prm.flip;
    auto count = [&](K raw) {
        const K t = KeyCodec<K>::enc(raw, prm.kind, flip);
#pragma unroll
        for (int p = 0; p < C::PASSES; ++p)
            if (p < P) atomicAdd(&my[p * 256 + digit_of(t, shift[p], mask[p])], 1u);
    };

    const size_t n = prm.n;
    const bool aligned = (reinterpret_cast<uintptr_t>(prm.keys) & 15) == 0;
    const size_t nvec = aligned ? n / C::PER_VEC : 0;
    const uint4 *vec = reinterpret_cast<const uint4 *>(prm.keys);
    const size_t stride = (size_t)gridDim.x * HIST_THREADS;
    size_t i = (size_t)blockIdx.x * HIST_THREADS + tid;
    for (; i + (HIST_UNROLL - 1) * stride < nvec; i += HIST_UNROLL * stride) {
        uint4 r[HIST_UNROLL];
#pragma unroll
        for (int u = 0; u < HIST_UNROLL; ++u) r[u] = __ldcs(vec + i + u * stride);
#pragma unroll
        for (int u = 0; u < HIST_UNROLL; ++u) {
            const K *ks = reinterpret_cast<const K *>(&r[u]);
#pragma unroll
            for (int e = 0; e < C::PER_VEC; ++e) count(ks[e]);
        }
    }
    for (; i < nvec; i += stride) {
        const uint4 r = __ldcs(vec + i);
        const K *ks = reinterpret_cast<const K *>(&r);
#pragma unroll
        for (int e = 0; e < C::PER_VEC; ++e) count(ks[e]);
    }
    // scalar remainder (and the whole array when it is not 16-byte aligned)
    const K *scal = reinterpret_cast<const K *>(prm.keys);
    for (size_t j = nvec * C::PER_VEC + (size_t)blockIdx.x * HIST_THREADS + tid; j < n; j += stride)
        count(scal[j]);

    // clear this CTA's share of the look-back status words
    for (size_t z = (size_t)blockIdx.x * HIST_THREADS + tid; z < prm.zero_vec; z += stride)
        prm.zero_ptr[z] = make_uint4(0, 0, 0, 0);

    __syncthreads();
    for (int b = tid; b < P * 256; b += HIST_THREADS) {
        uint32_t s = 0;
#pragma unroll
        for (int c = 0; c < C::COPIES; ++c) s += sh[c * C::PASSES * 256 + b];
        if (s) atomicAdd(&prm.hist[b], s);
    }
    if (!prm.plan) return;

    // The last CTA to finish turns the histograms into the pass plan.
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&prm.hdr->hist_blocks_done, 1u) == gridDim.x - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    uint32_t active = 0;
    for (int p = 0; p < P; ++p) {
        const uint32_t c = (tid < 256) ? __ldcg(&prm.hist[p * 256 + tid]) : 0u;
        const uint32_t ex = excl_scan_256(c, wsum);
        if (tid < 256) prm.digit_base[p * 256 + tid] = ex;
        // a pass whose digit is the same for every key leaves the order unchanged
        const int trivial = __syncthreads_or(tid < 256 && c == prm.n);
        if (!trivial) active |= 1u << p;
    }
    if (tid == 0) {
        uint32_t k = 0;
        for (int p = 0; p < P; ++p) {
            prm.hdr->ordinal[p] = k;
            if ((active >> p) & 1u) ++k;
        }
        prm.hdr->active_mask = active;
        prm.hdr->num_active = k;
    }
}

// ---------------------------------------------------------------------------
// One digit pass
// ---------------------------------------------------------------------------

template <typename K, bool PAIRS, int THREADS, int ITEMS> struct PassSmem {
    static constexpr int TILE = THREADS * ITEMS;
    static constexpr int WARPS = THREADS / 32;
    K keys[TILE];
    uint32_t vals[PAIRS ? TILE : 4];
    uint32_t whist[WARPS][256];  // per-warp digit counts, then warp-exclusive offsets
    uint32_t local[256];         // exclusive prefix of the tile's digit counts
    uint32_t binoff[256];        // global position of sorted-tile slot 0 of each digit
    uint32_t wsum[8];
    uint32_t tile;
    alignas(8) uint64_t bar;
};

struct PassParams {
    const void *keys_in;
    void *keys_out;
    void *keys_alt;
    const uint32_t *vals_in;
    uint32_t *vals_out;
    uint32_t *vals_alt;
    uint32_t n;
    int kind;
    uint64_t flip;
    int pass, num_passes, shift;
    uint32_t mask;
    int in_place;
    Header *hdr;
    const uint32_t *digit_base;
    uint32_t *status;
    uint32_t spin_limit;
    int fault_pass;
    uint32_t fault_tile;
};

template <typename K>
__device__ __forceinline__ void copy_range(const K *src, K *dst, size_t lo, size_t hi, int tid, int nthreads) {
    for (size_t i = lo + tid; i < hi; i += nthreads) dst[i] = src[i];
}

template <typename K, bool PAIRS, int THREADS, int ITEMS>
__global__ void __launch_bounds__(THREADS, 2) onesweep_pass_kernel(const PassParams prm) {
    using S = PassSmem<K, PAIRS, THREADS, ITEMS>;
    constexpr int TILE = S::TILE;
    constexpr int WARPS = S::WARPS;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    S &sm = *reinterpret_cast<S *>(smem_raw);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    Header *hdr = prm.hdr;
    const uint32_t A = hdr->num_active;
    const bool active = (hdr->active_mask >> prm.pass) & 1u;
    if (!active) {
        // Every pass is trivial: the input order is already sorted; the last
        // pass kernel copies it to the output (the in-place case needs none
        // for the keys and is finished by the copy kernel).
        if (A == 0 && prm.pass == prm.num_passes - 1 && !prm.in_place) {
            const size_t lo = (size_t)blockIdx.x * TILE, hi = min((size_t)prm.n, lo + TILE);
            copy_range(reinterpret_cast<const K *>(prm.keys_in), reinterpret_cast<K *>(prm.keys_out), lo, hi, tid,
                       THREADS);
            if (PAIRS) copy_range(prm.vals_in, prm.vals_out, lo, hi, tid, THREADS);
        }
        return;
    }
    const uint32_t k = hdr->ordinal[prm.pass];
    const bool first = (k == 0), last = (k + 1 == A);

    // buffers: the last active pass lands in the output (or in the scratch
    // buffer when an in-place call has an odd number of active passes, which
    // keeps every pass out of place; the copy kernel then finishes)
    const bool odd_in_place = prm.in_place && (A & 1u);
    K *kout = reinterpret_cast<K *>(prm.keys_out), *kalt = reinterpret_cast<K *>(prm.keys_alt);
    K *k_last = odd_in_place ? kalt : kout, *k_other = odd_in_place ? kout : kalt;
    const K *ksrc = first ? reinterpret_cast<const K *>(prm.keys_in) : ((((A - k) & 1u) == 0) ? k_last : k_other);
    K *kdst = (((A - 1 - k) & 1u) == 0) ? k_last : k_other;
    uint32_t *v_last = odd_in_place ? prm.vals_alt : prm.vals_out;
    uint32_t *v_other = odd_in_place ? prm.vals_out : prm.vals_alt;
    const uint32_t *vsrc = nullptr;
    uint32_t *vdst = nullptr;
    if (PAIRS) {
        vsrc = first ? prm.vals_in : ((((A - k) & 1u) == 0) ? v_last : v_other);
        vdst = (((A - 1 - k) & 1u) == 0) ? v_last : v_other;
    }

    // chained-scan states of this pass (rotated by ordinal, see common.cuh)
    const uint32_t st_agg = 1u + 2u * (k % 3u), st_inc = 2u + 2u * (k % 3u);

    if (tid == 0) {
        sm.tile = atomicAdd(&hdr->tile_counter[prm.pass], 1u);
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    for (int i = tid; i < WARPS * 256; i += THREADS) (&sm.whist[0][0])[i] = 0;
    __syncthreads();
    const uint32_t tile = sm.tile;
    const size_t tile_start = (size_t)tile * TILE;
    const uint32_t valid = (uint32_t)min((size_t)TILE, (size_t)prm.n - tile_start);

    // ---- tile load: one bulk async copy per array, or plain loads --------
    const K *gk = ksrc + tile_start;
    const bool bulk = (valid == TILE) && ((reinterpret_cast<uintptr_t>(gk) & 15) == 0) &&
                      (!PAIRS || ((reinterpret_cast<uintptr_t>(vsrc + tile_start) & 15) == 0));
    if (bulk) {
        if (tid == 0) {
            mbar_arrive_expect_tx(&sm.bar,
                                  TILE * (uint32_t)sizeof(K) + (PAIRS ? TILE * 4u : 0u));
            bulk_g2s(sm.keys, gk, TILE * (uint32_t)sizeof(K), &sm.bar);
            if (PAIRS) bulk_g2s(sm.vals, vsrc + tile_start, TILE * 4u, &sm.bar);
        }
        uint32_t polls = 0;
        while (!mbar_try_wait(&sm.bar, 0)) {
            if (++polls > prm.spin_limit) {
                record_error(hdr, ERR_COPY_TIMEOUT, ((uint32_t)prm.pass << 24) | (tile & 0xFFFFFFu));
                break;
            }
            if (polls > 16) __nanosleep(64);
        }
    } else {
        for (uint32_t i = tid; i < valid; i += THREADS) {
            sm.keys[i] = gk[i];
            if (PAIRS) sm.vals[i] = vsrc[tile_start + i];
        }
        __syncthreads();
    }

    // ---- stable rank within the tile --------------------------------------
    // Warp w owns tile slots [w*ITEMS*32, (w+1)*ITEMS*32); item i of lane l is
    // slot w*ITEMS*32 + 32 i + l, so (warp, item, lane) is input order.  Lanes
    // holding the same digit find each other with match.any; the lowest of
    // them advances the warp's counter for that digit by the group size.
    const K flip = (K)prm.flip;
    K keys[ITEMS];
    uint32_t ranks[ITEMS];
    uint32_t *whist = sm.whist[warp];
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
        const bool ok = idx < valid;
        K key = ok ? sm.keys[idx] : (K)0;
        if (first) key = KeyCodec<K>::enc(key, prm.kind, flip);
        keys[i] = key;
        const uint32_t d = digit_of(key, prm.shift, prm.mask);
        const uint32_t vmask = __ballot_sync(FULL, ok);
        ranks[i] = 0;
        if (ok) {
            const uint32_t peers = __match_any_sync(vmask, d);
            const uint32_t before = whist[d];
            __syncwarp(vmask);
            if (lane == __ffs(peers) - 1) whist[d] = before + __popc(peers);
            __syncwarp(vmask);
            ranks[i] = before + __popc(peers & lt);
        }
    }
    __syncthreads();

    // ---- tile digit counts, warp offsets, publish the aggregate ------------
    uint32_t cnt = 0;
    uint32_t *my_status = prm.status + (size_t)tile * 256;
    const bool faulty = (prm.fault_pass == prm.pass) && (prm.fault_tile == tile);
    if (tid < 256) {
        uint32_t run = 0;
#pragma unroll 4
        for (int w = 0; w < WARPS; ++w) {
            const uint32_t c = sm.whist[w][tid];
            sm.whist[w][tid] = run;
            run += c;
        }
        cnt = run;
        if (!faulty) st_relaxed_gpu(my_status + tid, ((tile == 0 ? st_inc : st_agg) << STATUS_COUNT_BITS) | run);
    }
    const uint32_t local = excl_scan_256(cnt, sm.wsum);

    // ---- decoupled look-back over the predecessors' status words ----------
    if (tid < 256) {
        uint32_t excl = 0;
        if (tile > 0) {
            uint32_t j = tile - 1;
            uint32_t polls = 0;
            for (;;) {
                const uint32_t s = ld_relaxed_gpu(prm.status + (size_t)j * 256 + tid);
                const uint32_t st = s >> STATUS_COUNT_BITS;
                if (st == st_agg || st == st_inc) {
                    excl += s & STATUS_COUNT_MASK;
                    if (st == st_inc || j == 0) break;
                    --j;
                    continue;
                }
                if (++polls > prm.spin_limit) {
                    record_error(hdr, ERR_LOOKBACK_TIMEOUT, ((uint32_t)prm.pass << 24) | (tile & 0xFFFFFFu));
                    break;
                }
                __nanosleep(polls < 64 ? 32 : 256);
            }
            if (!faulty)
                st_relaxed_gpu(my_status + tid, (st_inc << STATUS_COUNT_BITS) | ((excl + cnt) & STATUS_COUNT_MASK));
        }
        sm.local[tid] = local;
        sm.binoff[tid] = prm.digit_base[prm.pass * 256 + tid] + excl - local;
    }
    __syncthreads();

    // ---- reorder the tile in shared memory by (digit, rank) ---------------
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
        if (idx < valid) {
            const uint32_t d = digit_of(keys[i], prm.shift, prm.mask);
            ranks[i] += sm.local[d] + whist[d];  // slot in the sorted tile
            sm.keys[ranks[i]] = keys[i];
        }
    }
    if (PAIRS) {
        uint32_t vals[ITEMS];
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
            const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
            vals[i] = (idx < valid) ? sm.vals[idx] : 0u;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
            const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
            if (idx < valid) sm.vals[ranks[i]] = vals[i];
        }
    }
    __syncthreads();

    // ---- coalesced scatter: consecutive slots of one digit go to consecutive
    //      global positions ---------------------------------------------------
    for (uint32_t j = tid; j < valid; j += THREADS) {
        const K key = sm.keys[j];
        const uint32_t d = digit_of(key, prm.shift, prm.mask);
        const uint32_t pos = sm.binoff[d] + j;
        kdst[pos] = last ? KeyCodec<K>::dec(key, prm.kind, flip) : key;
        if (PAIRS) vdst[pos] = sm.vals[j];
    }
}

// ---------------------------------------------------------------------------
// Final copy for in-place calls
// ---------------------------------------------------------------------------

struct CopyParams {
    const void *keys_in;
    void *keys_out;
    const void *keys_alt;
    const uint32_t *vals_in;
    uint32_t *vals_out;
    const uint32_t *vals_alt;
    size_t key_bytes_total;
    size_t val_bytes_total;
    const Header *hdr;
};

__device__ void copy_bytes(const void *src, void *dst, size_t bytes) {
    if (src == dst || bytes == 0) return;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0) {
        const size_t nv = bytes / 16;
        const uint4 *s = reinterpret_cast<const uint4 *>(src);
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        for (size_t i = t0; i < nv; i += stride) d[i] = s[i];
        for (size_t i = nv * 16 + t0; i < bytes; i += stride)
            reinterpret_cast<unsigned char *>(dst)[i] = reinterpret_cast<const unsigned char *>(src)[i];
    } else {
        for (size_t i = t0; i < bytes; i += stride)
            reinterpret_cast<unsigned char *>(dst)[i] = reinterpret_cast<const unsigned char *>(src)[i];
    }
}

__global__ void __launch_bounds__(512) finish_copy_kernel(const CopyParams prm) {
    const uint32_t A = prm.hdr->num_active;
    if (A == 0) {
        copy_bytes(prm.keys_in, prm.keys_out, prm.key_bytes_total);
        if (prm.vals_out) copy_bytes(prm.vals_in, prm.vals_out, prm.val_bytes_total);
    } else if (A & 1u) {
        copy_bytes(prm.keys_alt, prm.keys_out, prm.key_bytes_total);
        if (prm.vals_out) copy_bytes(prm.vals_alt, prm.vals_out, prm.val_bytes_total);
    }
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------

int device_sms() {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    return sms;
}

template <typename K>
cudaError_t launch_hist(const RadixJob &job, cudaStream_t stream, bool plan, int *launches) {
    HistParams prm;
    prm.keys = job.keys_in;
    prm.n = (uint32_t)job.n;
    prm.kind = job.kind;
    prm.begin_bit = job.begin_bit;
    prm.end_bit = job.end_bit;
    prm.num_passes = job.num_passes;
    prm.flip = job.descending ? ~0ull : 0ull;
    prm.hist = job.hist;
    prm.digit_base = job.digit_base;
    prm.hdr = job.hdr;
    prm.zero_ptr = reinterpret_cast<uint4 *>(job.status);
    prm.zero_vec = plan ? (size_t)job.num_tiles * 256 * 4 / 16 : 0;
    prm.plan = plan ? 1 : 0;
    const size_t per_cta = (size_t)HIST_THREADS * HIST_UNROLL * HistCfg<K>::PER_VEC;
    size_t grid = std::max<size_t>((job.n + per_cta - 1) / per_cta, (prm.zero_vec + HIST_THREADS - 1) / HIST_THREADS);
    grid = std::min<size_t>(grid, (size_t)device_sms() * 2);
    grid = std::max<size_t>(grid, 1);
    upfront_histogram_kernel<K><<<(unsigned)grid, HIST_THREADS, 0, stream>>>(prm);
    ++*launches;
    timing_mark(stream);
    return cudaGetLastError();
}

template <typename K, bool PAIRS, int THREADS, int ITEMS>
cudaError_t launch_passes(const RadixJob &job, cudaStream_t stream, int *launches) {
    using S = PassSmem<K, PAIRS, THREADS, ITEMS>;
    auto kern = onesweep_pass_kernel<K, PAIRS, THREADS, ITEMS>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(S));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    PassParams prm;
    prm.keys_in = job.keys_in;
    prm.keys_out = job.keys_out;
    prm.keys_alt = job.keys_alt;
    prm.vals_in = job.vals_in;
    prm.vals_out = job.vals_out;
    prm.vals_alt = job.vals_alt;
    prm.n = (uint32_t)job.n;
    prm.kind = job.kind;
    prm.flip = job.descending ? ~0ull : 0ull;
    prm.num_passes = job.num_passes;
    prm.in_place = job.in_place ? 1 : 0;
    prm.hdr = job.hdr;
    prm.status = job.status;
    prm.spin_limit = job.spin_limit;
    prm.fault_pass = job.fault_pass;
    prm.fault_tile = job.fault_tile;
    for (int p = 0; p < job.num_passes; ++p) {
        prm.pass = p;
        prm.shift = job.begin_bit + 8 * p;
        const int bits = std::min(8, job.end_bit - prm.shift);
        prm.mask = (1u << bits) - 1u;
        prm.digit_base = job.digit_base;
        kern<<<job.num_tiles, THREADS, sizeof(S), stream>>>(prm);
        ++*launches;
        timing_mark(stream);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

// Tile shapes: 512 threads per CTA, two CTAs per SM; 16 keys per thread for
// 32-bit keys and 8 for 64-bit keys, so a tile is 32 KiB of keys.
uint32_t radix_tile_keys(int key_bytes, bool /*pairs*/) { return key_bytes == 8 ? 512u * 8u : 512u * 16u; }

cudaError_t launch_histograms(const RadixJob &job, cudaStream_t stream, int *launches) {
    if (job.key_bytes == 8) return launch_hist<uint64_t>(job, stream, false, launches);
    return launch_hist<uint32_t>(job, stream, false, launches);
}

cudaError_t launch_radix_sort(const RadixJob &job, cudaStream_t stream, int *launches) {
    cudaError_t e;
    if (job.key_bytes == 8) {
        e = launch_hist<uint64_t>(job, stream, true, launches);
        if (e != cudaSuccess) return e;
        e = job.pairs ? launch_passes<uint64_t, true, 512, 8>(job, stream, launches)
                      : launch_passes<uint64_t, false, 512, 8>(job, stream, launches);
    } else {
        e = launch_hist<uint32_t>(job, stream, true, launches);
        if (e != cudaSuccess) return e;
        e = job.pairs ? launch_passes<uint32_t, true, 512, 16>(job, stream, launches)
                      : launch_passes<uint32_t, false, 512, 16>(job, stream, launches);
    }
    if (e != cudaSuccess) return e;
    if (job.in_place) {
        CopyParams cp;
        cp.keys_in = job.keys_in;
        cp.keys_out = job.keys_out;
        cp.keys_alt = job.keys_alt;
        cp.vals_in = job.vals_in;
        cp.vals_out = job.pairs ? job.vals_out : nullptr;
        cp.vals_alt = job.vals_alt;
        cp.key_bytes_total = job.n * (size_t)job.key_bytes;
        cp.val_bytes_total = job.pairs ? job.n * 4 : 0;
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
