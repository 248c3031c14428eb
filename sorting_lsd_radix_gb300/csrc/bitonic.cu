// Bitonic tile sorter: one CTA (or one warp, or one thread) sorts a segment of
// up to 2^14 keys on chip.
//
// Network ("并行排序：从归并网络到 GPU 双调排序" §3.3-3.5, §4.2-4.3; kwkr.cn
// notes on bitonic vs LSD radix sort §2.2-2.3): for merge size k = 2^m,
// m = 1..log2(L), and stride j = k/2 .. 1, element i is compared with i ^ j;
// the pair is put in ascending order when bit m of i is 0 (the segment bit,
// taken from the index within the whole segment), descending otherwise.
// Segments whose length is not a power of two are padded with the all-ones
// code, which sorts after every key ("并行排序" §3.5; kwkr.cn notes §5.1).
// Descending output sorts the complemented codes ascending.
//
// Mapping: each thread holds KP = 2^K_LOG keys in registers.  In the layout
// with register-bit offset g0, register r of thread t holds the element whose
// index bits [g0, g0 + K_LOG) are r and whose other bits are t's bits; every
// stride 2^b with b in that range is then a compare-exchange between two
// registers of one thread.  A stage walks its strides from the top bit down,
// switching layout through shared memory (one store and one load per key)
// whenever it crosses into the next group of K_LOG bits; the blocked layout
// (g0 = 0) covers the K_LOG lowest bits.  Shared-memory rows are padded by one
// element per 2^max(K_LOG, 4) so that both layouts are free of bank conflicts.
#include <algorithm>

#include "launch.h"

namespace gbs {
namespace {

template <typename K, int L_LOG, int K_LOG> struct Shape {
    static constexpr int L = 1 << L_LOG;
    static constexpr int KP = 1 << K_LOG;
    static constexpr int S = L / KP;               // threads per segment
    static constexpr int T = S >= 128 ? S : 128;   // threads per CTA
    static constexpr int SEGS = T / S;             // segments per CTA
    static constexpr int PAD = K_LOG > 4 ? K_LOG : 4;  // one pad element per 2^PAD
    static constexpr int LP = L + ((L >> PAD) > 0 ? (L >> PAD) : 1);  // padded row length (elements)
    static constexpr bool WARP_LOCAL = S <= 32;
    static constexpr size_t SMEM = (size_t)SEGS * LP * sizeof(K);
};

template <bool WARP_LOCAL> __device__ __forceinline__ void tile_sync() {
    if (WARP_LOCAL)
        __syncwarp();
    else
        __syncthreads();
}

// Index within the segment of register r of thread t in layout g0.
template <int K_LOG> __device__ __forceinline__ int layout_index(int t, int r, int g0) {
    return (t & ((1 << g0) - 1)) | (r << g0) | ((t >> g0) << (g0 + K_LOG));
}

template <int PAD> __device__ __forceinline__ int padded(int i) { return i + (i >> PAD); }

template <typename K, int K_LOG, int PAD, bool WARP_LOCAL, int FROM, int TO>
__device__ __forceinline__ void relayout(K (&x)[1 << K_LOG], K *row, int t) {
    tile_sync<WARP_LOCAL>();
#pragma unroll
    for (int r = 0; r < (1 << K_LOG); ++r) row[padded<PAD>(layout_index<K_LOG>(t, r, FROM))] = x[r];
    tile_sync<WARP_LOCAL>();
#pragma unroll
    for (int r = 0; r < (1 << K_LOG); ++r) x[r] = row[padded<PAD>(layout_index<K_LOG>(t, r, TO))];
}

// Direction by complement.  Within merge stage M every compare-exchange pairs
// two elements whose index bit M is equal, so no key leaves the set of
// positions with bit M set during the stage.  Complementing the keys held at
// those positions for the duration of the stage turns their descending
// compare-exchanges into ascending ones: min/max of complemented keys is the
// complement of max/min.  Every exchange is then a plain ascending min/max,
// and the direction costs one XOR per key per stage instead of two selects
// per compare-exchange.
//
// Bit M of the segment index of register r of thread t in the blocked layout
// (register bits [0, K_LOG), thread bits above); 0 for M < 1, where no stage
// has run.
template <int K_LOG, int M> __device__ __forceinline__ uint32_t blocked_bit(int t, int r) {
    if constexpr (M < 1)
        return 0u;
    else if constexpr (M < K_LOG)
        return ((uint32_t)r >> M) & 1u;
    else
        return ((uint32_t)t >> (M - K_LOG)) & 1u;
}

// Between stage M - 1 and stage M (blocked layout): undo the complement of
// stage M - 1 and apply that of stage M.
template <typename K, int K_LOG, int M> __device__ __forceinline__ void switch_direction(K (&x)[1 << K_LOG], int t) {
#pragma unroll
    for (int r = 0; r < (1 << K_LOG); ++r) {
        const uint32_t b = blocked_bit<K_LOG, M - 1>(t, r) ^ blocked_bit<K_LOG, M>(t, r);
        x[r] ^= (K)0 - (K)b;
    }
}

__device__ __forceinline__ uint32_t key_min(uint32_t a, uint32_t b) { return umin(a, b); }
__device__ __forceinline__ uint32_t key_max(uint32_t a, uint32_t b) { return umax(a, b); }
__device__ __forceinline__ uint64_t key_min(uint64_t a, uint64_t b) { return a < b ? a : b; }
__device__ __forceinline__ uint64_t key_max(uint64_t a, uint64_t b) { return a < b ? b : a; }

// Ascending compare-exchange across register bit RB.
template <typename K, int K_LOG, int RB> __device__ __forceinline__ void exchange_regbit(K (&x)[1 << K_LOG]) {
#pragma unroll
    for (int r = 0; r < (1 << K_LOG); ++r) {
        if (r & (1 << RB)) continue;
        const int r2 = r | (1 << RB);
        const K a = x[r], b = x[r2];
        x[r] = key_min(a, b);
        x[r2] = key_max(a, b);
    }
}

template <typename K, int K_LOG, int G0, int B> __device__ __forceinline__ void strides_down(K (&x)[1 << K_LOG]) {
    exchange_regbit<K, K_LOG, B - G0>(x);
    if constexpr (B > G0) strides_down<K, K_LOG, G0, B - 1>(x);
}

// Register-bit offset of group q: q*K_LOG, kept inside the segment's index bits.
template <int K_LOG, int L_LOG> __host__ __device__ constexpr int group_g0(int q) {
    return q * K_LOG < L_LOG - K_LOG ? q * K_LOG : L_LOG - K_LOG;
}

// Stage M, register-bit group Q (top group QT first, down to group 0).  The
// top group holds bit M-1; each lower group takes the bits below the one
// above it.
template <typename K, int K_LOG, int PAD, bool WARP_LOCAL, int L_LOG, int M, int Q, int QT>
__device__ __forceinline__ void stage_groups(K (&x)[1 << K_LOG], K *row, int t) {
    constexpr int G0 = group_g0<K_LOG, L_LOG>(Q);
    constexpr int PREV = (Q == QT) ? 0 : group_g0<K_LOG, L_LOG>(Q + 1);
    constexpr int HI = (Q == QT) ? M - 1 : PREV - 1;
    static_assert(G0 >= 0 && G0 + K_LOG <= L_LOG && HI >= G0 && HI < G0 + K_LOG, "bad register-bit group");
    if constexpr (G0 != PREV) relayout<K, K_LOG, PAD, WARP_LOCAL, PREV, G0>(x, row, t);
    strides_down<K, K_LOG, G0, HI>(x);
    if constexpr (Q > 0) stage_groups<K, K_LOG, PAD, WARP_LOCAL, L_LOG, M, Q - 1, QT>(x, row, t);
}

// Stages M .. L_LOG; each starts and ends in the blocked layout.  The last
// stage complements nothing (bit L_LOG of every segment index is 0), so no
// key is left complemented.
template <typename K, int K_LOG, int PAD, bool WARP_LOCAL, int L_LOG, int M>
__device__ __forceinline__ void all_stages(K (&x)[1 << K_LOG], K *row, int t) {
    if constexpr (M <= L_LOG) {
        constexpr int QT = (M - 1) / K_LOG;
        switch_direction<K, K_LOG, M>(x, t);
        stage_groups<K, K_LOG, PAD, WARP_LOCAL, L_LOG, M, QT, QT>(x, row, t);
        all_stages<K, K_LOG, PAD, WARP_LOCAL, L_LOG, M + 1>(x, row, t);
    }
}

struct BitonicParams {
    const void *keys_in;
    void *keys_out;
    size_t num_segments;  // segments this launch sorts
    uint32_t seg_len;     // uniform mode: every segment's length
    int kind;
    uint64_t flip;
    // list mode (seg_ids != nullptr): the launch sorts segments seg_ids[0 ..
    // num_segments), segment id holding keys [offsets[id], offsets[id + 1])
    const uint32_t *seg_ids;
    const uint64_t *offsets;
};

// Resident threads per SM the kernel is compiled for (registers per thread =
// 65536 / this); 0 leaves the register count to the compiler.  More resident
// CTAs let one segment's global load and store overlap another's network.
#ifndef GBS_BITONIC_THREADS_PER_SM_32
#define GBS_BITONIC_THREADS_PER_SM_32 1024
#endif
#ifndef GBS_BITONIC_THREADS_PER_SM_64
#define GBS_BITONIC_THREADS_PER_SM_64 0
#endif
template <typename K, int T> constexpr int bitonic_min_blocks() {
    constexpr int per_sm = sizeof(K) == 8 ? GBS_BITONIC_THREADS_PER_SM_64 : GBS_BITONIC_THREADS_PER_SM_32;
    return per_sm / T > 1 ? per_sm / T : 1;
}

template <typename K, int L_LOG, int K_LOG>
__global__ void __launch_bounds__(Shape<K, L_LOG, K_LOG>::T, (bitonic_min_blocks<K, Shape<K, L_LOG, K_LOG>::T>()))
    bitonic_tile_kernel(const BitonicParams prm) {
    using Sh = Shape<K, L_LOG, K_LOG>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    K *sm = reinterpret_cast<K *>(smem_raw);
    const int tid = threadIdx.x;
    const int t = tid % Sh::S;
    K *row = sm + (tid / Sh::S) * Sh::LP;
    const size_t seg0 = (size_t)blockIdx.x * Sh::SEGS;
    const K *in = reinterpret_cast<const K *>(prm.keys_in);
    K *out = reinterpret_cast<K *>(prm.keys_out);
    const K flip = (K)prm.flip;
    const uint32_t len = prm.seg_len;

    // list mode: each of the CTA's segments has its own place and length
    __shared__ size_t s_base[Sh::SEGS];
    __shared__ uint32_t s_len[Sh::SEGS];
    const bool listed = prm.seg_ids != nullptr;
    if (listed) {
        for (int j = tid; j < Sh::SEGS; j += Sh::T) {
            size_t b = 0;
            uint32_t l = 0;
            if (seg0 + j < prm.num_segments) {
                const uint32_t id = prm.seg_ids[seg0 + j];
                b = (size_t)prm.offsets[id];
                l = (uint32_t)(prm.offsets[id + 1] - prm.offsets[id]);
            }
            s_base[j] = b;
            s_len[j] = l;
        }
        __syncthreads();
    }

    // coalesced load of this CTA's segments, encoded, padded with all-ones.
    // Whole segments of the padded length on 16-byte boundaries (the usual
    // case) move as 16-byte vectors; a vector never straddles a segment or a
    // shared-memory pad (both are multiples of the vector's keys).
    constexpr int VEC = 16 / (int)sizeof(K);
    const bool vec = !listed && Sh::L % VEC == 0 && len == (uint32_t)Sh::L && seg0 + Sh::SEGS <= prm.num_segments &&
                     ((reinterpret_cast<uintptr_t>(in + seg0 * len) | reinterpret_cast<uintptr_t>(out + seg0 * len)) &
                      15) == 0;
    if (listed && Sh::L >= VEC) {
        // VEC keys per step: one 16-byte load where the segment starts on a
        // 16-byte boundary and the step lies inside it, else key by key
        for (int e = tid; e < Sh::SEGS * Sh::L / VEC; e += Sh::T) {
            const int k0 = e * VEC, s = k0 >> L_LOG, i = k0 & (Sh::L - 1);
            const uint32_t len_s = s_len[s];
            const K *src = in + s_base[s] + i;
            K *dst = sm + s * Sh::LP + padded<Sh::PAD>(i);
            if ((uint32_t)i + VEC <= len_s && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
                const uint4 w = __ldcs(reinterpret_cast<const uint4 *>(src));
                const K *ks = reinterpret_cast<const K *>(&w);
#pragma unroll
                for (int u = 0; u < VEC; ++u) dst[u] = KeyCodec<K>::enc(ks[u], prm.kind, flip);
            } else {
#pragma unroll
                for (int u = 0; u < VEC; ++u)
                    dst[u] = ((uint32_t)i + u < len_s) ? KeyCodec<K>::enc(src[u], prm.kind, flip) : KeyCodec<K>::ALL_ONES;
            }
        }
    } else if (listed) {
        for (int e = tid; e < Sh::SEGS * Sh::L; e += Sh::T) {
            const int s = e >> L_LOG, i = e & (Sh::L - 1);
            K v = KeyCodec<K>::ALL_ONES;
            if ((uint32_t)i < s_len[s]) v = KeyCodec<K>::enc(in[s_base[s] + i], prm.kind, flip);
            sm[s * Sh::LP + padded<Sh::PAD>(i)] = v;
        }
    } else if (vec) {
        const uint4 *src = reinterpret_cast<const uint4 *>(in + seg0 * len);
        for (int e = tid; e < Sh::SEGS * Sh::L / VEC; e += Sh::T) {
            const uint4 w = __ldcs(src + e);
            const K *ks = reinterpret_cast<const K *>(&w);
            const int k0 = e * VEC, s = k0 >> L_LOG, i = k0 & (Sh::L - 1);
            K *dst = sm + s * Sh::LP + padded<Sh::PAD>(i);
#pragma unroll
            for (int u = 0; u < VEC; ++u) dst[u] = KeyCodec<K>::enc(ks[u], prm.kind, flip);
        }
    } else {
        for (int e = tid; e < Sh::SEGS * Sh::L; e += Sh::T) {
            const int s = e >> L_LOG, i = e & (Sh::L - 1);
            const size_t seg = seg0 + s;
            K v = KeyCodec<K>::ALL_ONES;
            if (seg < prm.num_segments && (uint32_t)i < len) v = KeyCodec<K>::enc(in[seg * len + i], prm.kind, flip);
            sm[s * Sh::LP + padded<Sh::PAD>(i)] = v;
        }
    }
    __syncthreads();
    K x[Sh::KP];
#pragma unroll
    for (int r = 0; r < Sh::KP; ++r) x[r] = row[padded<Sh::PAD>(layout_index<K_LOG>(t, r, 0))];

    all_stages<K, K_LOG, Sh::PAD, Sh::WARP_LOCAL, L_LOG, 1>(x, row, t);

    __syncthreads();
#pragma unroll
    for (int r = 0; r < Sh::KP; ++r) row[padded<Sh::PAD>(layout_index<K_LOG>(t, r, 0))] = x[r];
    __syncthreads();
    if (listed && Sh::L >= VEC) {
        for (int e = tid; e < Sh::SEGS * Sh::L / VEC; e += Sh::T) {
            const int k0 = e * VEC, s = k0 >> L_LOG, i = k0 & (Sh::L - 1);
            const uint32_t len_s = s_len[s];
            if ((uint32_t)i >= len_s) continue;
            K *dstg = out + s_base[s] + i;
            const K *src = sm + s * Sh::LP + padded<Sh::PAD>(i);
            if ((uint32_t)i + VEC <= len_s && (reinterpret_cast<uintptr_t>(dstg) & 15) == 0) {
                uint4 w;
                K *ks = reinterpret_cast<K *>(&w);
#pragma unroll
                for (int u = 0; u < VEC; ++u) ks[u] = KeyCodec<K>::dec(src[u], prm.kind, flip);
                __stcs(reinterpret_cast<uint4 *>(dstg), w);
            } else {
#pragma unroll
                for (int u = 0; u < VEC; ++u)
                    if ((uint32_t)i + u < len_s) dstg[u] = KeyCodec<K>::dec(src[u], prm.kind, flip);
            }
        }
    } else if (listed) {
        for (int e = tid; e < Sh::SEGS * Sh::L; e += Sh::T) {
            const int s = e >> L_LOG, i = e & (Sh::L - 1);
            if ((uint32_t)i < s_len[s])
                out[s_base[s] + i] = KeyCodec<K>::dec(sm[s * Sh::LP + padded<Sh::PAD>(i)], prm.kind, flip);
        }
    } else if (vec) {
        uint4 *dstv = reinterpret_cast<uint4 *>(out + seg0 * len);
        for (int e = tid; e < Sh::SEGS * Sh::L / VEC; e += Sh::T) {
            const int k0 = e * VEC, s = k0 >> L_LOG, i = k0 & (Sh::L - 1);
            const K *src = sm + s * Sh::LP + padded<Sh::PAD>(i);
            uint4 w;
            K *ks = reinterpret_cast<K *>(&w);
#pragma unroll
            for (int u = 0; u < VEC; ++u) ks[u] = KeyCodec<K>::dec(src[u], prm.kind, flip);
            __stcs(dstv + e, w);
        }
    } else {
        for (int e = tid; e < Sh::SEGS * Sh::L; e += Sh::T) {
            const int s = e >> L_LOG, i = e & (Sh::L - 1);
            const size_t seg = seg0 + s;
            if (seg < prm.num_segments && (uint32_t)i < len)
                out[seg * len + i] = KeyCodec<K>::dec(sm[s * Sh::LP + padded<Sh::PAD>(i)], prm.kind, flip);
        }
    }
}

template <typename K, int L_LOG, int K_LOG>
cudaError_t launch_shape(const BitonicParams &prm, cudaStream_t stream) {
    using Sh = Shape<K, L_LOG, K_LOG>;
    auto kern = bitonic_tile_kernel<K, L_LOG, K_LOG>;
    static PerDeviceOnce once;
    const cudaError_t e =
        once.run([&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Sh::SMEM); });
    if (e != cudaSuccess) return e;
    const size_t grid = (prm.num_segments + Sh::SEGS - 1) / Sh::SEGS;
    kern<<<(unsigned)grid, Sh::T, Sh::SMEM, stream>>>(prm);
    return cudaGetLastError();
}

template <typename K, int L_LOG>
cudaError_t launch_len(const BitonicParams &prm, cudaStream_t stream) {
    // Keys per thread, chosen by measurement on GB300.  4-byte keys: 32, but 16
    // for 2^11 and 2^12 keys (32 there needs more than the 64 registers that
    // keep several CTAs resident).  8-byte keys: 16, but 32 at 2^14 keys,
    // where 16 would need 1024 threads with at most 64 registers.
    constexpr int KMAX = sizeof(K) == 8 ? (L_LOG < 14 ? 4 : 5) : (L_LOG == 11 || L_LOG == 12) ? 4 : 5;
    constexpr int K_LOG = L_LOG < KMAX ? L_LOG : KMAX;
    return launch_shape<K, L_LOG, K_LOG>(prm, stream);
}

template <typename K>
cudaError_t launch_by_log(int l, const BitonicParams &prm, cudaStream_t stream) {
    switch (l) {
    case 1: return launch_len<K, 1>(prm, stream);
    case 2: return launch_len<K, 2>(prm, stream);
    case 3: return launch_len<K, 3>(prm, stream);
    case 4: return launch_len<K, 4>(prm, stream);
    case 5: return launch_len<K, 5>(prm, stream);
    case 6: return launch_len<K, 6>(prm, stream);
    case 7: return launch_len<K, 7>(prm, stream);
    case 8: return launch_len<K, 8>(prm, stream);
    case 9: return launch_len<K, 9>(prm, stream);
    case 10: return launch_len<K, 10>(prm, stream);
    case 11: return launch_len<K, 11>(prm, stream);
    case 12: return launch_len<K, 12>(prm, stream);
    case 13: return launch_len<K, 13>(prm, stream);
    case 14: return launch_len<K, 14>(prm, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_listed_bitonic(int kind, int key_bytes, const void *keys_in, void *keys_out,
                                  const uint32_t *seg_ids, size_t count, const uint64_t *offsets, int len_log,
                                  bool descending, cudaStream_t stream, int *launches) {
    BitonicParams prm;
    prm.keys_in = keys_in;
    prm.keys_out = keys_out;
    prm.num_segments = count;
    prm.seg_len = 0;
    prm.kind = kind;
    prm.flip = descending ? ~0ull : 0ull;
    prm.seg_ids = seg_ids;
    prm.offsets = offsets;
    ++*launches;
    const cudaError_t e = key_bytes == 8 ? launch_by_log<uint64_t>(len_log, prm, stream)
                                         : launch_by_log<uint32_t>(len_log, prm, stream);
    timing_mark(stream);
    return e;
}

cudaError_t launch_segmented_bitonic(int kind, int key_bytes, const void *keys_in, void *keys_out,
                                     size_t num_segments, size_t segment_len, bool descending,
                                     cudaStream_t stream, int *launches) {
    BitonicParams prm;
    prm.keys_in = keys_in;
    prm.keys_out = keys_out;
    prm.num_segments = num_segments;
    prm.seg_len = (uint32_t)segment_len;
    prm.kind = kind;
    prm.flip = descending ? ~0ull : 0ull;
    prm.seg_ids = nullptr;
    prm.offsets = nullptr;
    int l = 0;
    while ((size_t(1) << l) < segment_len) ++l;
    ++*launches;
    const cudaError_t e = key_bytes == 8 ? launch_by_log<uint64_t>(l, prm, stream)
                                         : launch_by_log<uint32_t>(l, prm, stream);
    timing_mark(stream);
    return e;
}

}  // namespace gbs

// ---------------------------------------------------------------------------
// Bucket boundaries of keys sorted by the top 16 bits of their code (the
// MSD-then-bitonic prototype): bounds[c] = first position whose bucket is at
// least c, for c = 0 .. 65536 (bounds[65536] = n).  Position i writes the
// boundaries of every bucket in (bucket(i-1), bucket(i)], so each of the
// 65537 entries is written exactly once.
// ---------------------------------------------------------------------------
namespace gbs {
namespace {

template <typename K>
__global__ void bucket_bounds_kernel(const K *keys, size_t n, int kind, K flip, int shift, uint64_t *bounds) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i <= n; i += stride) {
        const int64_t b = (i < n) ? (int64_t)(KeyCodec<K>::enc(keys[i], kind, flip) >> shift) : 65536;
        const int64_t prev = (i > 0) ? (int64_t)(KeyCodec<K>::enc(keys[i - 1], kind, flip) >> shift) : -1;
        for (int64_t c = prev + 1; c <= b; ++c) bounds[c] = i;
    }
}

}  // namespace

cudaError_t launch_bucket_bounds(int kind, int key_bytes, const void *keys, size_t n, bool descending,
                                 uint64_t *bounds, cudaStream_t stream, int *launches) {
    const size_t blocks = std::min<size_t>((n + 1 + 255) / 256, 4096);
    if (key_bytes == 8)
        bucket_bounds_kernel<uint64_t><<<(unsigned)blocks, 256, 0, stream>>>(
            reinterpret_cast<const uint64_t *>(keys), n, kind, descending ? ~0ull : 0ull, 48, bounds);
    else
        bucket_bounds_kernel<uint32_t><<<(unsigned)blocks, 256, 0, stream>>>(
            reinterpret_cast<const uint32_t *>(keys), n, kind, descending ? 0xFFFFFFFFu : 0u, 16, bounds);
    ++*launches;
    timing_mark(stream);
    return cudaGetLastError();
}

}  // namespace gbs
