// LSD radix sort with 11-bit digits (2048 digit values per pass): a measured
// prototype of the pass-count reduction the pages discuss (kwkr.cn notes on
// bitonic vs LSD radix sort §3.4 and §5.2: fewer passes, fewer bytes;
// "GPU基数排序：从CUB工程实现到性能调优" §4: digit width against the number of
// passes).  32-bit keys take 3 passes (11 + 11 + 10 bits) instead of 4,
// 64-bit keys 6 instead of 8.  Keys only, fewer than 2^29 keys (32-bit status
// words).  Selected with gbs_debug_set_radix_bits(11); the 8-bit kernels stay
// the library's path.
//
// Same structure as the 8-bit one-sweep pass (radix_impl.cuh): ticket, bulk
// tile copy, stable ballot rank, tile counts, chained scan with decoupled
// look-back, shared-memory reorder, coalesced scatter.  What changes with
// 2048 digit values:
//  - the rank takes 11 ballots; the peer mask is the AND of three table
//    entries (digit bits 0-4, 5-9 and 10), fetched with three shuffles;
//  - per-warp digit counters are 16-bit, two to a 32-bit word (8 KiB per
//    warp); the leader's atomic adds to its half of the word;
//  - each of the 256 threads owns 8 consecutive digit values in the count,
//    scan and look-back phases; the look-back reads its 8 status words of a
//    predecessor row with two 16-byte loads.
#include <cstring>

#include "radix_impl.cuh"

namespace gbs {
namespace {

constexpr int R11_BITS = 11;
constexpr int R11_DIGITS = 1 << R11_BITS;
constexpr int R11_THREADS = 256;
constexpr int R11_PER_THREAD = R11_DIGITS / R11_THREADS;  // digit values per thread (8)
constexpr int R11_MAX_PASSES = 6;                         // 64-bit keys
constexpr int R11_CTAS_PER_SM = 3;

// Digit of a code for an 11-bit pass: (t >> shift) & mask.
__device__ __forceinline__ uint32_t r11_digit(uint32_t t, int shift, uint32_t mask) { return (t >> shift) & mask; }
__device__ __forceinline__ uint32_t r11_digit(uint64_t t, int shift, uint32_t mask) {
    return (uint32_t)(t >> shift) & mask;
}

// ---------------------------------------------------------------------------
// Upfront histograms of every 11-bit digit position, and the pass plan
// ---------------------------------------------------------------------------

constexpr int R11_HIST_THREADS = 1024;

struct R11HistParams {
    const void *keys;
    uint32_t n;
    int begin_bit, end_bit, num_passes;
    uint32_t enc_a, enc_b;
    uint64_t enc_a64, enc_b64;
    uint32_t *hist;        // [passes][2048]
    uint32_t *digit_base;  // [passes][2048]
    Header *hdr;
    uint4 *zero_ptr;  // look-back status words to clear
    size_t zero_vec;
};

__device__ __forceinline__ uint32_t r11_code(uint32_t x, const R11HistParams &p) {
    return x ^ (((uint32_t)((int32_t)x >> 31) & p.enc_a) ^ p.enc_b);
}
__device__ __forceinline__ uint64_t r11_code(uint64_t x, const R11HistParams &p) {
    return x ^ (((uint64_t)((int64_t)x >> 63) & p.enc_a64) ^ p.enc_b64);
}

template <typename K>
__global__ void __launch_bounds__(R11_HIST_THREADS, 1) r11_histogram_kernel(const R11HistParams prm) {
    extern __shared__ __align__(16) uint32_t sh[];  // [passes][2048]
    __shared__ uint32_t wsum[32];
    __shared__ uint32_t s_last;
    const int tid = threadIdx.x;
    const int P = prm.num_passes;
    for (int i = tid; i < P * R11_DIGITS; i += R11_HIST_THREADS) sh[i] = 0;
    __syncthreads();
    int shift[R11_MAX_PASSES];
    uint32_t mask[R11_MAX_PASSES];
#pragma unroll
    for (int p = 0; p < R11_MAX_PASSES; ++p) {
        shift[p] = prm.begin_bit + R11_BITS * p;
        mask[p] = (p < P) ? ((1u << min(R11_BITS, prm.end_bit - shift[p])) - 1u) : 0u;
        if (p >= P) shift[p] = 0;
    }
    const K *keys = reinterpret_cast<const K *>(prm.keys);
    const size_t stride = (size_t)gridDim.x * R11_HIST_THREADS;
    for (size_t i = (size_t)blockIdx.x * R11_HIST_THREADS + tid; i < prm.n; i += stride) {
        const K t = r11_code(keys[i], prm);
#pragma unroll
        for (int p = 0; p < R11_MAX_PASSES; ++p)
            if (p < P) atomicAdd(&sh[p * R11_DIGITS + r11_digit(t, shift[p], mask[p])], 1u);
    }
    for (size_t z = (size_t)blockIdx.x * R11_HIST_THREADS + tid; z < prm.zero_vec; z += stride)
        prm.zero_ptr[z] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    for (int b = tid; b < P * R11_DIGITS; b += R11_HIST_THREADS)
        if (sh[b]) atomicAdd(&prm.hist[b], sh[b]);

    // the last CTA to finish turns the histograms into the pass plan
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&prm.hdr->hist_blocks_done, 1u) == gridDim.x - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    uint32_t active = 0;
    const int lane = tid & 31, warp = tid >> 5;
    for (int p = 0; p < P; ++p) {
        // thread tid owns digits 2 tid and 2 tid + 1
        const uint32_t c0 = __ldcg(&prm.hist[p * R11_DIGITS + 2 * tid]);
        const uint32_t c1 = __ldcg(&prm.hist[p * R11_DIGITS + 2 * tid + 1]);
        uint32_t x = c0 + c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(FULL, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        uint32_t base = 0;
        for (int w = 0; w < warp; ++w) base += wsum[w];
        const uint32_t ex = base + x - (c0 + c1);
        prm.digit_base[p * R11_DIGITS + 2 * tid] = ex;
        prm.digit_base[p * R11_DIGITS + 2 * tid + 1] = ex + c0;
        const int trivial = __syncthreads_or(c0 == prm.n || c1 == prm.n);
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
// One 11-bit digit pass
// ---------------------------------------------------------------------------

template <typename K, int ITEMS> struct R11Smem {
    static constexpr int TILE = R11_THREADS * ITEMS;
    static constexpr int WARPS = R11_THREADS / 32;
    K keys[TILE];
    // per-warp digit counters, 16 bits each, two to a word; after the count
    // phase: sorted-tile slot of the warp's first key of each digit
    uint32_t whist[WARPS][R11_DIGITS / 2];
    uint32_t binoff[R11_DIGITS];
    uint32_t wsum[8];
    uint32_t tile;
    alignas(8) uint64_t bar;
};

// Stable warp rank with 11-bit digits (see rank_warp for the 8-bit form).
template <bool ENC, bool FULLTILE, typename K, int ITEMS>
__device__ __forceinline__ void r11_rank_warp(const K *tile_keys, uint32_t *whist, const PassParams &prm, int warp,
                                              int lane, uint32_t valid, K (&keys)[ITEMS],
                                              PackedRanks<ITEMS> &ranks) {
    const PeerTableLane nl(lane);
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
        keys[i] = load_key<ENC>(tile_keys, idx, FULLTILE || idx < valid, prm);
    }
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const uint32_t d = r11_digit(keys[i], prm.shift, prm.mask);
        uint32_t b[R11_BITS];
#pragma unroll
        for (int k = 0; k < R11_BITS; ++k) b[k] = ballot_bits(d, 1u << k);
        // lane l: lanes whose digit bits 0-4 equal l; bits 5-9 equal l; bit 10 equals l & 1
        const uint32_t lo = nl.agree(b[0], 0) & nl.agree(b[1], 1) & nl.agree(b[2], 2) & nl.agree(b[3], 3) &
                            nl.agree(b[4], 4);
        const uint32_t mid = nl.agree(b[5], 0) & nl.agree(b[6], 1) & nl.agree(b[7], 2) & nl.agree(b[8], 3) &
                             nl.agree(b[9], 4);
        const uint32_t hi = nl.agree(b[10], 0);
        uint32_t peers = __shfl_sync(FULL, lo, (int)d) & __shfl_sync(FULL, mid, (int)(d >> 5)) &
                         __shfl_sync(FULL, hi, (int)(d >> 10));
        bool ok = true;
        if (!FULLTILE) {
            const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
            ok = idx < valid;
            const uint32_t vmask = ballot_bits(ok ? 1u : 0u, 1u);
            peers &= ok ? vmask : 0u;
        }
        uint32_t leader;
        asm("bfind.u32 %0, %1;" : "=r"(leader) : "r"(peers));
        const uint32_t below = __popc(peers & lt);
        const uint32_t half = (d & 1u) << 4;  // this digit's half of the counter word
        uint32_t before = 0;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.eq.u32 p, %1, %2;\n\t@p atom.shared.add.u32 %0, [%3], %4;\n\t}"
            : "+r"(before)
            : "r"((uint32_t)lane), "r"(leader), "r"(smem_u32(&whist[d >> 1])), "r"((below + 1u) << half));
        const uint32_t bw = __shfl_sync(FULL, before, (int)leader);
        ranks.set(i, ok ? ((bw >> half) & 0xFFFFu) + below : 0u);
    }
}

// Look-back for the 8 digit values [d0, d0 + 8) of one thread: reads a window
// of R11_WINDOW predecessor rows per round trip (its 8 status words of each row
// with two 16-byte loads), nearest first, adding each digit's aggregates up to
// its first inclusive prefix; a row whose word for a digit still unresolved has
// not been published stops the walk until it is (bounded wait).  One row per
// round trip measured fastest (u32, 1e8 keys: 2.58 ms per sort against 4.02
// and 4.07 for windows of 4 and 8 rows): a status row is 8 KiB here, and rows
// read ahead but not needed crowd the keys out of L2.
#ifndef GBS_R11_WINDOW
#define GBS_R11_WINDOW 1
#endif
constexpr int R11_WINDOW = GBS_R11_WINDOW;
__device__ __forceinline__ void r11_lookback(const PassParams &prm, Header *hdr, uint32_t tile, int d0,
                                             uint32_t st_agg, uint32_t (&excl)[R11_PER_THREAD]) {
    constexpr int CB = StatusWord<uint32_t>::COUNT_BITS;
    constexpr uint32_t CM = StatusWord<uint32_t>::COUNT_MASK;
    const uint32_t *status = reinterpret_cast<const uint32_t *>(prm.status);
    uint32_t open = (1u << R11_PER_THREAD) - 1u;  // digits still walking back
    int32_t next = (int32_t)tile - 1;             // nearest row not yet added
    uint32_t polls = 0;
    while (open && next >= 0) {
        uint4 v[R11_WINDOW][2];
#pragma unroll
        for (int r = 0; r < R11_WINDOW; ++r) {
            if (next - r >= 0) {
                const uint4 *row = reinterpret_cast<const uint4 *>(status + (size_t)(next - r) * R11_DIGITS + d0);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v[r][h].x), "=r"(v[r][h].y), "=r"(v[r][h].z), "=r"(v[r][h].w)
                                 : "l"(row + h)
                                 : "memory");
            }
        }
        int used = 0;
#pragma unroll
        for (int r = 0; r < R11_WINDOW; ++r) {
            if (used < r || !open) break;  // an earlier row stopped the walk, or every digit is done
            if (next - r < 0) {            // before tile 0: every digit's prefix is complete
                open = 0;
                break;
            }
            const uint32_t w[R11_PER_THREAD] = {v[r][0].x, v[r][0].y, v[r][0].z, v[r][0].w,
                                                v[r][1].x, v[r][1].y, v[r][1].z, v[r][1].w};
            bool blocked = false;
#pragma unroll
            for (int j = 0; j < R11_PER_THREAD; ++j)
                if ((open >> j) & 1u) blocked |= ((w[j] >> CB) - st_agg) > 1u;
            if (blocked) break;
#pragma unroll
            for (int j = 0; j < R11_PER_THREAD; ++j) {
                if ((open >> j) & 1u) {
                    excl[j] += w[j] & CM;
                    if (((w[j] >> CB) - st_agg) == 1u) open &= ~(1u << j);  // inclusive prefix: done
                }
            }
            used = r + 1;
        }
        next -= used;
        if (used == 0 && open) {
            if (++polls > prm.spin_limit) {
                record_error(hdr, ERR_LOOKBACK_TIMEOUT, ((uint32_t)prm.pass << 24) | (tile & 0xFFFFFFu));
                break;
            }
            __nanosleep(polls < 64 ? 32 : 256);
        }
    }
}

template <bool FULLTILE, typename K, int ITEMS>
__device__ __forceinline__ void r11_pass_tile(R11Smem<K, ITEMS> &sm, const PassParams &prm, Header *hdr,
                                              uint32_t tile, uint32_t valid, uint32_t A, uint32_t k, bool first) {
    constexpr int WARPS = R11_THREADS / 32;
    constexpr int CB = StatusWord<uint32_t>::COUNT_BITS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    K keys[ITEMS];
    PackedRanks<ITEMS> ranks;
    if (first)
        r11_rank_warp<true, FULLTILE>(sm.keys, sm.whist[warp], prm, warp, lane, valid, keys, ranks);
    else
        r11_rank_warp<false, FULLTILE>(sm.keys, sm.whist[warp], prm, warp, lane, valid, keys, ranks);
    __syncthreads();

    const bool last = (k + 1 == A) && !prm.identity;
    const uint32_t st_agg = 1u + 2u * (k % 3u), st_inc = 2u + 2u * (k % 3u);
    const PassIO<K, 0> io(prm, A, k);
    K *kdst = io.kdst;
    const bool faulty = (prm.fault_pass == prm.pass) && (prm.fault_tile == tile);
    uint32_t *my_status = reinterpret_cast<uint32_t *>(prm.status) + (size_t)tile * R11_DIGITS;

    // ---- counts of this thread's 8 digits, warp offsets (exclusive over warps)
    const int d0 = tid * R11_PER_THREAD;
    uint32_t cnt[R11_PER_THREAD];
#pragma unroll
    for (int j = 0; j < R11_PER_THREAD; ++j) cnt[j] = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        uint4 *p = reinterpret_cast<uint4 *>(&sm.whist[w][d0 / 2]);  // 4 words: digits d0 .. d0 + 7
        uint4 v = *p;
        uint32_t *vw = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t c_lo = vw[j] & 0xFFFFu, c_hi = vw[j] >> 16;
            vw[j] = cnt[2 * j] | (cnt[2 * j + 1] << 16);
            cnt[2 * j] += c_lo;
            cnt[2 * j + 1] += c_hi;
        }
        *p = v;
    }
    uint32_t total = 0;
#pragma unroll
    for (int j = 0; j < R11_PER_THREAD; ++j) {
        if (!faulty) st_relaxed_gpu(my_status + d0 + j, ((tile == 0 ? st_inc : st_agg) << CB) | cnt[j]);
        total += cnt[j];
    }
    // tile-local exclusive prefix of each digit
    const uint32_t base = excl_scan_256<false>(total, sm.wsum);
    uint32_t local[R11_PER_THREAD];
    {
        uint32_t run = base;
#pragma unroll
        for (int j = 0; j < R11_PER_THREAD; ++j) {
            local[j] = run;
            run += cnt[j];
        }
    }
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        uint4 *p = reinterpret_cast<uint4 *>(&sm.whist[w][d0 / 2]);
        uint4 v = *p;
        uint32_t *vw = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) vw[j] += local[2 * j] | (local[2 * j + 1] << 16);  // slots < 2^16
        *p = v;
    }
    __syncthreads();

    // ---- reorder the tile in shared memory by (digit, rank) ---------------
    const uint16_t *woff = reinterpret_cast<const uint16_t *>(sm.whist[warp]);
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
        if (FULLTILE || idx < valid) {
            const uint32_t slot = ranks.get(i) + woff[r11_digit(keys[i], prm.shift, prm.mask)];
            sm.keys[slot] = keys[i];
        }
    }

    // ---- look-back for this thread's 8 digits; publish the inclusive prefix
    uint32_t excl[R11_PER_THREAD];
#pragma unroll
    for (int j = 0; j < R11_PER_THREAD; ++j) excl[j] = 0;
    if (tile > 0) {
        r11_lookback(prm, hdr, tile, d0, st_agg, excl);
        if (!faulty) {
#pragma unroll
            for (int j = 0; j < R11_PER_THREAD; ++j)
                st_relaxed_gpu(my_status + d0 + j,
                               (st_inc << CB) | ((excl[j] + cnt[j]) & StatusWord<uint32_t>::COUNT_MASK));
        }
    }
    bool out_of_range = false;
#pragma unroll
    for (int j = 0; j < R11_PER_THREAD; ++j) {
        const uint32_t db = prm.digit_base[prm.pass * R11_DIGITS + d0 + j];
        sm.binoff[d0 + j] = db + excl[j] - local[j];
        out_of_range |= cnt[j] != 0 && (uint64_t)db + excl[j] + cnt[j] > (uint64_t)prm.n;
    }
    if (__syncthreads_or(out_of_range)) {
        if (tid == 0) record_error(hdr, ERR_COPY_TIMEOUT, ((uint32_t)prm.pass << 24) | (tile & 0xFFFFFFu));
        return;
    }

    // ---- coalesced scatter ------------------------------------------------
    for (uint32_t j = tid; j < valid; j += R11_THREADS) {
        const K key = sm.keys[j];
        const uint32_t pos = sm.binoff[r11_digit(key, prm.shift, prm.mask)] + j;
        kdst[pos] = last ? Xform<K>::dec(key, prm) : key;
    }
}

template <typename K, int ITEMS>
__global__ void __launch_bounds__(R11_THREADS, R11_CTAS_PER_SM) r11_pass_kernel(const PassParams prm) {
    using S = R11Smem<K, ITEMS>;
    constexpr int TILE = S::TILE;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    S &sm = *reinterpret_cast<S *>(smem_raw);
    const int tid = threadIdx.x;
    Header *hdr = prm.hdr;
    const uint32_t A = hdr->num_active;
    if (!((hdr->active_mask >> prm.pass) & 1u)) {
        // every pass trivial: the last pass kernel copies the keys to the output
        if (A == 0 && prm.pass == prm.num_passes - 1 && !prm.in_place && (size_t)blockIdx.x * TILE < prm.n) {
            const size_t lo = (size_t)blockIdx.x * TILE, hi = min((size_t)prm.n, lo + TILE);
            copy_range(reinterpret_cast<const K *>(prm.keys_in), reinterpret_cast<K *>(prm.keys_out), lo, hi, tid,
                       R11_THREADS);
        }
        return;
    }
    const uint32_t k = hdr->ordinal[prm.pass];
    const bool first = (k == 0) && !prm.identity;
    const PassIO<K, 0> io(prm, A, k);
    const K *ksrc = io.ksrc;
    const bool aligned = (reinterpret_cast<uintptr_t>(ksrc) & 15) == 0;
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
        const uint32_t t = atomicAdd(&hdr->tile_counter[prm.pass], 1u);
        sm.tile = t;
        const size_t start = (size_t)t * TILE;
        if (aligned && start + TILE <= (size_t)prm.n) {
            mbar_arrive_expect_tx(&sm.bar, TILE * (uint32_t)sizeof(K));
            bulk_g2s(sm.keys, ksrc + start, TILE * (uint32_t)sizeof(K), &sm.bar);
        }
        const size_t pf = (size_t)t + prm.prefetch_ahead;
        if (prm.prefetch_ahead != 0 && aligned && (pf + 1) * TILE <= (size_t)prm.n)
            prefetch_l2_bulk(ksrc + pf * TILE, TILE * (uint32_t)sizeof(K));
    }
    for (int i = tid; i < S::WARPS * R11_DIGITS / 2; i += R11_THREADS) (&sm.whist[0][0])[i] = 0;
    __syncthreads();
    const uint32_t tile = sm.tile;
    const size_t tile_start = (size_t)tile * TILE;
    const uint32_t valid = tile_start < prm.n ? (uint32_t)min((size_t)TILE, (size_t)prm.n - tile_start) : 0u;
    if (valid == TILE && aligned) {
        wait_phase(&sm.bar, 0, prm, hdr, tile);
    } else {
        for (uint32_t i = tid; i < valid; i += R11_THREADS) sm.keys[i] = ksrc[tile_start + i];
        __syncthreads();
    }
    if (valid == TILE)
        r11_pass_tile<true, K, ITEMS>(sm, prm, hdr, tile, valid, A, k, first);
    else
        r11_pass_tile<false, K, ITEMS>(sm, prm, hdr, tile, valid, A, k, first);
}

// Keys per thread: 32 for 32-bit keys (8192-key tiles), 16 for 64-bit keys
// (4096-key tiles), both about 74 KiB of shared memory per CTA with the
// counters and bases, three CTAs per SM.
template <typename K> struct R11Shape;
template <> struct R11Shape<uint32_t> {
    static constexpr int ITEMS = 32;
};
template <> struct R11Shape<uint64_t> {
    static constexpr int ITEMS = 16;
};

template <typename K> cudaError_t r11_sort(const RadixJob &job, cudaStream_t stream, int *launches) {
    constexpr int ITEMS = R11Shape<K>::ITEMS;
    using S = R11Smem<K, ITEMS>;
    static PerDeviceOnce once;
    cudaError_t e = once.run([] {
        cudaError_t r = cudaFuncSetAttribute(r11_pass_kernel<K, ITEMS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(S));
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(r11_histogram_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(R11_MAX_PASSES * R11_DIGITS * sizeof(uint32_t)));
        return r;
    });
    if (e != cudaSuccess) return e;
    const CodeConsts c = code_consts(job.kind, job.descending);
    R11HistParams hp;
    hp.keys = job.keys_in;
    hp.n = (uint32_t)job.n;
    hp.begin_bit = job.begin_bit;
    hp.end_bit = job.end_bit;
    hp.num_passes = job.num_passes;
    hp.enc_a = c.a32;
    hp.enc_b = c.b32;
    hp.enc_a64 = c.a64;
    hp.enc_b64 = c.b64;
    hp.hist = job.hist;
    hp.digit_base = job.digit_base;
    hp.hdr = job.hdr;
    hp.zero_ptr = reinterpret_cast<uint4 *>(job.status);
    hp.zero_vec = (size_t)job.num_tiles * R11_DIGITS * 4 / 16;
    const int sms = device_sms();
    r11_histogram_kernel<K><<<sms, R11_HIST_THREADS, (size_t)job.num_passes * R11_DIGITS * 4, stream>>>(hp);
    ++*launches;
    timing_mark(stream);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    PassParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.keys_in = job.keys_in;
    prm.keys_out = job.keys_out;
    prm.keys_alt = job.keys_alt;
    prm.n = (uint32_t)job.n;
    prm.flip = job.descending ? ~0ull : 0ull;
    prm.enc_a = c.a32;
    prm.enc_b = c.b32;
    prm.enc_a64 = c.a64;
    prm.enc_b64 = c.b64;
    prm.identity = (sizeof(K) == 8 ? (c.a64 | c.b64) == 0ull : (c.a32 | c.b32) == 0u) ? 1 : 0;
    prm.num_passes = job.num_passes;
    prm.in_place = job.in_place ? 1 : 0;
    prm.hdr = job.hdr;
    prm.status = job.status;
    prm.spin_limit = job.spin_limit;
    prm.fault_pass = job.fault_pass;
    prm.fault_tile = job.fault_tile;
    prm.digit_base = job.digit_base;
    prm.prefetch_ahead = (uint32_t)(sms * R11_CTAS_PER_SM / 2);
    for (int p = 0; p < job.num_passes; ++p) {
        prm.pass = p;
        prm.shift = job.begin_bit + R11_BITS * p;
        prm.mask = (1u << std::min(R11_BITS, job.end_bit - prm.shift)) - 1u;
        r11_pass_kernel<K, ITEMS><<<job.num_tiles, R11_THREADS, sizeof(S), stream>>>(prm);
        ++*launches;
        timing_mark(stream);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (job.in_place) {
        CopyParams cp;
        cp.keys_in = job.keys_in;
        cp.keys_out = job.keys_out;
        cp.keys_alt = job.keys_alt;
        cp.vals_in = nullptr;
        cp.vals_out = nullptr;
        cp.vals_alt = nullptr;
        cp.key_bytes_total = job.n * sizeof(K);
        cp.val_bytes_total = 0;
        cp.hdr = job.hdr;
        const size_t blocks = std::min<size_t>((cp.key_bytes_total / 16 + 511) / 512 + 1, (size_t)sms * 4);
        finish_copy_kernel<<<(unsigned)blocks, 512, 0, stream>>>(cp);
        ++*launches;
        timing_mark(stream);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

uint32_t radix11_tile_keys(int key_bytes) {
    return (uint32_t)R11_THREADS * (key_bytes == 8 ? R11Shape<uint64_t>::ITEMS : R11Shape<uint32_t>::ITEMS);
}

cudaError_t launch_radix11_sort(const RadixJob &job, cudaStream_t stream, int *launches) {
    return job.key_bytes == 8 ? r11_sort<uint64_t>(job, stream, launches)
                              : r11_sort<uint32_t>(job, stream, launches);
}

}  // namespace gbs
