// LSD radix sort kernels (8-bit digits): the upfront digit histograms with
// the device-side pass plan, the one-sweep digit pass (tile load, stable
// ballot warp rank, chained scan with decoupled look-back, shared-memory
// staged scatter) and the final copy.
//
// Method: kwkr.cn notes on bitonic vs LSD radix sort §3.1-3.2 (count, exclusive
// prefix, stable placement; block-local counts plus a global base instead of
// global atomics) and §3.4 (skip passes whose digit is constant);
// "GPU基数排序：从CUB工程实现到性能调优" §3 (histogram -> scan -> scatter per
// pass, a stable in-block rank instead of an atomic cursor) and §4 (8-bit
// digits, 16-byte vector loads); "并行排序：从归并网络到 GPU 双调排序" §8.1
// (warp-level histograms, block-local sort before the global write).
#pragma once

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "launch.h"

namespace gbs {
namespace {

constexpr uint32_t FULL = 0xFFFFFFFFu;

// ---------------------------------------------------------------------------
// Block-wide exclusive scan of one value per thread for threads 0..255; all
// threads of the block must call it.  wsum: 8 words of shared memory.  TRAIL:
// end with a barrier, so that wsum may be written again right after; a caller
// that reaches a barrier of its own before touching wsum passes false.
// ---------------------------------------------------------------------------
template <bool TRAIL = true> __device__ __forceinline__ uint32_t excl_scan_256(uint32_t v, uint32_t *wsum) {
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
    if (TRAIL) __syncthreads();
    return base + x - v;
}

// ---------------------------------------------------------------------------
// Peer mask: the lanes of the (fully active) warp whose 8-bit digit equals
// this lane's.  One ballot per digit bit gives the warp's eight bit planes.
// Lane l builds two table entries: the mask of lanes whose low five digit
// bits equal l (planes 0..4) and the mask of lanes whose top three bits equal
// l & 7 (planes 5..7).  Every lane then fetches the entries of its own low and
// high part with two shuffles (the low index is the digit itself: a shuffle
// uses its source lane modulo 32); their AND is the peer mask.  Must be called
// by all 32 lanes.
//
// A plane b agrees with bit k of the lane index where b ^ c_k has its bit
// set, c_k = 0 when that lane bit is set and all ones when it is clear.
// GBS_PEER_IMAD=1 writes b ^ c_k as b * (c_k | 1) + c_k (c_k is 0 or -1), a
// multiply-add on the FMA pipe instead of a logic op; it needs five more
// registers per thread and measured slower at 32 keys per thread.
// ---------------------------------------------------------------------------
#ifndef GBS_PEER_IMAD
#define GBS_PEER_IMAD 0
#endif
#ifndef GBS_ATOM_CLOBBER
#define GBS_ATOM_CLOBBER 0
#endif
#ifndef GBS_STORE_FULL
#define GBS_STORE_FULL 1
#endif



struct PeerTableLane {
    uint32_t c[5];  // 0 where bit k of the lane index is set, all ones where it is clear
    uint32_t m[5];  // c[k] | 1: +1 or -1
    __device__ __forceinline__ explicit PeerTableLane(int lane) {
#pragma unroll
        for (int k = 0; k < 5; ++k) {
            c[k] = (((uint32_t)lane >> k) & 1u) - 1u;
            m[k] = c[k] | 1u;
        }
    }
    __device__ __forceinline__ uint32_t agree(uint32_t b, int k) const {
#if GBS_PEER_IMAD
        return b * m[k] + c[k];
#else
        return b ^ c[k];
#endif
    }
};

__device__ __forceinline__ void warp_peer_halves(uint32_t d, const PeerTableLane &tl, uint32_t &e_lo,
                                                 uint32_t &e_hi) {
    uint32_t b[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = ballot_bits(d, 1u << k);
    const uint32_t lo = tl.agree(b[0], 0) & tl.agree(b[1], 1) & tl.agree(b[2], 2) & tl.agree(b[3], 3) &
                        tl.agree(b[4], 4);
    const uint32_t hi = tl.agree(b[5], 0) & tl.agree(b[6], 1) & tl.agree(b[7], 2);
    e_lo = __shfl_sync(FULL, lo, (int)d);         // lanes agreeing on digit bits 0..4
    e_hi = __shfl_sync(FULL, hi, (int)(d >> 5));  // ... and on bits 5..7
}

// ---------------------------------------------------------------------------
// Upfront histogram of all digit passes (one read of the keys)
// ---------------------------------------------------------------------------

constexpr int HIST_THREADS = 1024;  // one CTA per SM
constexpr int HIST_UNROLL = 4;

// Counters live in per-lane columns: counter (pass p, digit d) of column c is
// word (p*256 + d) * COLS + c, and lane l uses column l % COLS.  With 32
// columns every lane of a warp hits its own bank, so the shared-memory
// atomics of one instruction never conflict (the columns are shared by the
// CTA's warps, whose atomics are separate instructions).
template <typename K> struct HistCfg;
template <> struct HistCfg<uint32_t> {
    static constexpr int PASSES = 4, COLS = 32, PER_VEC = 4;
};
template <> struct HistCfg<uint64_t> {
    static constexpr int PASSES = 8, COLS = 16, PER_VEC = 2;
};
template <typename K> constexpr size_t hist_smem_bytes() {
    return (size_t)HistCfg<K>::PASSES * 256 * HistCfg<K>::COLS * sizeof(uint32_t);
}

struct HistParams {
    const void *keys;
    uint32_t n;
    int kind, begin_bit, end_bit, num_passes;
    uint64_t flip;
    uint32_t enc_a, enc_b;  // branch-free key code: x ^ ((x >>s (w-1)) & a) ^ b (code_consts)
    uint64_t enc_a64, enc_b64;
    uint32_t *hist;
    uint32_t *digit_base;
    Header *hdr;
    uint4 *zero_ptr;  // look-back status words to clear
    size_t zero_vec;  // ... as 16-byte vectors
    int plan;         // compute the pass plan in the last CTA
};

// The code of a key for the full-width histogram (no per-key switch on the
// key kind).
__device__ __forceinline__ uint32_t hist_code(uint32_t x, const HistParams &p) {
    return x ^ (((uint32_t)((int32_t)x >> 31) & p.enc_a) ^ p.enc_b);
}
__device__ __forceinline__ uint64_t hist_code(uint64_t x, const HistParams &p) {
    return x ^ (((uint64_t)((int64_t)x >> 63) & p.enc_a64) ^ p.enc_b64);
}

// FULL: the bit range is the whole key, so every pass's digit is one byte of
// the code (one byte permute) and the number of passes is fixed.
template <typename K, bool FULL>
__global__ void __launch_bounds__(HIST_THREADS, 1) upfront_histogram_kernel(const HistParams prm) {
    using C = HistCfg<K>;
    extern __shared__ __align__(16) uint32_t sh[];
    __shared__ uint32_t wsum[8];
    __shared__ uint32_t s_last;
    const int tid = threadIdx.x;
    const int P = prm.num_passes;

    for (int i = tid; i < P * 256 * C::COLS; i += HIST_THREADS) sh[i] = 0;
    __syncthreads();

    uint32_t *my = sh + (tid & 31) % C::COLS;
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
        if constexpr (FULL) {
            const K t = hist_code(raw, prm);
#pragma unroll
            for (int p = 0; p < C::PASSES; ++p) {
                const uint32_t w = (sizeof(K) == 8 && p >= 4) ? (uint32_t)((uint64_t)t >> 32) : (uint32_t)t;
                atomicAdd(&my[(p * 256 + __byte_perm(w, 0u, 0x4440u | (uint32_t)(p & 3))) * C::COLS], 1u);
            }
        } else {
            const K t = KeyCodec<K>::enc(raw, prm.kind, flip);
#pragma unroll
            for (int p = 0; p < C::PASSES; ++p)
                if (p < P) atomicAdd(&my[(p * 256 + digit_of(t, shift[p], mask[p])) * C::COLS], 1u);
        }
    };

    const size_t n = prm.n;
    const bool aligned = (reinterpret_cast<uintptr_t>(prm.keys) & 15) == 0;
    const size_t nvec = aligned ? n / C::PER_VEC : 0;
    const uint4 *vec = reinterpret_cast<const uint4 *>(prm.keys);
    const size_t stride = (size_t)gridDim.x * HIST_THREADS;
    size_t i = (size_t)blockIdx.x * HIST_THREADS + tid;
    // software-pipelined: the next HIST_UNROLL vectors are in flight while
    // the current ones are counted
    if (i + (HIST_UNROLL - 1) * stride < nvec) {
        uint4 r[HIST_UNROLL];
#pragma unroll
        for (int u = 0; u < HIST_UNROLL; ++u) r[u] = __ldcs(vec + i + u * stride);
        for (;;) {
            const size_t inext = i + HIST_UNROLL * stride;
            const bool more = inext + (HIST_UNROLL - 1) * stride < nvec;
            uint4 q[HIST_UNROLL];
            if (more) {
#pragma unroll
                for (int u = 0; u < HIST_UNROLL; ++u) q[u] = __ldcs(vec + inext + u * stride);
            }
#pragma unroll
            for (int u = 0; u < HIST_UNROLL; ++u) {
                const K *ks = reinterpret_cast<const K *>(&r[u]);
#pragma unroll
                for (int e = 0; e < C::PER_VEC; ++e) count(ks[e]);
            }
            i = inext;
            if (!more) break;
#pragma unroll
            for (int u = 0; u < HIST_UNROLL; ++u) r[u] = q[u];
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
#pragma unroll 8
        for (int c = 0; c < C::COLS; ++c) s += sh[b * C::COLS + ((c + b) % C::COLS)];  // rotated: no conflicts
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

// Value type of a pass with VB value bytes per key (0: keys only).
template <int VB> using ValueT = typename std::conditional<VB == 8, uint64_t, uint32_t>::type;

template <typename K, int VB, int THREADS, int ITEMS> struct PassSmem {
    static constexpr int TILE = THREADS * ITEMS;
    static constexpr int WARPS = THREADS / 32;
    K keys[TILE];
    ValueT<VB> vals[VB ? TILE : 4];
    // per-warp digit counters; after the count phase: sorted-tile slot of the
    // warp's first key of each digit
    uint32_t whist[WARPS][256];
    uint32_t binoff[256];  // global position of sorted-tile slot 0 of each digit
    uint32_t wsum[8];
    uint32_t tile;
    uint32_t num_active;  // active passes of this call
    uint32_t ordinal;     // rank of this pass among them
    alignas(8) uint64_t bar;
};

struct PassParams {
    const void *keys_in;
    void *keys_out;
    void *keys_alt;
    const void *vals_in;  // ValueT<VB> arrays (unused when keys only)
    void *vals_out;
    void *vals_alt;
    uint32_t n;
    // order-preserving code of a key: x ^ ((x >>s (w-1)) & a) ^ b (code_consts)
    uint32_t enc_a, enc_b;
    uint64_t enc_a64, enc_b64;
    uint64_t flip;  // all ones when descending
    int pass, num_passes, shift;
    uint32_t mask;
    uint32_t perm_sel;  // byte-permute selector of the digit byte (byte-aligned passes)
    int in_place;
    int identity;  // the key code is the identity (no transform on load or store)
    Header *hdr;
    const uint32_t *digit_base;
    void *status;  // SW words: uint32_t below 2^29 keys, uint64_t above
    uint32_t spin_limit;
    int fault_pass;
    uint32_t fault_tile;
    // the CTA of tile t prefetches tile t + prefetch_ahead into L2 (0: none);
    // set to about half the CTAs resident on the device, so the data arrive
    // well before that tile's CTA starts and are still in L2 when it does
    uint32_t prefetch_ahead;
};

template <typename K> struct Xform;
template <> struct Xform<uint32_t> {
    static __device__ __forceinline__ uint32_t enc(uint32_t x, const PassParams &p) {
        return x ^ (((uint32_t)((int32_t)x >> 31) & p.enc_a) ^ p.enc_b);
    }
    static __device__ __forceinline__ uint32_t dec(uint32_t t, const PassParams &p) {
        const uint32_t f = (uint32_t)p.flip;
        const uint32_t u = t ^ f;  // code without the descending complement
        return u ^ ((~(uint32_t)((int32_t)u >> 31) & p.enc_a) ^ (p.enc_b ^ f));
    }
};
template <> struct Xform<uint64_t> {
    static __device__ __forceinline__ uint64_t enc(uint64_t x, const PassParams &p) {
        return x ^ (((uint64_t)((int64_t)x >> 63) & p.enc_a64) ^ p.enc_b64);
    }
    static __device__ __forceinline__ uint64_t dec(uint64_t t, const PassParams &p) {
        const uint64_t u = t ^ p.flip;  // code without the descending complement
        return u ^ ((~(uint64_t)((int64_t)u >> 63) & p.enc_a64) ^ (p.enc_b64 ^ p.flip));
    }
};

// Digit of a code for this pass.  BYTE: the digit is a whole byte of the
// code (begin_bit a multiple of 8 and an 8-bit digit), extracted with one
// byte permute.
template <bool BYTE> __device__ __forceinline__ uint32_t pass_digit(uint32_t t, const PassParams &p) {
    return BYTE ? __byte_perm(t, 0u, p.perm_sel) : digit_of(t, p.shift, p.mask);
}
template <bool BYTE> __device__ __forceinline__ uint32_t pass_digit(uint64_t t, const PassParams &p) {
    if (BYTE) {
        const uint32_t w = p.shift >= 32 ? (uint32_t)(t >> 32) : (uint32_t)t;
        return __byte_perm(w, 0u, p.perm_sel);
    }
    return digit_of(t, p.shift, p.mask);
}

// dst[lo, hi) = src[lo, hi) by the CTA's threads, 16 bytes at a time when both
// ranges are 16-byte aligned.
template <typename K>
__device__ __forceinline__ void copy_range(const K *src, K *dst, size_t lo, size_t hi, int tid, int nthreads) {
    const K *s = src + lo;
    K *d = dst + lo;
    const size_t cnt = hi - lo;
    size_t done = 0;
    if (((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(d)) & 15) == 0) {
        constexpr size_t PER = 16 / sizeof(K);
        const size_t nv = cnt / PER;
        const uint4 *sv = reinterpret_cast<const uint4 *>(s);
        uint4 *dv = reinterpret_cast<uint4 *>(d);
        for (size_t i = tid; i < nv; i += nthreads) dv[i] = __ldcs(sv + i);
        done = nv * PER;
    }
    for (size_t i = done + tid; i < cnt; i += nthreads) d[i] = s[i];
}

// Stable warp rank of a full tile's keys (see the kernel); ENC applies the
// key code on load (first active pass).  The highest lane of each digit group
// adds the group size to the warp's counter with one shared-memory atomic and
// hands the old value to its peers.
// In-tile ranks are kept as 16-bit halves, two per register.
template <int ITEMS> struct PackedRanks {
    uint32_t r[(ITEMS + 1) / 2];
    __device__ __forceinline__ void set(int i, uint32_t v) {  // v < 2^16
        if (i & 1)
            r[i >> 1] = __byte_perm(r[i >> 1], v, 0x5410);
        else
            r[i >> 1] = v;
    }
    __device__ __forceinline__ void replace(int i, uint32_t v) {
        if (i & 1)
            r[i >> 1] = (r[i >> 1] & 0xFFFFu) | (v << 16);
        else
            r[i >> 1] = (r[i >> 1] & 0xFFFF0000u) | v;
    }
    __device__ __forceinline__ uint32_t get(int i) const { return (i & 1) ? (r[i >> 1] >> 16) : (r[i >> 1] & 0xFFFFu); }
};

// Stable warp rank.  Warp w owns tile slots [w*ITEMS*32, (w+1)*ITEMS*32);
// item i of lane l is slot w*ITEMS*32 + 32 i + l, so (warp, item, lane) is
// input order.  Lanes holding the same digit find each other (peer mask); the
// highest of them advances the warp's counter for that digit by the group
// size with one shared-memory atomic and hands the old value to its peers.
// ENC applies the key code on load (first active pass).  Output: keys (coded)
// and their ranks within the warp's digit groups; whist ends holding the
// warp's digit counts.
template <bool ENC, typename K>
__device__ __forceinline__ K load_key(const K *tile_keys, uint32_t idx, bool ok, const PassParams &prm) {
    K key = ok ? tile_keys[idx] : (K)0;
    if (ENC) key = Xform<K>::enc(key, prm);
    return key;
}

template <bool ENC, bool BYTE, bool FULLTILE, typename K, int ITEMS>
__device__ __forceinline__ void rank_warp(const K *tile_keys, uint32_t *whist, const PassParams &prm, int warp,
                                          int lane, uint32_t valid, K (&keys)[ITEMS], PackedRanks<ITEMS> &ranks) {
    const PeerTableLane nl(lane);
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
        keys[i] = load_key<ENC>(tile_keys, idx, FULLTILE || idx < valid, prm);
    }
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const uint32_t d = pass_digit<BYTE>(keys[i], prm);
        uint32_t e_lo, e_hi;
        warp_peer_halves(d, nl, e_lo, e_hi);
        uint32_t peers = e_lo & e_hi;
        bool ok = true;
        if (!FULLTILE) {
            const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
            ok = idx < valid;
            const uint32_t vmask = ballot_bits(ok ? 1u : 0u, 1u);
            peers &= ok ? vmask : 0u;
        }
        // leader: the highest lane of the group (bfind: index of the top set
        // bit; all ones for the empty mask of a lane past the tile's end, which
        // then matches no lane)
        uint32_t leader;
        asm("bfind.u32 %0, %1;" : "=r"(leader) : "r"(peers));
        // peers below this lane; at the leader (the top lane) that is the
        // group size minus one
        const uint32_t below = __popc(peers & lt);
        // the leader's atomic, predicated rather than branched around
        uint32_t before = 0;
#if GBS_ATOM_CLOBBER
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.eq.u32 p, %1, %2;\n\t@p atom.shared.add.u32 %0, [%3], %4;\n\t}"
            : "+r"(before)
            : "r"((uint32_t)lane), "r"(leader), "r"(smem_u32(&whist[d])), "r"(below + 1u)
            : "memory");
#else
        // volatile keeps the warp's atomics in program order; no memory
        // clobber: nothing reads the counters through ordinary loads before
        // the CTA barrier that ends the rank, so the compiler may move other
        // items' work across the atomic
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.eq.u32 p, %1, %2;\n\t@p atom.shared.add.u32 %0, [%3], %4;\n\t}"
            : "+r"(before)
            : "r"((uint32_t)lane), "r"(leader), "r"(smem_u32(&whist[d])), "r"(below + 1u));
#endif
        const uint32_t b = __shfl_sync(FULL, before, (int)leader);
        ranks.set(i, ok ? b + below : 0u);
    }
}

// Coalesced scatter of the sorted tile: consecutive slots of one digit go to
// consecutive global positions.  DEC applies the inverse key code (last pass).
#ifndef GBS_STORE_UNROLL
#define GBS_STORE_UNROLL 4
#endif
constexpr int STORE_UNROLL = GBS_STORE_UNROLL;
template <bool DEC, bool BYTE, typename K, int VB, int THREADS>
__device__ __forceinline__ void store_tile(const K *sk, const ValueT<VB> *sv, const uint32_t *binoff, uint32_t valid,
                                           K *kdst, ValueT<VB> *vdst, const PassParams &prm, int tid) {
#pragma unroll STORE_UNROLL
    for (uint32_t j = tid; j < valid; j += THREADS) {
        const K key = sk[j];
        const uint32_t pos = binoff[pass_digit<BYTE>(key, prm)] + j;
        // always true unless a bounded wait gave up (an error is then recorded):
        // counts taken from a tile that never landed must not move a store out
        // of the output
        if (pos < prm.n) {
            kdst[pos] = DEC ? Xform<K>::dec(key, prm) : key;
            if (VB) vdst[pos] = sv[j];
        }
    }
}

// Full-tile form: every slot holds a key, and the caller has checked once for
// the whole tile that every digit's positions lie inside the output.
template <bool DEC, bool BYTE, typename K, int VB, int THREADS, int ITEMS>
__device__ __forceinline__ void store_tile_full(const K *sk, const ValueT<VB> *sv, const uint32_t *binoff, K *kdst,
                                                ValueT<VB> *vdst, const PassParams &prm, int tid) {
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const uint32_t j = (uint32_t)(tid + it * THREADS);
        const K key = sk[j];
        const uint32_t pos = binoff[pass_digit<BYTE>(key, prm)] + j;
        kdst[pos] = DEC ? Xform<K>::dec(key, prm) : key;
        if (VB) vdst[pos] = sv[j];
    }
}

// Bounded wait for phase `parity` of the tile-load barrier; a copy that never
// lands records ERR_COPY_TIMEOUT instead of hanging.
__device__ __forceinline__ void wait_phase(uint64_t *bar, uint32_t parity, const PassParams &prm, Header *hdr,
                                           uint32_t tile) {
    uint32_t polls = 0;
    while (!mbar_try_wait(bar, parity & 1u)) {
        if (++polls > prm.spin_limit) {
            record_error(hdr, ERR_COPY_TIMEOUT, ((uint32_t)prm.pass << 24) | (tile & 0xFFFFFFu));
            break;
        }
        if (polls > 16) __nanosleep(64);
    }
}

#ifndef LOOKBACK_WINDOW
#define LOOKBACK_WINDOW 6
#endif

// Status words of predecessors lb_next, lb_next - 1, ... for digit d; a
// position before tile 0 reads as an inclusive prefix of 0.
template <int W, typename SW>
__device__ __forceinline__ void load_window(SW (&sw)[W], const SW *status, int32_t lb_next, int d, uint32_t st_inc) {
#pragma unroll
    for (int w = 0; w < W; ++w)
        sw[w] = (lb_next - w >= 0) ? ld_relaxed_gpu(status + (size_t)(lb_next - w) * 256 + d)
                                   : ((SW)st_inc << StatusWord<SW>::COUNT_BITS);
}

// Adds a window's counts, nearest predecessor first, through the first
// inclusive prefix (done); stops before a predecessor that has published
// nothing yet.  used: predecessors consumed.
template <int W, typename SW>
__device__ __forceinline__ void add_window(const SW (&sw)[W], uint32_t st_agg, uint32_t &excl, int &used,
                                           bool &done) {
    constexpr int CB = StatusWord<SW>::COUNT_BITS;
    constexpr SW CM = StatusWord<SW>::COUNT_MASK;
    // this pass's states are st_agg (aggregate) and st_agg + 1 (inclusive
    // prefix).  Subtracting the aggregate state's bits leaves the count of an
    // aggregate and a value above COUNT_MASK for any other word (unsigned
    // wrap-around included), so one subtraction both tests and extracts.
    const SW agg = (SW)st_agg << CB;
    used = 0;
    done = false;
#pragma unroll
    for (int w = 0; w < W; ++w) {
        const SW c = sw[w] - agg;
        if (c > CM) {  // not an aggregate of this pass: an inclusive prefix ends the walk
            const SW ci = c - ((SW)1 << CB);
            if (ci <= CM) {
                excl += (uint32_t)ci;
                used = w + 1;
                done = true;
            }
            break;
        }
        excl += (uint32_t)c;
        used = w + 1;
    }
}

// Exclusive prefix of digit d over the tiles before `tile` > 0 (decoupled
// look-back): reads LOOKBACK_WINDOW predecessors per round trip, adds the
// aggregates from the nearest one back to the first inclusive prefix, and
// waits (bounded) only at a predecessor that has published nothing yet.
template <typename SW>
__device__ __forceinline__ uint32_t lookback_excl(const PassParams &prm, Header *hdr, uint32_t tile, int d,
                                                  uint32_t st_agg, uint32_t st_inc) {
    uint32_t excl = 0;
    int32_t lb_next = (int32_t)tile - 1;  // nearest predecessor not yet added
    uint32_t polls = 0;
    bool done = false;
    while (!done) {
        SW sw[LOOKBACK_WINDOW];
        load_window(sw, reinterpret_cast<const SW *>(prm.status), lb_next, d, st_inc);
        int used;
        add_window(sw, st_agg, excl, used, done);
        if (done) break;
        lb_next -= used;
        if (used == 0) {
            if (++polls > prm.spin_limit) {
                record_error(hdr, ERR_LOOKBACK_TIMEOUT, ((uint32_t)prm.pass << 24) | (tile & 0xFFFFFFu));
                break;
            }
            __nanosleep(polls < 64 ? 32 : 256);
        }
    }
    return excl;
}

// The tile's count of digit d (thread d < 256), the sum of the warps'
// counters.  WRITE_RUN: the counters also become each warp's exclusive offset
// within the digit's keys (else warp_offsets does that after the tile scan,
// with one store per counter instead of two).
template <int WARPS, bool WRITE_RUN>
__device__ __forceinline__ uint32_t tile_digit_count(uint32_t (*whist)[256], int d) {
    uint32_t run = 0;
#pragma unroll 4
    for (int w = 0; w < WARPS; ++w) {
        const uint32_t c = whist[w][d];
        if (WRITE_RUN) whist[w][d] = run;
        run += c;
    }
    return run;
}

// Sorted-tile slot of each warp's first key of digit d, from the digit's
// offset in the tile (local).  RUN_WRITTEN: the counters already hold the
// warps' exclusive offsets within the digit.
template <int WARPS, bool RUN_WRITTEN>
__device__ __forceinline__ void warp_offsets(uint32_t (*whist)[256], int d, uint32_t local) {
    uint32_t run = local;
#pragma unroll 4
    for (int w = 0; w < WARPS; ++w) {
        const uint32_t c = whist[w][d];
        whist[w][d] = RUN_WRITTEN ? c + local : run;
        run += c;
    }
}

// Source and destination buffers of active pass number k of A.  The last
// active pass lands in the output (or in the scratch buffer when an in-place
// call has an odd number of active passes, which keeps every pass out of
// place; the copy kernel then finishes).
template <typename K, int VB> struct PassIO {
    using V = ValueT<VB>;
    const K *ksrc;
    K *kdst;
    const V *vsrc = nullptr;
    V *vdst = nullptr;
    __device__ __forceinline__ PassIO(const PassParams &prm, uint32_t A, uint32_t k) {
        const bool odd_in_place = prm.in_place && (A & 1u);
        K *kout = reinterpret_cast<K *>(prm.keys_out), *kalt = reinterpret_cast<K *>(prm.keys_alt);
        K *k_last = odd_in_place ? kalt : kout, *k_other = odd_in_place ? kout : kalt;
        const bool src_last = ((A - k) & 1u) == 0, dst_last = ((A - 1 - k) & 1u) == 0;
        ksrc = (k == 0) ? reinterpret_cast<const K *>(prm.keys_in) : (src_last ? k_last : k_other);
        kdst = dst_last ? k_last : k_other;
        if (VB) {
            V *vout = reinterpret_cast<V *>(prm.vals_out), *valt = reinterpret_cast<V *>(prm.vals_alt);
            V *v_last = odd_in_place ? valt : vout;
            V *v_other = odd_in_place ? vout : valt;
            vsrc = (k == 0) ? reinterpret_cast<const V *>(prm.vals_in) : (src_last ? v_last : v_other);
            vdst = dst_last ? v_last : v_other;
        }
    }
};

// Everything after the tile load: stable rank, tile counts and aggregate,
// reorder in shared memory, look-back, scatter.  FULLTILE: the tile holds
// TILE keys (every tile but a ragged last one).
template <bool FULLTILE, typename K, int VB, int THREADS, int ITEMS, bool BYTE, typename SW>
__device__ __forceinline__ void pass_tile(PassSmem<K, VB, THREADS, ITEMS> &sm, const PassParams &prm, Header *hdr,
                                          const uint32_t valid, const bool first) {
    constexpr bool PAIRS = VB != 0;
    using V = ValueT<VB>;
    constexpr int WARPS = THREADS / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // ---- stable rank within the tile --------------------------------------
    K keys[ITEMS];
    PackedRanks<ITEMS> ranks;
    uint32_t *whist = sm.whist[warp];
    if (first)
        rank_warp<true, BYTE, FULLTILE>(sm.keys, whist, prm, warp, lane, valid, keys, ranks);
    else
        rank_warp<false, BYTE, FULLTILE>(sm.keys, whist, prm, warp, lane, valid, keys, ranks);
    __syncthreads();

    // values not needed during the rank are fetched now, so that they hold no
    // registers across it
    const uint32_t tile = sm.tile, A = sm.num_active, k = sm.ordinal;
    const bool last = (k + 1 == A) && !prm.identity;
    // chained-scan states of this pass (rotated by ordinal, see common.cuh)
    const uint32_t st_agg = 1u + 2u * (k % 3u), st_inc = 2u + 2u * (k % 3u);
    const uint32_t dbase = (tid < 256) ? prm.digit_base[prm.pass * 256 + tid] : 0u;
    const PassIO<K, VB> io(prm, A, k);
    K *kdst = io.kdst;
    V *vdst = io.vdst;

    // ---- tile digit counts, warp offsets, publish the aggregate ------------
    uint32_t cnt = 0;
    constexpr int CB = StatusWord<SW>::COUNT_BITS;
    // 32-bit keys write the warps' offsets once, after the tile scan; for
    // 64-bit keys that form measured slower (its register allocation spills
    // more), so they write the offsets within the digit first and add the
    // tile offset after the scan
    constexpr bool RUN_FIRST = sizeof(K) == 8;
    const bool faulty = (prm.fault_pass == prm.pass) && (prm.fault_tile == tile);
    SW *my_status = reinterpret_cast<SW *>(prm.status) + (size_t)tile * 256;
    if (tid < 256) {
        cnt = tile_digit_count<WARPS, RUN_FIRST>(sm.whist, tid);
        if (!faulty) st_relaxed_gpu(my_status + tid, ((SW)(tile == 0 ? st_inc : st_agg) << CB) | cnt);
    }
    // (wsum is not written again before the barrier after the offsets)
    const uint32_t local = excl_scan_256<false>(cnt, sm.wsum);
    if (tid < 256) {
        // sorted-tile slot of each warp's first key of digit tid
        warp_offsets<WARPS, RUN_FIRST>(sm.whist, tid, local);
    }
    __syncthreads();

    // ---- reorder the tile in shared memory by (digit, rank) ---------------
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
        if (FULLTILE || idx < valid) {
            const uint32_t slot = ranks.get(i) + whist[pass_digit<BYTE>(keys[i], prm)];
            if (PAIRS) ranks.replace(i, slot);
            sm.keys[slot] = keys[i];
        }
    }
    if (PAIRS) {
        V vals[ITEMS];
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
            const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
            vals[i] = (idx < valid) ? sm.vals[idx] : V(0);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
            const uint32_t idx = (uint32_t)warp * (ITEMS * 32) + i * 32 + lane;
            if (idx < valid) sm.vals[ranks.get(i)] = vals[i];
        }
    }

    // ---- decoupled look-back over the predecessors' status words ----------
    // Each digit's thread reads LOOKBACK_WINDOW predecessors per round trip
    // (registers are free again: the tile's keys now sit in shared memory),
    // adds the aggregates from the nearest one back to the first inclusive
    // prefix, and waits (bounded) only at a predecessor that has published
    // nothing yet.
    bool out_of_range = false;
    if (tid < 256) {
        uint32_t excl = 0;
        if (tile > 0) {
            excl = lookback_excl<SW>(prm, hdr, tile, tid, st_agg, st_inc);
            if (!faulty)
                st_relaxed_gpu(my_status + tid, ((SW)st_inc << CB) | ((SW)(excl + cnt) & StatusWord<SW>::COUNT_MASK));
        }
        sm.binoff[tid] = dbase + excl - local;
        // every position of digit tid lies in [dbase + excl, dbase + excl + cnt); with counts
        // from a tile that never landed (a bounded wait gave up) they may not
        out_of_range = cnt != 0 && (uint64_t)dbase + excl + cnt > (uint64_t)prm.n;
    }
#if GBS_STORE_FULL
    if (FULLTILE) {
        const int bad = __syncthreads_or(out_of_range);
        if (bad) {
            if (tid == 0) record_error(hdr, ERR_COPY_TIMEOUT, ((uint32_t)prm.pass << 24) | (tile & 0xFFFFFFu));
            return;
        }
        if (last)
            store_tile_full<true, BYTE, K, VB, THREADS, ITEMS>(sm.keys, sm.vals, sm.binoff, kdst, vdst, prm, tid);
        else
            store_tile_full<false, BYTE, K, VB, THREADS, ITEMS>(sm.keys, sm.vals, sm.binoff, kdst, vdst, prm, tid);
        return;
    }
#endif
    (void)out_of_range;
    __syncthreads();

    if (last)
        store_tile<true, BYTE, K, VB, THREADS>(sm.keys, sm.vals, sm.binoff, valid, kdst, vdst, prm, tid);
    else
        store_tile<false, BYTE, K, VB, THREADS>(sm.keys, sm.vals, sm.binoff, valid, kdst, vdst, prm, tid);
}

// Launch shapes of the pass kernel: threads per CTA x keys per thread, and the
// CTAs kept resident per SM (which sets the register budget: 65536 / (CTAs x
// threads), in steps of 8).  Four 256-thread CTAs (64 registers) suit u32
// keys.  Values and 64-bit keys need more registers per key: three CTAs at 80
// registers then hold more keys per tile without spilling, which measured
// faster than four smaller tiles with spills or two larger ones.  More,
// smaller tiles per SM let the latency-bound phases (tile load, look-back,
// scatter) overlap other tiles' ranking; larger tiles spend less on per-tile
// costs.
#ifndef GBS_U32_THREADS
#define GBS_U32_THREADS 256
#endif
#ifndef GBS_U32_ITEMS
#define GBS_U32_ITEMS 32
#endif
#ifndef GBS_U32_CTAS
#define GBS_U32_CTAS 4
#endif
#ifndef GBS_U32_PAIR_THREADS
#define GBS_U32_PAIR_THREADS 256
#endif
#ifndef GBS_U32_PAIR_ITEMS
#define GBS_U32_PAIR_ITEMS 32
#endif
#ifndef GBS_U32_PAIR_CTAS
#define GBS_U32_PAIR_CTAS 3
#endif
#ifndef GBS_U64_THREADS
#define GBS_U64_THREADS 256
#endif
#ifndef GBS_U64_ITEMS
#define GBS_U64_ITEMS 24
#endif
#ifndef GBS_U64_CTAS
#define GBS_U64_CTAS 3
#endif
#ifndef GBS_U64_PAIR_THREADS
#define GBS_U64_PAIR_THREADS 256
#endif
#ifndef GBS_U64_PAIR_ITEMS
#define GBS_U64_PAIR_ITEMS 20
#endif
#ifndef GBS_U64_PAIR_CTAS
#define GBS_U64_PAIR_CTAS 3
#endif
// 64-bit values
#ifndef GBS_U32_V64_THREADS
#define GBS_U32_V64_THREADS 256
#endif
#ifndef GBS_U32_V64_ITEMS
#define GBS_U32_V64_ITEMS 20
#endif
#ifndef GBS_U32_V64_CTAS
#define GBS_U32_V64_CTAS 3
#endif
#ifndef GBS_U64_V64_THREADS
#define GBS_U64_V64_THREADS 256
#endif
#ifndef GBS_U64_V64_ITEMS
#define GBS_U64_V64_ITEMS 16
#endif
#ifndef GBS_U64_V64_CTAS
#define GBS_U64_V64_CTAS 3
#endif

template <typename K, int VB> struct PassShape;
template <> struct PassShape<uint32_t, 0> {
    static constexpr int THREADS = GBS_U32_THREADS, ITEMS = GBS_U32_ITEMS, CTAS = GBS_U32_CTAS;
};
template <> struct PassShape<uint32_t, 4> {
    static constexpr int THREADS = GBS_U32_PAIR_THREADS, ITEMS = GBS_U32_PAIR_ITEMS, CTAS = GBS_U32_PAIR_CTAS;
};
template <> struct PassShape<uint32_t, 8> {
    static constexpr int THREADS = GBS_U32_V64_THREADS, ITEMS = GBS_U32_V64_ITEMS, CTAS = GBS_U32_V64_CTAS;
};
template <> struct PassShape<uint64_t, 0> {
    static constexpr int THREADS = GBS_U64_THREADS, ITEMS = GBS_U64_ITEMS, CTAS = GBS_U64_CTAS;
};
template <> struct PassShape<uint64_t, 4> {
    static constexpr int THREADS = GBS_U64_PAIR_THREADS, ITEMS = GBS_U64_PAIR_ITEMS, CTAS = GBS_U64_PAIR_CTAS;
};
template <> struct PassShape<uint64_t, 8> {
    static constexpr int THREADS = GBS_U64_V64_THREADS, ITEMS = GBS_U64_V64_ITEMS, CTAS = GBS_U64_V64_CTAS;
};

template <typename K, int VB, int THREADS, int ITEMS, bool BYTE, typename SW>
__global__ void __launch_bounds__(THREADS, PassShape<K, VB>::CTAS)
    onesweep_pass_kernel(const PassParams prm) {
    constexpr bool PAIRS = VB != 0;
    using V = ValueT<VB>;
    static_assert(THREADS * ITEMS <= 65536, "in-tile ranks are 16-bit");
    using S = PassSmem<K, VB, THREADS, ITEMS>;
    constexpr int TILE = S::TILE;
    constexpr int WARPS = S::WARPS;
    // one thread per digit in the count, scan and look-back phases
    static_assert(THREADS >= 256 && THREADS % 32 == 0, "the pass kernel needs at least 256 threads");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    S &sm = *reinterpret_cast<S *>(smem_raw);

    const int tid = threadIdx.x;
    Header *hdr = prm.hdr;
    const uint32_t A = hdr->num_active;
    const bool active = (hdr->active_mask >> prm.pass) & 1u;
    if (!active) {
        // Every pass is trivial: the input order is already sorted; the last
        // pass kernel copies it to the output (the in-place case needs none
        // for the keys and is finished by the copy kernel).
        if (A == 0 && prm.pass == prm.num_passes - 1 && !prm.in_place && (size_t)blockIdx.x * TILE < prm.n) {
            const size_t lo = (size_t)blockIdx.x * TILE, hi = min((size_t)prm.n, lo + TILE);
            copy_range(reinterpret_cast<const K *>(prm.keys_in), reinterpret_cast<K *>(prm.keys_out), lo, hi, tid,
                       THREADS);
            if (PAIRS)
                copy_range(reinterpret_cast<const V *>(prm.vals_in), reinterpret_cast<V *>(prm.vals_out), lo, hi, tid,
                           THREADS);
        }
        return;
    }
    const uint32_t k = hdr->ordinal[prm.pass];
    // the key code is applied on the first active pass's load and undone on
    // the last one's store, unless it is the identity (unsigned ascending)
    const bool first = (k == 0) && !prm.identity;

    const PassIO<K, VB> io(prm, A, k);
    const K *ksrc = io.ksrc;
    const V *vsrc = io.vsrc;

    const bool aligned = ((reinterpret_cast<uintptr_t>(ksrc) & 15) == 0) &&
                         (!PAIRS || ((reinterpret_cast<uintptr_t>(vsrc) & 15) == 0));
    const uint32_t tx_bytes = TILE * (uint32_t)(sizeof(K) + VB);

    // ---- tile and its load -----------------------------------------------
    // The CTA's tile is its block index, so the copy is issued at once.  The
    // look-back of tile t waits for tiles below t, which relies on the CTAs of
    // a grid being dispatched in increasing block order, as the hardware does
    // (the common single-pass scans rely on the same).  An atomic ticket would
    // guarantee progress whatever the dispatch order, but its round trip sits
    // before every tile copy: 3.5% per sort.  Every wait here is bounded, so a
    // predecessor that never ran would end in a recorded timeout, never a hang.
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
        const uint32_t t = blockIdx.x;
        sm.tile = t;
        const size_t start = (size_t)t * TILE;
        if (aligned && start + TILE <= (size_t)prm.n) {
            mbar_arrive_expect_tx(&sm.bar, tx_bytes);
            bulk_g2s(sm.keys, ksrc + start, TILE * (uint32_t)sizeof(K), &sm.bar);
            if (PAIRS) bulk_g2s(sm.vals, vsrc + start, TILE * (uint32_t)VB, &sm.bar);
        }
        const size_t pf = (size_t)t + prm.prefetch_ahead;
        if (prm.prefetch_ahead != 0 && aligned && (pf + 1) * TILE <= (size_t)prm.n) {
            prefetch_l2_bulk(ksrc + pf * TILE, TILE * (uint32_t)sizeof(K));
            if (PAIRS) prefetch_l2_bulk(vsrc + pf * TILE, TILE * (uint32_t)VB);
        }
    }
    if (tid == 0) {
        sm.num_active = A;
        sm.ordinal = k;
    }
    for (int i = tid; i < WARPS * 256; i += THREADS) (&sm.whist[0][0])[i] = 0;
    __syncthreads();
    const uint32_t tile = sm.tile;
    const size_t tile_start = (size_t)tile * TILE;
    const uint32_t valid = tile_start < prm.n ? (uint32_t)min((size_t)TILE, (size_t)prm.n - tile_start) : 0u;
    if (valid == TILE && aligned) {
        wait_phase(&sm.bar, 0, prm, hdr, tile);
    } else {
        for (uint32_t i = tid; i < valid; i += THREADS) {
            sm.keys[i] = ksrc[tile_start + i];
            if (PAIRS) sm.vals[i] = vsrc[tile_start + i];
        }
        __syncthreads();
    }

    if (valid == TILE)
        pass_tile<true, K, VB, THREADS, ITEMS, BYTE, SW>(sm, prm, hdr, valid, first);
    else
        pass_tile<false, K, VB, THREADS, ITEMS, BYTE, SW>(sm, prm, hdr, valid, first);
}

// ---------------------------------------------------------------------------
// Final copy for in-place calls
// ---------------------------------------------------------------------------

struct CopyParams {
    const void *keys_in;
    void *keys_out;
    const void *keys_alt;
    const void *vals_in;
    void *vals_out;
    const void *vals_alt;
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

// SM count of the current device (cached per device).
inline int device_sms() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    int sms = (dev >= 0 && dev < 64) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (sms <= 0) {
        if (dev < 0 || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return 1;
        if (dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
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
    {
        const CodeConsts c = code_consts(job.kind, job.descending);
        prm.enc_a = c.a32;
        prm.enc_b = c.b32;
        prm.enc_a64 = c.a64;
        prm.enc_b64 = c.b64;
    }
    prm.hist = job.hist;
    prm.digit_base = job.digit_base;
    prm.hdr = job.hdr;
    prm.zero_ptr = reinterpret_cast<uint4 *>(job.status);
    prm.zero_vec = plan ? (size_t)job.num_tiles * 256 * (job.wide_status ? 8 : 4) / 16 : 0;
    prm.plan = plan ? 1 : 0;
    const bool full = job.begin_bit == 0 && job.end_bit == 8 * (int)sizeof(K);
    static PerDeviceOnce once;
    cudaError_t e = once.run([] {
        cudaError_t r = cudaFuncSetAttribute(upfront_histogram_kernel<K, true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hist_smem_bytes<K>());
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(upfront_histogram_kernel<K, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)hist_smem_bytes<K>());
        return r;
    });
    if (e != cudaSuccess) return e;
    const size_t per_cta = (size_t)HIST_THREADS * HIST_UNROLL * HistCfg<K>::PER_VEC;
    size_t grid = std::max<size_t>((job.n + per_cta - 1) / per_cta, (prm.zero_vec + HIST_THREADS - 1) / HIST_THREADS);
    grid = std::min<size_t>(grid, (size_t)device_sms());
    grid = std::max<size_t>(grid, 1);
    if (full)
        upfront_histogram_kernel<K, true><<<(unsigned)grid, HIST_THREADS, hist_smem_bytes<K>(), stream>>>(prm);
    else
        upfront_histogram_kernel<K, false><<<(unsigned)grid, HIST_THREADS, hist_smem_bytes<K>(), stream>>>(prm);
    ++*launches;
    timing_mark(stream);
    return cudaGetLastError();
}

// One pass-kernel instantiation: the one-time shared-memory attribute set-up
// and the launch of one CTA per tile.
template <typename K, int VB, int THREADS, int ITEMS, bool BYTE, typename SW> struct PassLaunch {
    using S = PassSmem<K, VB, THREADS, ITEMS>;
    static cudaError_t launch(uint32_t num_tiles, const PassParams &prm, cudaStream_t stream) {
        static PerDeviceOnce once;
        const cudaError_t e = once.run([] {
            return cudaFuncSetAttribute(onesweep_pass_kernel<K, VB, THREADS, ITEMS, BYTE, SW>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(S));
        });
        if (e != cudaSuccess) return e;
        onesweep_pass_kernel<K, VB, THREADS, ITEMS, BYTE, SW><<<num_tiles, THREADS, sizeof(S), stream>>>(prm);
        return cudaGetLastError();
    }
};

template <typename K, int VB, int THREADS, int ITEMS, typename SW>
cudaError_t launch_passes(const RadixJob &job, cudaStream_t stream, int *launches) {
    const bool byte_digits = (job.begin_bit % 8) == 0;
    PassParams prm;
    prm.keys_in = job.keys_in;
    prm.keys_out = job.keys_out;
    prm.keys_alt = job.keys_alt;
    prm.vals_in = job.vals_in;
    prm.vals_out = job.vals_out;
    prm.vals_alt = job.vals_alt;
    prm.n = (uint32_t)job.n;
    prm.flip = job.descending ? ~0ull : 0ull;
    {
        const CodeConsts c = code_consts(job.kind, job.descending);
        prm.enc_a = c.a32;
        prm.enc_b = c.b32;
        prm.enc_a64 = c.a64;
        prm.enc_b64 = c.b64;
        prm.identity = (sizeof(K) == 8 ? (c.a64 | c.b64) == 0ull : (c.a32 | c.b32) == 0u) ? 1 : 0;
    }
    prm.num_passes = job.num_passes;
    prm.in_place = job.in_place ? 1 : 0;
    prm.hdr = job.hdr;
    prm.status = job.status;
    prm.spin_limit = job.spin_limit;
    prm.fault_pass = job.fault_pass;
    prm.fault_tile = job.fault_tile;
    prm.digit_base = job.digit_base;
    prm.prefetch_ahead = (uint32_t)(device_sms() * PassShape<K, VB>::CTAS / 2);
    for (int p = 0; p < job.num_passes; ++p) {
        prm.pass = p;
        prm.shift = job.begin_bit + 8 * p;
        const int bits = std::min(8, job.end_bit - prm.shift);
        prm.mask = (1u << bits) - 1u;
        prm.perm_sel = 0x4440u | (uint32_t)((prm.shift & 31) >> 3);
        const cudaError_t e =
            (byte_digits && bits == 8) ? PassLaunch<K, VB, THREADS, ITEMS, true, SW>::launch(job.num_tiles, prm, stream)
                                       : PassLaunch<K, VB, THREADS, ITEMS, false, SW>::launch(job.num_tiles, prm, stream);
        if (e != cudaSuccess) return e;
        ++*launches;
        timing_mark(stream);
    }
    return cudaSuccess;
}

// Every digit pass of a radix job, with status words of type SW.
template <typename K, int VB, typename SW>
cudaError_t launch_shape(const RadixJob &job, cudaStream_t stream, int *launches) {
    return launch_passes<K, VB, PassShape<K, VB>::THREADS, PassShape<K, VB>::ITEMS, SW>(job, stream, launches);
}

template <typename SW> cudaError_t launch_all_passes(const RadixJob &job, cudaStream_t stream, int *launches) {
    if (job.key_bytes == 8)
        return job.val_bytes == 8 ? launch_shape<uint64_t, 8, SW>(job, stream, launches)
               : job.val_bytes    ? launch_shape<uint64_t, 4, SW>(job, stream, launches)
                                  : launch_shape<uint64_t, 0, SW>(job, stream, launches);
    return job.val_bytes == 8 ? launch_shape<uint32_t, 8, SW>(job, stream, launches)
           : job.val_bytes    ? launch_shape<uint32_t, 4, SW>(job, stream, launches)
                              : launch_shape<uint32_t, 0, SW>(job, stream, launches);
}

}  // namespace

}  // namespace gbs
