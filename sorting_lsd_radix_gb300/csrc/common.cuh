// Shared device helpers of the gbsort CUDA library: key codes, inline PTX
// wrappers (mbarrier, bulk async copy, relaxed global accesses) and the
// layout of the work buffer's header.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace gbs {

// ---------------------------------------------------------------------------
// Key kinds and order-preserving codes
// ---------------------------------------------------------------------------
//
// Unsigned keys are their own code.  Signed keys flip the sign bit
// ("GPU基数排序：从CUB工程实现到性能调优", §5.2).  Floats invert every bit
// when the sign is set and only the sign bit otherwise (kwkr.cn notes on
// bitonic vs LSD radix sort §3.3; "GPU基数排序" §5.3, which extends the same
// map to doubles), so -0.0 gets the code just below +0.0.  Descending sorts
// the complemented code ascending.

enum KeyKind : int { KIND_U32 = 0, KIND_I32 = 1, KIND_F32 = 2, KIND_U64 = 3, KIND_I64 = 4, KIND_F64 = 5 };

// The same codes without a switch on the kind: code(x) = x ^ ((x >>s (w-1)) & a) ^ b
// for key width w, with a = all bits but the sign for floats (else 0) and
// b = the sign bit for signed and float kinds (else 0), complemented when
// descending.
struct CodeConsts {
    uint32_t a32, b32;
    uint64_t a64, b64;
};
inline CodeConsts code_consts(int kind, bool descending) {
    const bool fl = kind == KIND_F32 || kind == KIND_F64;
    const bool sg = fl || kind == KIND_I32 || kind == KIND_I64;
    CodeConsts c;
    c.a32 = fl ? 0x7FFFFFFFu : 0u;
    c.b32 = (sg ? 0x80000000u : 0u) ^ (descending ? 0xFFFFFFFFu : 0u);
    c.a64 = fl ? 0x7FFFFFFFFFFFFFFFull : 0ull;
    c.b64 = (sg ? 0x8000000000000000ull : 0ull) ^ (descending ? ~0ull : 0ull);
    return c;
}

__host__ __device__ __forceinline__ uint32_t encode32(uint32_t x, int kind, uint32_t flip) {
    uint32_t t;
    if (kind == KIND_F32) {
        uint32_t m = (uint32_t)((int32_t)x >> 31) | 0x80000000u;  // all ones if negative, else sign bit
        t = x ^ m;
    } else if (kind == KIND_I32) {
        t = x ^ 0x80000000u;
    } else {
        t = x;
    }
    return t ^ flip;
}

__host__ __device__ __forceinline__ uint32_t decode32(uint32_t t, int kind, uint32_t flip) {
    t ^= flip;
    if (kind == KIND_F32) {
        // top bit set: came from a non-negative float, only the sign bit was flipped
        uint32_t m = (uint32_t)(~((int32_t)t >> 31)) | 0x80000000u;
        return t ^ m;
    }
    if (kind == KIND_I32) return t ^ 0x80000000u;
    return t;
}

__host__ __device__ __forceinline__ uint64_t encode64(uint64_t x, int kind, uint64_t flip) {
    uint64_t t;
    if (kind == KIND_F64)
        t = x ^ ((uint64_t)((int64_t)x >> 63) | 0x8000000000000000ull);  // all ones if negative, else sign bit
    else if (kind == KIND_I64)
        t = x ^ 0x8000000000000000ull;
    else
        t = x;
    return t ^ flip;
}
__host__ __device__ __forceinline__ uint64_t decode64(uint64_t t, int kind, uint64_t flip) {
    t ^= flip;
    if (kind == KIND_F64) return t ^ ((uint64_t)(~((int64_t)t >> 63)) | 0x8000000000000000ull);
    if (kind == KIND_I64) return t ^ 0x8000000000000000ull;
    return t;
}

template <typename K> struct KeyCodec;
template <> struct KeyCodec<uint32_t> {
    static __device__ __forceinline__ uint32_t enc(uint32_t x, int kind, uint32_t flip) { return encode32(x, kind, flip); }
    static __device__ __forceinline__ uint32_t dec(uint32_t t, int kind, uint32_t flip) { return decode32(t, kind, flip); }
    static constexpr uint32_t ALL_ONES = 0xFFFFFFFFu;
};
template <> struct KeyCodec<uint64_t> {
    static __device__ __forceinline__ uint64_t enc(uint64_t x, int kind, uint64_t flip) { return encode64(x, kind, flip); }
    static __device__ __forceinline__ uint64_t dec(uint64_t t, int kind, uint64_t flip) { return decode64(t, kind, flip); }
    static constexpr uint64_t ALL_ONES = ~0ull;
};

// Digit of a code: (t >> shift) & mask with mask = 2^bits - 1, bits <= 8.
__device__ __forceinline__ uint32_t digit_of(uint32_t t, int shift, uint32_t mask) {
    return (t >> shift) & mask;
}
__device__ __forceinline__ uint32_t digit_of(uint64_t t, int shift, uint32_t mask) {
    return (uint32_t)(t >> shift) & mask;
}

// ---------------------------------------------------------------------------
// Work-buffer header (first 256 bytes of d_temp, zeroed at the start of
// every radix call).
// ---------------------------------------------------------------------------

constexpr int MAX_PASSES = 8;
constexpr uint32_t ERR_LOOKBACK_TIMEOUT = 1;
constexpr uint32_t ERR_COPY_TIMEOUT = 2;

struct alignas(256) Header {
    uint32_t error;             // 0 = ok, else ERR_* (first error wins)
    uint32_t error_detail;      // pass * 2^24 + tile of the first error
    uint32_t hist_blocks_done;  // upfront-histogram CTAs finished (last-CTA plan)
    uint32_t num_active;        // passes whose digit is not constant
    uint32_t active_mask;       // bit p set: pass p runs
    uint32_t ordinal[MAX_PASSES];       // rank of pass p among active passes
    uint32_t tile_counter[MAX_PASSES];  // tile tickets of pass p (11-bit prototype; the 8-bit passes use block indices)
};
static_assert(sizeof(Header) == 256, "header must be 256 bytes");

// Tile status word of the chained scan: a 3-bit state in the top bits, a
// count below.  Active pass with ordinal k uses states AGG = 1 + 2(k mod 3)
// (tile count only) and INC = 2 + 2(k mod 3) (inclusive prefix).
// Consecutive active passes therefore never mistake each other's words for
// their own, so the status array is zeroed once per call and then reused by
// every pass.  32-bit words (29-bit counts) serve sorts of fewer than 2^29
// keys; larger sorts use 64-bit words (61-bit counts), which hold any
// prefix of up to 2^32 - 1 keys.
template <typename SW> struct StatusWord;
template <> struct StatusWord<uint32_t> {
    static constexpr int COUNT_BITS = 29;
    static constexpr uint32_t COUNT_MASK = (1u << COUNT_BITS) - 1;
    static constexpr uint64_t MAX_KEYS = COUNT_MASK;  // largest prefix a word holds
};
template <> struct StatusWord<uint64_t> {
    static constexpr int COUNT_BITS = 61;
    static constexpr uint64_t COUNT_MASK = (1ull << COUNT_BITS) - 1;
    static constexpr uint64_t MAX_KEYS = 0xFFFFFFFFull;  // keys are counted in 32 bits elsewhere
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Ballot of "(x & m) != 0" over a fully active warp, as one and/setp/vote
// sequence.  Measured on sm_103a, __ballot_sync on the same comparison issues
// about 3.7 integer-pipe instructions per ballot and this form about 1.4.
#ifndef GBS_BALLOT_VOLATILE
#define GBS_BALLOT_VOLATILE 1
#endif
__device__ __forceinline__ uint32_t ballot_bits(uint32_t x, uint32_t m) {
    uint32_t r;
#if GBS_BALLOT_VOLATILE
    asm volatile(
#else
    asm(
#endif
        "{\n\t.reg .pred p;\n\t.reg .b32 t;\n\tand.b32 t, %1, %2;\n\tsetp.ne.u32 p, t, 0;\n\t"
        "vote.sync.ballot.b32 %0, p, 0xffffffff;\n\t}"
        : "=r"(r)
        : "r"(x), "r"(m));
    return r;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    // make the initialised barrier visible to the async (bulk-copy) proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bulk (non-tensor) async copy global -> this CTA's shared memory; completion
// is signalled on `bar` as `bytes` transaction bytes.  Both addresses must be
// 16-byte aligned and bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Hint: fetch global bytes [src, src + bytes) into L2 (no completion signal,
// nothing written).  src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Records the first device-side error in the header.
__device__ __forceinline__ void record_error(Header *h, uint32_t code, uint32_t detail) {
    if (atomicCAS(&h->error, 0u, code) == 0u) atomicExch(&h->error_detail, detail);
}

}  // namespace gbs
