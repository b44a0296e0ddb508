// Device helpers of libisd: counter-based uniforms, inline PTX for mbarriers,
// bulk copies and programmatic dependent launch, warp reductions, sequence
// lookup.  sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <math.h>

namespace isd {

constexpr int kMaxStride = 32;
constexpr uint64_t kTagAccept = 0, kTagCorrect = 1, kTagBonus = 2, kTagPropose = 3;
constexpr float kLog2e = 1.4426950408889634f;

// Time bounds of the persistent verify kernel's waits, in nanoseconds of the
// global timer: far above any legitimate wait, far below a hang.
constexpr uint64_t kWaitNs = 1000000000ull;       // stage barriers, task flags
constexpr uint64_t kDrainWaitNs = 4000000000ull;  // waiting for other CTAs' work

// Error word bits (workspace): set when a bounded wait gave up.
constexpr int kErrWaitTimeout = 1;

// ---------------------------------------------------------------------------
// Philox4x64-10 — Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3" (SC'11), the 4-word, 64-bit Philox bijection with ten
// rounds and the Weyl key schedule.  All four output words for one counter
// and key.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3, uint64_t k0,
                                              uint64_t k1, uint64_t out[4]) {
    constexpr uint64_t kMul0 = 0xD2E7470EE14C6C93ULL, kMul1 = 0xCA5A826395121157ULL;
    constexpr uint64_t kWeyl0 = 0x9E3779B97F4A7C15ULL, kWeyl1 = 0xBB67AE8584CAA73BULL;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += kWeyl0;
            k1 += kWeyl1;
        }
        const uint64_t hi0 = __umul64hi(kMul0, c0), lo0 = kMul0 * c0;
        const uint64_t hi1 = __umul64hi(kMul1, c2), lo1 = kMul1 * c2;
        const uint64_t n0 = hi1 ^ c1 ^ k0;
        const uint64_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

// Output word 0 alone (the decision uniforms use only it).
__device__ __forceinline__ uint64_t philox4x64_10_word0(uint64_t c0, uint64_t c1, uint64_t c2,
                                                        uint64_t c3, uint64_t k0, uint64_t k1) {
    uint64_t out[4];
    philox4x64_10(c0, c1, c2, c3, k0, k1, out);
    return out[0];
}

// The uniform of one decision: counter (offset, sequence, position, purpose),
// key (seed, 0); top 24 bits of word 0 times 2^-24 (exact in float).
__device__ __forceinline__ float decision_uniform(uint64_t seed, uint64_t offset, uint64_t seq,
                                                  uint64_t pos, uint64_t tag) {
    const uint64_t w = philox4x64_10_word0(offset, seq, pos, tag, seed, 0);
    return (float)(uint32_t)(w >> 40) * (1.0f / 16777216.0f);
}

// ---------------------------------------------------------------------------
// Arithmetic
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(e)/T for T > 0; the same expression everywhere so every kernel derives
// bit-identical scales.
__device__ __forceinline__ float inv_temp_log2e(float T) { return __fdiv_rn(kLog2e, T); }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Argmax partial: larger value wins, equal values go to the lower index.
__device__ __forceinline__ void merge_argmax(float& M, int& I, float m, int i) {
    if (m > M || (m == M && i < I)) {
        M = m;
        I = i;
    }
}

// ---------------------------------------------------------------------------
// Batch layout
// ---------------------------------------------------------------------------
struct SeqInfo {
    int start;
    int len;
    float T;
    bool in_range;  // 0 <= start <= end <= total
    bool ok;        // in range, stride in [1, 32], temperature valid
};

__device__ __forceinline__ bool temperature_ok(float T) {
    return isfinite(T) && (T == 0.0f || T >= 1.17549435e-38f);
}

__device__ __forceinline__ SeqInfo seq_info(const int32_t* offs, const float* temp, int i,
                                            int total) {
    SeqInfo s;
    s.start = __ldg(offs + i);
    const int end = __ldg(offs + i + 1);
    s.len = end - s.start;
    s.T = __ldg(temp + i);
    s.in_range = s.start >= 0 && end <= total && s.len >= 0;
    s.ok = s.in_range && s.len >= 1 && s.len <= kMaxStride && temperature_ok(s.T);
    return s;
}

// Largest i in [0, C) with offs[i] <= r (offsets non-decreasing).
__device__ __forceinline__ int seq_of_position(const int32_t* offs, int C, int r) {
    int lo = 0, hi = C - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(offs + mid) <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Packed arithmetic of sm_100+: two bf16 maxima, two fp32 fused multiply-adds
// or additions per instruction.  A float pair lives in one 64-bit register.
__device__ __forceinline__ uint32_t hmax2_bf16(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f2(uint64_t r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// ---------------------------------------------------------------------------
// Global-memory communication between CTAs of one grid
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// 64-bit words that carry a flag in their high half and 32 bits of data in
// their low half.  An aligned 64-bit access is single-copy atomic, so a
// reader that sees the flag also sees the data written with it: a consumer
// polls the data itself, with no fence and no second load.
__device__ __forceinline__ uint64_t flagged(uint32_t flag, uint32_t data) {
    return (static_cast<uint64_t>(flag) << 32) | data;
}
__device__ __forceinline__ uint64_t ld_volatile_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_volatile_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.volatile.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// Two flagged words at once (each 64-bit half is its own atomic access).
__device__ __forceinline__ void st_volatile_v2u64(uint64_t* p, uint64_t v0, uint64_t v1) {
    asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(v0), "l"(v1) : "memory");
}
__device__ __forceinline__ void ld_volatile_v2u64(const uint64_t* p, uint64_t& v0, uint64_t& v1) {
    asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(v0), "=l"(v1) : "l"(p) : "memory");
}

// Loads that bypass L1 (data written by other CTAs of the running grid).
__device__ __forceinline__ int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }
__device__ __forceinline__ void st_volatile(int* p, int v) { *reinterpret_cast<volatile int*>(p) = v; }
// Device-scope add that publishes this thread's earlier writes and acquires
// the writes published by earlier adds to the same counter.
__device__ __forceinline__ int atomic_add_acq_rel(int* p, int v) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// A release store and an acquire load of a 64-bit word (gpu scope).
__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ---------------------------------------------------------------------------
// Shared-memory barriers, bulk copies, PDL (inline PTX)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// 16-byte global -> shared copy that bypasses L1 (cp.async); many can be in
// flight from one thread, completed together by cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Orders this thread's earlier generic-proxy accesses to shared memory before
// its later async-proxy ones (a bulk copy into a buffer it has read).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking check whether the phase of `parity` has completed.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait with a suspend-time hint: the thread sleeps in hardware until the phase
// completes or about `ns` nanoseconds pass; true if the phase completed.
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
        : "memory");
    return done != 0;
}

// Wait bounded by the global timer; false on timeout.  Sleeps in hardware
// between checks, so a waiting warp issues almost no instructions.
__device__ __forceinline__ bool mbar_wait_ns(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait_for(bar, parity, 1000)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_for(bar, parity, 10000)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// The same copy with an L2 cache-eviction policy (createpolicy below).
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                   uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// L2 policy for lines read once: the first the L2 gives up.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch: wait for the grids this one depends on, and
// allow the dependent grid to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

// ---------------------------------------------------------------------------
// Streaming reductions shared by the verify and propose kernels
// ---------------------------------------------------------------------------
// Tempered softmax weight relative to a reference mc = max * c2.
__device__ __forceinline__ float soft_w(float x, float c2, float mc) { return ex2_approx(__fmaf_rn(x, c2, -mc)); }

// Softmax partials in the mc domain: (mc, s) holds sum exp2(x c2 - mc).
__device__ __forceinline__ void merge_mc(float& M, float& S, float m, float s) {
    if (m == -INFINITY) return;
    if (m > M) {
        S = (M == -INFINITY) ? s : S * ex2_approx(M - m) + s;
        M = m;
    } else {
        S += s * ex2_approx(m - M);
    }
}

// Element j (0 .. 16/E - 1) of a 16-byte vector, as float.
template <int E>
__device__ __forceinline__ float vec_elem(const uint4& v, int j) {
    const uint32_t w = j < (8 / E) ? (j < (4 / E) ? v.x : v.y) : (j < (12 / E) ? v.z : v.w);
    if constexpr (E == 2) return (j & 1) ? bf16hi(w) : bf16lo(w);
    else return __uint_as_float(w);
}

// Largest element of a 16-byte vector.
template <int E>
__device__ __forceinline__ float vec_max(const uint4& v) {
    if constexpr (E == 2) {
        const uint32_t m = hmax2_bf16(hmax2_bf16(v.x, v.y), hmax2_bf16(v.z, v.w));
        return fmaxf(bf16lo(m), bf16hi(m));
    } else {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
}

// Sum of exp2(x c2 - mc) over a 16-byte vector, added to a packed accumulator.
template <int E>
__device__ __forceinline__ void soft_vec(const uint4& v, uint64_t C2, uint64_t NMC, uint64_t& acc) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; j += (E == 2 ? 1 : 2)) {
        float y0, y1;
        if constexpr (E == 2)
            unpack_f2(fma_f2(pack_f2(bf16lo(w[j]), bf16hi(w[j])), C2, NMC), y0, y1);
        else
            unpack_f2(fma_f2(pack_f2(__uint_as_float(w[j]), __uint_as_float(w[j + 1])), C2, NMC), y0, y1);
        acc = add_f2(acc, pack_f2(ex2_approx(y0), ex2_approx(y1)));
    }
}

}  // namespace isd
