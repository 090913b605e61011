// Device building blocks shared by the BFP kernels (sm_103a):
//   - 1D bulk copies global -> shared (the TMA engine's cp.async.bulk) completing
//     on shared-memory mbarriers, with bounded waits;
//   - release/acquire counters for cross-block dataflow, with bounded waits;
//   - the BFP fragment unpack: one 32-bit word of the tile-record layout
//     (include/bfpmoe.h) -> tensor-core A-fragment registers of fp16 lanes
//     (sign << 15 | magnitude), i.e. +-m * 2^-24 as fp16 subnormals, exact;
//   - mma.sync m16n8k16 (fp16 x fp16 -> fp32), one BFP block per instruction;
//   - activation fragments: bf16 rows scaled by a power of two into fp16.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bfp {
namespace dev {

constexpr int kWarp = 32;
constexpr uint32_t kMaskBfp4 = 0x80078007u;
constexpr uint32_t kMaskBfp8 = 0x807F807Fu;
constexpr int kRecCodes = 512;  // code bytes at the start of every tile record (exponents follow)
constexpr int kStatusTimeout = 7;  // stored as -BFP_ETIMEOUT in the status word

struct WaitCfg {
    int64_t iters;     // polling iterations before giving up
    uint64_t nanos;    // and a wall-clock bound from %globaltimer
};

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
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
// Bounded wait for the phase with the given parity; false = gave up (or *abort was raised).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const WaitCfg &w,
                                          const volatile int *abort) {
    if (mbar_test(bar, parity)) return true;
    uint64_t t0 = global_ns();
    for (int64_t i = 1; i < w.iters; ++i) {
        if (mbar_test(bar, parity)) return true;
        if (abort && *abort) return false;
        if (global_ns() - t0 > w.nanos) return false;
    }
    return false;
}

// ------------------------------------------------------- bulk copy (TMA, 1D)
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
// L2 policy for data read once per launch (streamed weights): first to be evicted, so that what is
// reused across launches (the kernel's code, activations, router weights, workspace) stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// L2 policy for small data read by every launch (router rows): last to be evicted.
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Orders this thread's view of global memory (generic proxy) before its later bulk copies
// (async proxy) read it: data other blocks wrote and this thread acquired.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// Orders this thread's earlier shared-memory accesses (generic proxy) before its later bulk copies
// into shared memory (async proxy): needed before a copy overwrites memory the CTA has read.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------ cross-block counters
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Bounded wait until *p >= target; false = gave up.
__device__ __forceinline__ bool wait_counter(const uint32_t *p, uint32_t target, const WaitCfg &w) {
    if (ld_acquire(p) >= target) return true;
    uint64_t t0 = global_ns();
    for (int64_t i = 1; i < w.iters; ++i) {
        __nanosleep(64);
        if (ld_acquire(p) >= target) return true;
        if (global_ns() - t0 > w.nanos) return false;
    }
    return false;
}
// Bounded wait until *p >= target, polling without a pause between loads (each acquire load is an L2 round
// trip already); false = gave up.
__device__ __forceinline__ bool poll_counter(const uint32_t *p, uint32_t target, const WaitCfg &w) {
    if (ld_acquire(p) >= target) return true;
    const uint64_t t0 = global_ns();
    for (int64_t i = 1; i < w.iters; ++i) {
        if (ld_acquire(p) >= target) return true;
        if (global_ns() - t0 > w.nanos) return false;
    }
    return false;
}
// First error wins; the word is cleared only by the host (bfp_workspace_init).
__device__ __forceinline__ void raise_status(uint32_t *status, uint32_t code) { atomicCAS(status, 0u, code); }

// ------------------------------------------------ programmatic dependent launch
// Lets the next kernel on the stream be scheduled (its CTAs start as this grid's CTAs leave).
__device__ __forceinline__ void grid_dep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the kernels this one depends on have finished and their memory is visible (returns at
// once when the launch had no such dependency).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// --------------------------------------------------------- named barriers
__device__ __forceinline__ void bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Barrier that also ORs a predicate over the participating threads (same answer in all of them).
__device__ __forceinline__ bool bar_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------ BFP unpack
__device__ __forceinline__ uint32_t rotr(uint32_t v, int s) { return __funnelshift_r(v, v, s); }

// BFP4 word (one block, 8 codes of this lane) -> A fragment a[0..3].
__device__ __forceinline__ void unpack_bfp4(uint32_t w, uint32_t a[4]) {
    a[0] = w & kMaskBfp4;
    a[1] = rotr(w, 4) & kMaskBfp4;
    a[2] = rotr(w, 8) & kMaskBfp4;
    a[3] = rotr(w, 12) & kMaskBfp4;
}
// BFP8 words (one block: w0 = cols 2t|2t+1, w1 = cols 2t+8|2t+9) -> A fragment.
__device__ __forceinline__ void unpack_bfp8(uint32_t w0, uint32_t w1, uint32_t a[4]) {
    a[0] = w0 & kMaskBfp8;
    a[1] = rotr(w0, 8) & kMaskBfp8;
    a[2] = w1 & kMaskBfp8;
    a[3] = rotr(w1, 8) & kMaskBfp8;
}

// 2^(E-127) for an exponent byte (E = 0 -> 0; the block is all zero then).
__device__ __forceinline__ float exp_scale(uint32_t word, int byte) {
    return __uint_as_float(((word >> (8 * byte)) & 0xFFu) << 23);
}

// D = A(16x16 fp16) * B(16x8 fp16) + C, fp32.
__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A(16x16 bf16) * B(16x8 bf16) + D, fp32.
__device__ __forceinline__ void mma16816_bf16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ----------------------------------------------------- activation helpers
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Power-of-two exponent that brings max|v| into [2^14, 2^15) (0 for an all-zero row),
// clamped to 126 so that 2^shift is an fp32 normal (rows below 2^-112 stay tiny, still exact).
__device__ __forceinline__ int frag_shift(float maxabs) {
    uint32_t e = (__float_as_uint(maxabs) >> 23) & 0xFFu;
    const int s = maxabs > 0.f ? 141 - (int)e : 0;
    return s > 126 ? 126 : s;
}

// 2^e as fp32 for e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }
// x * 2^e for |e| <= 252 in two exact power-of-two steps (exact unless the result leaves the normal range).
__device__ __forceinline__ float mul_pow2(float x, int e) {
    const int e1 = e / 2;
    return (x * pow2f(e1)) * pow2f(e - e1);
}

// Pack two fp32 values already scaled into fp16 range as an fp16x2 word (low = first).
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Activation-fragment layout: for activation group grp (8 rows) and block b, 64 words (256 B)
// holding the mma.sync B fragment of every lane: lane 4g + t owns words {2s, 2s+1} with
// s = (4g + t) ^ frag_swz(b), i.e. row 8*grp + g, cols (2t, 2t+1) and (2t+8, 2t+9) of the block.
// The XOR swizzle permutes lanes within a block (so a warp's fragment read stays one
// conflict-free 256-byte access) and spreads a warp's writes of one row across banks.
__device__ __forceinline__ int frag_swz(int b) { return (b & 7) << 2; }
// Index (in uint2 units) of lane `lane`'s fragment of block b in group grp.
__device__ __forceinline__ int frag_idx(int grp, int b, int lane, int kbp) {
    return (grp * kbp + b) * kWarp + (lane ^ frag_swz(b));
}
// Word address of pair j (cols 2j, 2j+1) of block b of row r.
__device__ __forceinline__ int frag_word(int r, int b, int j, int kbp) {
    return (frag_idx(r >> 3, b, 4 * (r & 7) + (j & 3), kbp) << 1) + (j >> 2);
}

// Deterministic warp sum / max (butterfly; every lane gets the same value).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace dev
}  // namespace bfp
