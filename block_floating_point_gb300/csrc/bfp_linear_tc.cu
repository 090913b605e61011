// Dense BFP projection on the 5th-generation tensor cores: y[m x n] = x[m x k] . W^T
// for several rows of x (up to 32) in one pass over W, the multi-row decode
// projection (Qwen3.8-27B s27v6 card, "What changed in this release": up to 32
// rows fit one tile row, so a 16-user step still reads every weight once).
//
// The same layer as bfp_linear.cu; what changes is where the block exponent
// goes. The mma.sync path multiplies each 16-value block on its own and folds
// 2^(E-127) into the fp32 sum right after, which costs 4 FMAs per activation
// group and block (16 at 32 rows). Here a cluster of two CTAs owns 128 weight
// rows (the MMA's M), each CTA half of k, streamed in chunks of 128:
//   - a producer warp requests every chunk's records (1D bulk copies, the TMA
//     engine; the first stages before the previous kernel has finished), as
//     many stages ahead as shared memory holds;
//   - eight unpack warps, one per 16-row group, place the BFP codes as fp16
//     values with the exponent folded in: per row and chunk a reference
//     exponent Er = the largest of the chunk's 8 block exponents, each block
//     scaled by 2^(E - Er) (one packed fp16 multiply per pair; exact for blocks
//     within 2^15 of the row's largest in the chunk, and within 2^-16 of the
//     chunk's largest value otherwise), into the K-major core-matrix layout
//     the MMA reads from shared memory;
//   - one thread issues tcgen05.mma (kind::f16, fp32 accumulators in tensor
//     memory, M = 128, N = 16 or 32 activation rows, 8 MMAs of k16 per chunk)
//     against the activation rows, converted once per CTA to fp16 scaled by a
//     power of two per row (as in bfp_linear), and commits to an mbarrier;
//   - four epilogue warps read each chunk's accumulator tile from tensor
//     memory (tcgen05.ld, one row per thread) and add it into fp32 registers
//     scaled by 2^(Er - 117 - mb): one FMA per output per chunk;
//   - at the end the second CTA writes its sums into the first's shared memory
//     (distributed shared memory), which adds them (first + second) and writes y.
// Two operand stages and eight accumulator tiles rotate, so the unpack of a
// chunk overlaps the MMAs of the one before and the read-back lags freely.
// All waits are bounded and report BFP_ETIMEOUT.
#include <cuda_fp16.h>

#include <algorithm>

#include "bfp_launch.h"
#include "bfp_tc.h"

namespace bfp {

using namespace dev;

namespace {

constexpr int kTcRows = 128;    // weight rows per CTA (the MMA's M)
constexpr int kTcK = 128;       // k per chunk
constexpr int kTcGroups = 8;    // 16-row groups per CTA, one unpack warp each
constexpr int kTcEpi0 = 8;      // warps 8-11 read the accumulators back (tensor-memory lanes 32 (w % 4) ..)
constexpr int kTcMmaWarp = 12;  // lane 0 issues the MMAs; the warp owns the tensor-memory allocation
constexpr int kTcProdWarp = 13; // lanes request the record copies
constexpr int kTcWarps = 14;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcRawMax = 16;   // record stages at most (as many as shared memory holds)
constexpr int kTcA = 2;         // operand stages (a stage is free again once its chunk's MMAs are done)
constexpr int kTcD = 8;         // accumulator tiles in tensor memory (the read-back may lag this many chunks)
constexpr int kTcCols = 256;    // tensor-memory columns: kTcD tiles of up to 32
constexpr int kTcXLoads = 10;   // 16-byte activation loads per thread (32 rows x 1024 of k at most)

struct TcArgs {
    const uint8_t *w;
    int64_t n;
    int ng, k, kc, rec, rpc;  // rpc: records of one row group per chunk
    const uint16_t *x;
    int64_t ldx;
    int m, nm;                // rows of x; the MMA's N (16 or 32)
    float *y;
    uint16_t *yb;
    int64_t ldy;
    uint32_t *status;
    int nr;                        // record stages
    int off_a, off_raw, off_misc;  // shared memory: B at 0, then the A stages, the record stages, bookkeeping
    WaitCfg wait;
};

struct TcMisc {
    uint64_t raw_full[kTcRawMax], raw_empty[kTcRawMax];
    uint64_t a_full[kTcA], mma_done[kTcD], d_free[kTcD];
    int eref[kTcD][kTcRows];  // reference exponent of each row of the tile's chunk
    int shift[32];         // power-of-two scale of each activation row
    uint32_t rmax[32];     // max |x| of each row over this CTA's half of k (bf16 bits); pmax: the partner's
    uint32_t pmax[32];
    uint32_t tmem;         // base address of the allocation
    int flags[2];          // [0] abort
};

__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    // shared-memory matrix descriptor: start >> 4, leading (k) and stride (8-row group) byte offsets >> 4, the
    // fixed 0b001 at bits 46-48, no swizzle (K-major core matrices of 8 rows x 16 bytes)
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 consecutive fp32 columns of this thread's tensor-memory lane (the warp's 32 lanes).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t v[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Byte offset of element (row r, k) in a K-major core-matrix layout with kg8 = k / 8 groups per row band.
__device__ __forceinline__ uint32_t cm_off(int r, int k, int kg8) {
    return (uint32_t)((((r >> 3) * kg8 + (k >> 3)) * 8 + (r & 7)) * 16 + (k & 7) * 2);
}
// fp16x2 factor 2^(15 - d) for a block d binades below its row's reference (0 beyond 2^-14: the block's
// values are below 2^-23 of the row's largest there, and flush).
__device__ __forceinline__ uint32_t tc_scale(int d) {
    const uint32_t e = d < 30 ? (uint32_t)(30 - d) : 0u;
    return (e << 10) | (e << 26);
}
// Both CTAs of the cluster meet here (release / acquire on shared memory across the cluster).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Address of the same shared-memory location in the cluster's first CTA.
__device__ __forceinline__ uint32_t map_rank0(uint32_t saddr) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(saddr));
    return r;
}
// ... and in the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_f32x4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}
// Bounded wait for an mbarrier phase that pauses between polls (warps that wait leave the issue slots to
// the unpack warps); false = gave up (or *abort was raised).
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, const WaitCfg &w, const volatile int *abort) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (int64_t i = 1; i < w.iters; ++i) {
        __nanosleep(64);
        if (mbar_test(bar, parity)) return true;
        if (abort && *abort) return false;
        if (global_ns() - t0 > w.nanos) return false;
    }
    return false;
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t s) {
    __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&s));
    return *reinterpret_cast<uint32_t *>(&r);
}

}  // namespace

template <int FMT>
__global__ void __launch_bounds__(kTcThreads, 1) bfp_linear_tc_kernel(const __grid_constant__ TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int CB = FMT == 4 ? 4 : 2;  // blocks per record
    constexpr int MB = FMT == 4 ? 3 : 7;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    // a cluster of two CTAs per 128-row tile, each half of k; the second adds its sums into the first's
    const int tile = blockIdx.x >> 1, half = blockIdx.x & 1;
    const int rg0 = tile * kTcGroups;
    const int ngc = min(kTcGroups, a.ng - rg0);  // row groups of this tile
    const int kh = a.k / 2;                       // this CTA's share of k
    const int kg8 = kh / 8;                       // 8-value groups along it (B's layout)
    const int nch = kh / kTcK;                    // chunks of this CTA
    const int q0 = half * nch;                    // its first chunk of the row
    const int NR = a.nr;
    const uint32_t raw_bytes = (uint32_t)(a.rpc * a.rec);  // one row group's records of a chunk
    uint8_t *const sB = smem;
    uint8_t *const sA = smem + a.off_a;          // [kTcA][128 x 64] fp16, core matrices
    uint8_t *const sRaw = smem + a.off_raw;      // [nr][8 row groups][rpc records]
    TcMisc *ms = reinterpret_cast<TcMisc *>(smem + a.off_misc);
    volatile int *vflags = ms->flags;

    if (tid == 0) {
        for (int i = 0; i < NR; ++i) {
            mbar_init(&ms->raw_full[i], 1);
            mbar_init(&ms->raw_empty[i], kTcGroups);
        }
        for (int b = 0; b < kTcA; ++b) mbar_init(&ms->a_full[b], kTcGroups);
        for (int b = 0; b < kTcD; ++b) {
            mbar_init(&ms->mma_done[b], 1);
            mbar_init(&ms->d_free[b], 4);
        }
        mbar_fence_init();
        ms->flags[0] = ms->flags[1] = 0;
    }
    if (tid < 32) ms->rmax[tid] = 0u;
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&ms->tmem)),
                     "r"(kTcCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem;
    grid_dep_launch_dependents();
    auto fail_wait = [&]() {
        if (lane == 0) {
            vflags[0] = 1;
            raise_status(a.status, kStatusTimeout);
        }
    };
    const uint64_t pol = l2_evict_first();  // the weights are read once
    // producer: chunk q's records of row group j -> stage q % NR (lanes j < ngc, one copy each)
    auto produce = [&](int q) {
        const int st = q % NR;
        if (lane == 0) mbar_arrive_expect_tx(&ms->raw_full[st], raw_bytes * (uint32_t)ngc);
        __syncwarp();
        if (lane < ngc)
            bulk_g2s_hint(sRaw + (size_t)(st * kTcGroups + lane) * raw_bytes,
                          a.w + ((int64_t)(rg0 + lane) * a.kc + (int64_t)(q0 + q) * a.rpc) * a.rec, raw_bytes,
                          &ms->raw_full[st], pol);
        __syncwarp();
    };
    int issued = 0;  // producer: chunks requested
    if (warp == kTcProdWarp)  // the first stages do not depend on the previous kernel
        for (; issued < min(NR, nch); ++issued) produce(issued);
    grid_dep_wait();  // x may come from the previous kernel

    // ---- the activation rows as B: this CTA's half of k, fp16 scaled by 2^shift per row (rows past m zero),
    //      K-major core matrices. All loads in flight at once; each row's maximum over both halves (the two
    //      CTAs exchange theirs), so both scale a row alike.
    uint4 xv[kTcXLoads];
    // piece j of this thread: warp item wi = (tid >> 5) + j * kTcWarps covers rows 8 (wi % nb) + (lane & 7) and
    // 16-byte pieces 4 (wi / nb) + (lane >> 3) (nb = nm / 8 row bands): full sectors on the loads, 128 contiguous
    // bytes per 8 lanes on the stores into the core matrices
    const int nb = a.nm / 8;
    auto piece = [&](int j, int &r, int &kq) {
        const int wi = warp + j * kTcWarps;
        r = 8 * (wi % nb) + (lane & 7);
        kq = 4 * (wi / nb) + (lane >> 3);
    };
#pragma unroll
    for (int j = 0; j < kTcXLoads; ++j) {
        int r, kq;
        piece(j, r, kq);
        xv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (kq < kg8 && r < a.m)
            xv[j] = *reinterpret_cast<const uint4 *>(a.x + (int64_t)r * a.ldx + half * kh + 8 * kq);
    }
#pragma unroll
    for (int j = 0; j < kTcXLoads; ++j) {
        int r, kq;
        piece(j, r, kq);
        uint32_t m2 = __vmaxu2(__vmaxu2(xv[j].x & 0x7FFF7FFFu, xv[j].y & 0x7FFF7FFFu),
                               __vmaxu2(xv[j].z & 0x7FFF7FFFu, xv[j].w & 0x7FFF7FFFu));
        uint32_t mr = max(m2 & 0xFFFFu, m2 >> 16);
        mr = max(mr, __shfl_xor_sync(0xffffffffu, mr, 8));  // the 4 lanes of one row
        mr = max(mr, __shfl_xor_sync(0xffffffffu, mr, 16));
        if (lane < 8 && kq < kg8 && r < a.m) atomicMax(&ms->rmax[r], mr);
    }
    __syncthreads();
    if (tid < a.m) st_cluster_u32(map_rank(smem_addr(&ms->pmax[tid]), (uint32_t)(1 - half)), ms->rmax[tid]);
    cluster_sync();
    if (tid < a.m) ms->shift[tid] = frag_shift(bf16_bits_to_f32(max(ms->rmax[tid], ms->pmax[tid])));
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kTcXLoads; ++j) {
        int r, kq;
        piece(j, r, kq);
        if (kq < kg8) {
            uint4 o = make_uint4(0u, 0u, 0u, 0u);
            if (r < a.m) {
                const float sc = pow2f(ms->shift[r]);
                const uint32_t w4[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
                uint32_t h4[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    h4[q] = pack_half2(bf16_bits_to_f32(w4[q] & 0xFFFFu) * sc, bf16_bits_to_f32(w4[q] >> 16) * sc);
                o = make_uint4(h4[0], h4[1], h4[2], h4[3]);
            }
            *reinterpret_cast<uint4 *>(sB + cm_off(r, 8 * kq, kg8)) = o;
        }
    }
    fence_proxy_async_shared();  // B is read by the tensor cores
    __syncthreads();

    float acc[32];  // epilogue warps: their row's sums over this CTA's chunks
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    if (warp == kTcProdWarp) {
        // ---- producer: the remaining chunks, each into the stage the unpack warps have released
        for (; issued < nch && !vflags[0]; ++issued) {
            const int st = issued % NR;
            if (!__all_sync(0xffffffffu, tc_wait(&ms->raw_empty[st], (uint32_t)(issued / NR - 1) & 1u, a.wait,
                                                   vflags))) {
                fail_wait();
                break;
            }
            __syncwarp();
            produce(issued);
        }
    } else if (warp == kTcMmaWarp) {
        // ---- one thread issues each chunk's 8 MMAs (k16 each): operands from stage q % kTcA, accumulators in
        //      tile q % kTcD
        const uint32_t idesc = (1u << 4) | ((uint32_t)(a.nm >> 3) << 17) | ((uint32_t)(kTcRows >> 4) << 24);
        int done = 0;  // chunks committed
        if (lane == 0) {
            for (int q = 0; q < nch && !vflags[0]; ++q) {
                const int sa = q % kTcA, d = q % kTcD;
                if (!tc_wait(&ms->a_full[sa], (uint32_t)(q / kTcA) & 1u, a.wait, vflags) ||
                    (q >= kTcD && !tc_wait(&ms->d_free[d], (uint32_t)(q / kTcD - 1) & 1u, a.wait, vflags))) {
                    fail_wait();
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_addr(sA + (size_t)sa * kTcRows * kTcK * 2);
                const uint32_t b0 = smem_addr(sB) + (uint32_t)q * (kTcK / 8) * 128;
#pragma unroll
                for (int j = 0; j < kTcK / 16; ++j)
                    tc_mma(tmem + (uint32_t)(d * 32), tc_desc(a0 + j * 256, 128, (kTcK / 8) * 128),
                           tc_desc(b0 + j * 256, 128, (uint32_t)kg8 * 128), idesc, j > 0);
                tc_commit(&ms->mma_done[d]);
                done = q + 1;
            }
            // no MMA may still run when the tensor memory is freed
            if (done > 0) {
                const int q = done - 1;
                const WaitCfg drain{int64_t(1) << 40, 1000000000ull};
                mbar_wait(&ms->mma_done[q % kTcD], (uint32_t)(q / kTcD) & 1u, drain, nullptr);
            }
        }
        __syncwarp();
    } else if (warp < kTcGroups) {
        // ---- unpack warp: row group `warp` of every chunk, codes -> fp16 with the exponent folded in
        const bool live = warp < ngc;
        const int R0 = warp * 16 + g;  // rows R0 and R0 + 8 of the CTA's 128 (lane (g, t4))
        for (int q = 0; q < nch; ++q) {
            const int st = q % NR, sa = q % kTcA, d = q % kTcD;
            bool ok = mbar_wait(&ms->raw_full[st], (uint32_t)(q / NR) & 1u, a.wait, vflags);
            // the stage's previous chunk has been multiplied; the tile's previous chunk read back (its exponents)
            if (ok && q >= kTcA)
                ok = mbar_wait(&ms->mma_done[(q - kTcA) % kTcD], (uint32_t)((q - kTcA) / kTcD) & 1u, a.wait, vflags);
            if (ok && q >= kTcD) ok = mbar_wait(&ms->d_free[d], (uint32_t)(q / kTcD - 1) & 1u, a.wait, vflags);
            if (!__all_sync(0xffffffffu, ok)) {
                fail_wait();
                break;
            }
            __syncwarp();
            uint8_t *dA = sA + (size_t)sa * kTcRows * kTcK * 2;
            if (live) {
                const uint8_t *rp = sRaw + (size_t)(st * kTcGroups + warp) * raw_bytes;
                // this lane's rows' exponents: per record, blocks in order, (row g, row g + 8) byte pairs
                constexpr int RPCM = kTcK / 32;  // most records of a row group per chunk (BFP8)
                uint32_t ew[RPCM][2];
                uint4 wq[RPCM];
#pragma unroll
                for (int r = 0; r < RPCM; ++r) {
                    if (r < a.rpc) {
                        wq[r] = *reinterpret_cast<const uint4 *>(rp + (size_t)r * a.rec + 16 * lane);
                        if constexpr (CB == 4) {
                            const uint2 e2 = *reinterpret_cast<const uint2 *>(rp + (size_t)r * a.rec + 512 + 8 * g);
                            ew[r][0] = e2.x;
                            ew[r][1] = e2.y;
                        } else {
                            ew[r][0] = *reinterpret_cast<const uint32_t *>(rp + (size_t)r * a.rec + 512 + 4 * g);
                            ew[r][1] = 0u;
                        }
                    } else {
                        wq[r] = make_uint4(0u, 0u, 0u, 0u);
                        ew[r][0] = ew[r][1] = 0u;
                    }
                }
                // exponent of (row g or g + 8, chunk block kb), kb = 0 .. 3
                auto ex = [&](int kb, int hi) -> int {
                    const int r = kb / CB, bb = kb % CB;
                    return (int)((ew[r][bb >> 1] >> (8 * (2 * (bb & 1) + hi))) & 0xFFu);
                };
                int er0 = 0, er1 = 0;
#pragma unroll
                for (int kb = 0; kb < kTcK / 16; ++kb) {
                    er0 = max(er0, ex(kb, 0));
                    er1 = max(er1, ex(kb, 1));
                }
#pragma unroll
                for (int kb = 0; kb < kTcK / 16; ++kb) {
                    const int r = kb / CB, bb = kb % CB;
                    uint32_t av[4];
                    if constexpr (FMT == 4) {
                        const uint32_t wsel = bb == 0 ? wq[r].x : bb == 1 ? wq[r].y : bb == 2 ? wq[r].z : wq[r].w;
                        unpack_bfp4(wsel, av);
                    } else {
                        if (bb == 0)
                            unpack_bfp8(wq[r].x, wq[r].y, av);
                        else
                            unpack_bfp8(wq[r].z, wq[r].w, av);
                    }
                    const uint32_t s0 = tc_scale(er0 - ex(kb, 0)), s1 = tc_scale(er1 - ex(kb, 1));
                    const int kk = kb * 16 + 2 * t4;
                    *reinterpret_cast<uint32_t *>(dA + cm_off(R0, kk, kTcK / 8)) = hmul2_bits(av[0], s0);
                    *reinterpret_cast<uint32_t *>(dA + cm_off(R0 + 8, kk, kTcK / 8)) = hmul2_bits(av[1], s1);
                    *reinterpret_cast<uint32_t *>(dA + cm_off(R0, kk + 8, kTcK / 8)) = hmul2_bits(av[2], s0);
                    *reinterpret_cast<uint32_t *>(dA + cm_off(R0 + 8, kk + 8, kTcK / 8)) = hmul2_bits(av[3], s1);
                }
                if (t4 == 0) {
                    ms->eref[d][R0] = er0;
                    ms->eref[d][R0 + 8] = er1;
                }
            } else {
                // rows past the matrix: zero operands
                for (int i = lane; i < 16 * kTcK / 8; i += 32)
                    *reinterpret_cast<uint4 *>(dA + cm_off(warp * 16 + i / (kTcK / 8), 8 * (i % (kTcK / 8)), kTcK / 8)) =
                        make_uint4(0u, 0u, 0u, 0u);
                if (lane < 16) ms->eref[d][warp * 16 + lane] = 0;
            }
            fence_proxy_async_shared();  // the operands are read by the tensor cores
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ms->a_full[sa]);
                mbar_arrive(&ms->raw_empty[st]);
            }
        }
    } else if (warp >= kTcEpi0 && warp < kTcEpi0 + 4) {
        // ---- epilogue warp: tensor-memory lanes 32 e .. 32 e + 31 = rows of the CTA; each chunk's tile added
        //      into registers scaled by 2^(Er - 117 - mb)
        const int e = warp & 3;
        const int row = 32 * e + lane;
        for (int q = 0; q < nch; ++q) {
            const int d = q % kTcD;
            if (!__all_sync(0xffffffffu, tc_wait(&ms->mma_done[d], (uint32_t)(q / kTcD) & 1u, a.wait, vflags))) {
                fail_wait();
                break;
            }
            __syncwarp();
            tc_fence_after();
            uint32_t v[32];
            tc_ld32(tmem + ((uint32_t)(32 * e) << 16) + (uint32_t)(d * 32), v);
            const int ee = min(max(ms->eref[d][row] - 117 - MB, -126), 127);
            const float f = pow2f(ee);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < a.nm) acc[j] = fmaf(__uint_as_float(v[j]), f, acc[j]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms->d_free[d]);
        }
    }
    // ---- the pair's sums meet in the first CTA (its operand stages are free by now): the second writes its
    //      rows' sums into them, then the first adds (first + second, fixed order) and writes y
    tc_fence_before();
    cluster_sync();
    float *const recv = reinterpret_cast<float *>(sA);  // [128 rows][32]
    if (half == 1 && warp >= kTcEpi0 && warp < kTcEpi0 + 4) {
        const int row = 32 * (warp & 3) + lane;
        const uint32_t dst = map_rank0(smem_addr(recv + row * 32));
#pragma unroll
        for (int j = 0; j < 32; j += 4) st_cluster_f32x4(dst + 4 * j, acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
    }
    cluster_sync();
    if (half == 0 && warp >= kTcEpi0 && warp < kTcEpi0 + 4) {
        const int row = 32 * (warp & 3) + lane;
        const int64_t nrow = (int64_t)tile * kTcRows + row;
        if (!vflags[0] && nrow < a.n) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j < a.m) {
                    const float v = mul_pow2(acc[j] + recv[row * 32 + j], -ms->shift[j]);
                    if (a.y) a.y[(int64_t)j * a.ldy + nrow] = v;
                    if (a.yb) a.yb[(int64_t)j * a.ldy + nrow] = f32_to_bf16_bits(v);
                }
            }
        }
    }
    // every copy requested has landed before the CTA leaves (the producer's stages)
    if (warp == kTcProdWarp && lane == 0) {
        const WaitCfg drain{int64_t(1) << 40, 1000000000ull};
        for (int q = max(0, issued - NR); q < issued; ++q)
            mbar_wait(&ms->raw_full[q % NR], (uint32_t)(q / NR) & 1u, drain, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTcMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcCols));
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
template <int FMT>
static int launch_tc_t(const TcArgs &a, int ncta, size_t smem, cudaStream_t st) {
    auto kern = bfp_linear_tc_kernel<FMT>;
    int rc = set_smem_attr(reinterpret_cast<const void *>(kern), (int)smem, "cudaFuncSetAttribute(bfp_linear_tc)");
    if (rc) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ncta);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;  // the two halves of a tile, co-scheduled
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return cuda_fail(e, "launch bfp_linear_tc");
    return BFP_OK;
}

int linear_tc_launch(const Geometry &g, const uint8_t *w, const uint16_t *x, int m, int64_t ldx, float *y,
                     uint16_t *y_bf16, int64_t ldy, uint32_t *status, cudaStream_t st) {
    if (m < 1 || m > 32 || g.k % (2 * kTcK) != 0) return kTcNotApplicable;
    {
        // the activation pieces: (nm / 8) row bands x (k / 2 / 32) groups of four 16-byte pieces, one per warp item
        const int64_t items = (int64_t)((m > 16 ? 32 : 16) / 8) * ((g.k / 2) / 32);
        if (items > (int64_t)kTcXLoads * kTcWarps) return kTcNotApplicable;
    }
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    TcArgs a;
    a.nm = m > 16 ? 32 : 16;
    const size_t sb = align_up((size_t)a.nm * (g.k / 2) * 2, 1024);  // this CTA's half of the activation rows
    const int rpc = kTcK / (16 * g.cb);
    a.off_a = (int)sb;
    a.off_raw = (int)(sb + kTcA * (size_t)kTcRows * kTcK * 2);
    const size_t stage = (size_t)kTcGroups * rpc * g.rec;
    // as many record stages as shared memory holds (bytes in flight per SM), at least 3
    const int64_t room = (int64_t)di.smem_optin - 128 - (int64_t)align_up(sizeof(TcMisc), 16) - (int64_t)a.off_raw;
    a.nr = (int)std::min<int64_t>(kTcRawMax, room / (int64_t)stage);
    if (a.nr < 3) return kTcNotApplicable;
    a.off_misc = (int)align_up((size_t)a.off_raw + (size_t)a.nr * stage, 16);
    const size_t smem = align_up((size_t)a.off_misc + sizeof(TcMisc), 128);
    if ((int64_t)smem > (int64_t)di.smem_optin) return kTcNotApplicable;
    a.w = w;
    a.n = g.n;
    a.ng = (int)g.ng;
    a.k = (int)g.k;
    a.kc = (int)g.kc;
    a.rec = g.rec;
    a.rpc = rpc;
    a.x = x;
    a.ldx = ldx;
    a.m = m;
    a.y = y;
    a.yb = y_bf16;
    a.ldy = ldy;
    a.status = status;
    a.wait = WaitCfg{kDefaultWaitIters, kDefaultWaitNanos};
    const int ncta = 2 * (int)((g.ng + kTcGroups - 1) / kTcGroups);  // two CTAs (one cluster) per tile
    return g.fmt == BFP_FMT_BFP4 ? launch_tc_t<4>(a, ncta, smem, st) : launch_tc_t<8>(a, ncta, smem, st);
}

static int g_linear_path = 0;
int linear_path() { return g_linear_path; }

}  // namespace bfp

extern "C" int bfp_set_linear_path(int mode) {
    if (mode < 0 || mode > 2) return bfp::fail(BFP_EINVAL, "linear path must be 0, 1 or 2");
    bfp::g_linear_path = mode;
    return BFP_OK;
}
