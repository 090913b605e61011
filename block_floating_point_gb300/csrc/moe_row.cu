// One-row MoE decode layer: moe_decode_layer (and the layers of moe_stack_decode)
// with m = 1, the single-sequence decode step. One launch runs one layer, or up
// to 48 layers of one shape in order (the decode stack), the residual row
// passing from layer to layer inside the launch.
//
// What it computes is the layer of moe_layer.cu (Qwen3.6-35B-A3B card, "Fused
// decode kernels": MoE decode of one row through device top-k routing and
// batched expert streams; 256 experts, top-8 plus a shared expert:
// qwen3.6-a3b-blackhole page):
//     l = Wr x (+bias) -> softmax -> top-k -> renormalise -> for each selected
//     expert  D (silu(G x) * (U x))  combined with the routing weights, plus
//     sigmoid(g . x) * shared(x).
//
// With one row the step is short (top_k + 1 experts, 16 MB at the full size:
// about 2.3 us of HBM time), so this kernel is built around the length of the
// dependent chain rather than around throughput:
//   - every CTA's work is fixed at launch. One row always selects exactly
//     top_k experts, so the list [shared f-tiles, f-tiles of slot 0, slot 1,
//     ...] (an f-tile: 16 ffn rows of gate and up over the whole hidden
//     dimension) and each CTA's range of it (whole f-tiles, split evenly) are
//     known before the router runs; only which expert fills a slot is not;
//   - each CTA owns whole row groups of the output (16 hidden rows) for the
//     down projections of every selected expert and sums them itself in slot
//     order: no combine pass, no third grid-wide wait;
//   - what does not depend on the previous kernel or on the routing (the CTA's
//     router rows, its shared-expert f-tiles and shared down rows) is requested
//     before the kernel waits for the previous kernel to finish;
//   - everything a CTA reads (about 115 KB at the full size) fits in its shared
//     memory: each slot's f-tiles are requested (1D bulk copies, the TMA
//     engine) in the top-k round that decides the slot, the down rows once the
//     gate/up bytes are in;
//   - two grid-wide exchanges per layer: the router logits (then one warp of
//     every CTA takes the top-k) and h; a third between layers (the residual
//     row), all through (epoch, value) words, no counters.
// Contractions run on the tensor cores (mma.sync m16n8k16, BFP codes placed so
// that a rotate and a mask give exact fp16 values, one BFP block per MMA, its
// 2^(E-127) folded into the fp32 sum right after); with one row only column 0
// of the activation operand is used (column 4 carries the low half of h in the
// down projection). All waits are bounded and report BFP_ETIMEOUT.
#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "bfp_launch.h"
#include "bfp_trace.h"
#include "moe_common.cuh"

namespace bfp {

using namespace dev;

constexpr int kRowWarps = 16;
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kRowPieces = 8;    // most partial tiles per warp (one per gate/up unit; one per run of down records)
constexpr int kRowMaxRg = 4;     // most output row groups per CTA
constexpr int kRowMaxUnits = 32; // most f-tile units per CTA (one thread per (unit, row) sums their pieces)
constexpr int kRowMaxRouterRows = 4;  // most router rows (with the shared-gate row) per CTA
constexpr int kRowRouterRegs = 4;     // 16-byte router vectors held by each thread

// One layer's weights (every layer of a launch has the same shape).
struct RowLayer {
    const uint16_t *router;
    const float *rbias;
    const uint16_t *sgate;
    const uint8_t *gu, *dn, *sgu, *sdn;
};
constexpr int kRowStackMax = 48;  // layers one launch runs (a longer stack takes several launches)

struct RowArgs {
    int H, E, F, K, Fs, ncta, nl;
    const uint16_t *x;
    int norm;
    float eps;
    int64_t gu_stride, dn_stride;
    float *y;
    uint16_t *h_out;
    int32_t *topk_idx;
    float *topk_w;
    uint32_t *status;
    // exchange between CTAs, no counters: every value goes out as one 64-bit word (epoch << 32 | fp32 bits),
    // so a reader that sees this launch's epoch in a word has that word's value; epoch: this launch's
    // number minus one (read at the start, advanced by CTA 0 once every CTA has published its logits)
    uint32_t *epoch;
    unsigned long long *lgw;  // [CTA][lsb]: every CTA's mailbox of router logits, the shared-gate logit last
    int lsb;                  // words per mailbox
    unsigned long long *hw;   // [K + 1][Fmax] h of each slot (slot K: the shared expert)
    unsigned long long *xw;   // [H / 2] the residual row after a layer (two bf16 per word), for the next layer
    int rec, kc_h, kc_f, kc_fs, nft, nft_s, ng_d, Fmax, kbf;
    int off_stage, off_xc, off_hc, off_p1, off_p2, off_misc;
    WaitCfg wait, wait_data;
    int16_t ub[kRowMaxCta + 1];  // CTA c takes f-tile units [ub[c], ub[c + 1]) of the list
    RowLayer layer[kRowStackMax];  // layers 0 .. nl - 1, applied in order (topk_idx: K entries per layer)
};

struct RowMisc {
    uint64_t bar_x, bar_p2sh, bar_p2rt;
    uint64_t bar_u[kRowMaxUnits];  // one per f-tile unit of the CTA (its gate and up row groups, one copy)
    int shift_s[kMaxTopK + 1];  // power-of-two scale of each slot's h fragments
    float wsl[kMaxTopK + 1];    // routing weight of each slot; slot K: the shared gate sigmoid(g . x)
    int esl[kMaxTopK];          // expert of each slot
    int p2g0[kRowWarps];        // first (row group, slot) group in each warp's down range
    float red[kRowWarps][4];    // per-warp partial logits (up to 4 router rows)
    alignas(16) float sst[kRowWarps];     // per-warp partial sums of squares of the row
    alignas(16) uint32_t smx[kRowWarps];  // per-warp maxima of |x| (bf16 bits)
    float lgv[4];               // the CTA's logits of the current pass
    int flags[4];               // [0] abort
    uint32_t ep;                // the epoch word at the start of the launch
    int slot_ready[kMaxTopK + 1];  // the slot's h operands are in shared memory
};

__device__ __forceinline__ unsigned long long tag_word(uint32_t tag, float v) {
    return ((unsigned long long)tag << 32) | __float_as_uint(v);
}
__device__ __forceinline__ uint32_t word_tag(unsigned long long w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ float word_value(unsigned long long w) { return __uint_as_float((uint32_t)w); }
// Loads of words another CTA writes, for polling loops: strong (relaxed, gpu scope) loads, so they are
// served by L2 and never merged with or hoisted out of the loop's earlier iterations; each 64-bit element
// is read whole.
__device__ __forceinline__ unsigned long long ld_word(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ ulonglong2 ld_words2(const unsigned long long *p) {
    ulonglong2 v;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}
// The matching store (relaxed, gpu scope).
__device__ __forceinline__ void st_word(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Compact one-row operands (the B side of m16n8k16, only a few columns used). Per block, the x row has
// kXEnt uint2: the fragment pairs of lanes (0, t), t = 0..3 (column 0), then a zero pair; h has kHEnt:
// hi pairs of lanes (0, t) (column 0), lo pairs of lanes (4, t) (column 4), a zero pair. Lane (g, t)
// reads entry xsel / hsel: no branch, and lanes of unused columns read the zero pair.
constexpr int kXEnt = 5;
constexpr int kHEnt = 9;

// Group index (row group j, slot s) = j * (K + 1) + s of down item i; items run (row group, slot, record)
// with IPR = K * kc_f + kc_fs items per row group (slot K, the shared expert, last).
__device__ __forceinline__ int row_p2_group(int i, int IPR, int K, int kc_f) {
    const int j = i / IPR, rem = i - j * IPR;
    return j * (K + 1) + (rem < K * kc_f ? rem / kc_f : K);
}

// acc[r][0] / acc[r][1] (rows g and g + 8 of the record's 16, the columns the operand fills) += sum over the
// record's blocks of 2^(E-127) * (A_r . B). B of block b for this lane: bop[b * NE + sel].
template <int FMT, int NREC, int NE>
__device__ __forceinline__ void row_mma(const uint8_t *const recs[NREC], const uint2 *bop, int sel, int lane,
                                        float acc[NREC][2]) {
    constexpr int CB = FMT == 4 ? 4 : 2;
    const int g = lane >> 2;
    uint4 wq[NREC];
    uint32_t ew[NREC][2];
#pragma unroll
    for (int r = 0; r < NREC; ++r) {
        wq[r] = *reinterpret_cast<const uint4 *>(recs[r] + 16 * lane);
        // exponent bytes of rows g (even) and g + 8 (odd), blocks in order: 2 * CB bytes at 2 * CB * g
        if constexpr (CB == 4) {
            const uint2 e = *reinterpret_cast<const uint2 *>(recs[r] + kRecCodes + 8 * g);
            ew[r][0] = e.x;
            ew[r][1] = e.y;
        } else {
            ew[r][0] = *reinterpret_cast<const uint32_t *>(recs[r] + kRecCodes + 4 * g);
            ew[r][1] = 0u;
        }
    }
#pragma unroll
    for (int b = 0; b < CB; ++b) {
        const uint2 bx = bop[b * NE + sel];
#pragma unroll
        for (int r = 0; r < NREC; ++r) {
            uint32_t av[4];
            if constexpr (FMT == 4) {
                const uint32_t wsel = b == 0 ? wq[r].x : b == 1 ? wq[r].y : b == 2 ? wq[r].z : wq[r].w;
                unpack_bfp4(wsel, av);
            } else {
                if (b == 0)
                    unpack_bfp8(wq[r].x, wq[r].y, av);
                else
                    unpack_bfp8(wq[r].z, wq[r].w, av);
            }
            const uint32_t ewd = ew[r][b >> 1];
            const float s0 = exp_scale(ewd, 2 * (b & 1)), s1 = exp_scale(ewd, 2 * (b & 1) + 1);
            float cc[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(cc, av, bx.x, bx.y);
            acc[r][0] = fmaf(s0, cc[0], acc[r][0]);
            acc[r][1] = fmaf(s1, cc[2], acc[r][1]);
        }
    }
}

// MULTI: several layers per launch (a.nl); otherwise exactly one (the loop and the exchange of the residual row
// compile away).
template <int FMT, bool MULTI>
__global__ void __launch_bounds__(kRowThreads, 1) moe_row_kernel(const __grid_constant__ RowArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int CB = FMT == 4 ? 4 : 2;
    constexpr int MB = FMT == 4 ? 3 : 7;
    constexpr int NW = kRowWarps;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, c = blockIdx.x;
    const int g = lane >> 2, t4 = lane & 3;
    RowMisc *ms = reinterpret_cast<RowMisc *>(smem + a.off_misc);
    volatile int *vflags = ms->flags;
#ifdef BFP_TRACE
    // trace builds: thread 0 stamps %globaltimer (slot i) and its SM cycle count (slot 64 + i); lane 0 of every
    // warp can stamp its own slot
    unsigned long long *const trp = g_bfp_trace ? g_bfp_trace + (size_t)blockIdx.x * BFP_TRACE_SLOTS : nullptr;
#define STAMP(i)                                                     \
    do {                                                             \
        if (trp && threadIdx.x == 0) {                               \
            trp[(i)] = global_ns();                                  \
            trp[64 + (i)] = (unsigned long long)clock64();           \
        }                                                            \
        __syncwarp();                                                \
    } while (0)
#define WSTAMP(base)                                                            \
    do {                                                                        \
        if (trp && (threadIdx.x & 31) == 0) trp[(base) + (threadIdx.x >> 5)] = global_ns(); \
        __syncwarp();                                                           \
    } while (0)
#define CSTAMP(i)                                                         \
    do {                                                                  \
        if (trp && threadIdx.x == 0) trp[(i)] = (unsigned long long)clock64(); \
        __syncwarp();                                                     \
    } while (0)
#else
#define CSTAMP(i) \
    do {          \
    } while (0)
#define STAMP(i) \
    do {         \
    } while (0)
#define WSTAMP(base) \
    do {             \
    } while (0)
#endif
    STAMP(0);

    // ---- this CTA's share (all fixed at launch)
    const int u0 = a.ub[c], nu = a.ub[c + 1] - u0;  // f-tile units [u0, u0 + nu) of the list
    const int64_t ubytes = 2 * (int64_t)a.kc_h * a.rec;  // one unit: its gate and up row groups, as stored
    uint8_t *const w1 = smem;                             // the units, one after another
    uint8_t *const w2 = smem + nu * ubytes;               // then the down items (row group, slot, record)
    uint16_t *const xs = reinterpret_cast<uint16_t *>(smem + a.off_stage);  // activation row [H] bf16
    uint2 *const xc = reinterpret_cast<uint2 *>(smem + a.off_xc);           // [kc_h * CB blocks][kXEnt]
    uint2 *const hc = reinterpret_cast<uint2 *>(smem + a.off_hc);           // [slot][kbf blocks][kHEnt]
    float *const p1p = reinterpret_cast<float *>(smem + a.off_p1);          // [warp][piece][gate, up][16]
    float *const p2p = reinterpret_cast<float *>(smem + a.off_p2);          // [warp][piece][16]
    // gate/up: every warp takes the same slice [k0w, k1w) of chunks (one gate record and the up record of the
    // same k) of every unit, so that a unit is computed by all warps at once as soon as it lands
    const int k0w = warp * a.kc_h / NW, k1w = (warp + 1) * a.kc_h / NW;
    const int nrg = c < a.ng_d ? (a.ng_d - c + a.ncta - 1) / a.ncta : 0;  // row groups c, c + ncta, ...
    const int IPR = a.K * a.kc_f + a.kc_fs;
    const int I2 = nrg * IPR;
    const int it0 = warp * I2 / NW, it1 = (warp + 1) * I2 / NW;
    const int E1 = a.E + 1;
    const int rr0 = router_row_start(c, E1, a.ncta), rr1 = router_row_start(c + 1, E1, a.ncta);
    const int re = min(rr1, a.E);
    const int xsel = g == 0 ? t4 : 4;                        // compact x operand entry of this lane
    const int hsel = g == 0 ? t4 : (g == 4 ? 4 + t4 : 8);    // compact h operand entry of this lane

    if (tid == 0) {
        mbar_init(&ms->bar_x, 1);
        mbar_init(&ms->bar_p2sh, 1);
        mbar_init(&ms->bar_p2rt, 1);
        for (int j = 0; j < nu; ++j) mbar_init(&ms->bar_u[j], 1);
        mbar_fence_init();
        for (int i = 0; i < 4; ++i) ms->flags[i] = 0;
        for (int i = 0; i <= kMaxTopK; ++i) ms->slot_ready[i] = 0;
    }
    if (lane == 0)  // where each warp's down range starts (read by the combine, which avoids divisions)
        ms->p2g0[warp] = it1 > it0 ? row_p2_group(it0, IPR, a.K, a.kc_f) : 0;
    __syncthreads();
    // dependent launch: the next kernel may take the SMs as this one's CTAs leave
    grid_dep_launch_dependents();

    bool bad = false;
    uint32_t armed_u = 0u;     // thread 0: units whose copy it issued (this layer)
    bool armed_p2rt = false;   // thread 0: the routed down rows issued (this layer)
    bool armed_p2sh = false;   // thread 32: the shared down rows issued (this layer)
    bool routed = false;       // warp 0: the top-k is done and the routed f-tile units are requested
    uint32_t par = 0u;         // phase parity of this layer's copies (one phase per layer on each barrier)
    const uint64_t pol = l2_evict_first();  // weights are read once per launch
    // Pieces of this warp: fn(local unit j, first record, end record) for every unit, in order (piece j).
    auto for_pieces = [&](auto fn) {
        if (k1w > k0w)
            for (int j = 0; j < nu; ++j) fn(j, k0w, k1w);
    };
    // Copy of unit j (its gate and up row groups are adjacent in the packed matrix) to its place in shared memory.
    auto copy_unit = [&](const uint8_t *src, int j) {
        mbar_arrive_expect_tx(&ms->bar_u[j], (uint32_t)ubytes);
        bulk_g2s_hint(w1 + j * ubytes, src, (uint32_t)ubytes, &ms->bar_u[j], pol);
        armed_u |= 1u << j;
    };
    auto abort_warp = [&]() {
        bad = true;
        if (lane == 0) {
            vflags[0] = 1;
            raise_status(a.status, kStatusTimeout);
        }
    };
    // Gate/up pieces of one kind (shared or routed), in this warp's order; partial tiles to shared memory.
    auto run_pieces = [&](bool shared_kind) {
        for_pieces([&](int j, int k0, int k1) {
            const int pi = j;
            const bool sh = u0 + j < a.nft_s;
            if (sh == shared_kind) {
                if (!bad && !__all_sync(0xffffffffu, mbar_wait(&ms->bar_u[j], par, a.wait_data, vflags))) abort_warp();
                __syncwarp();  // reconverge before the warp-wide MMAs (lane 0 may have polled alone)
                float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
                const bool first_routed = !sh && (j == 0 || u0 + j == a.nft_s);
                if (first_routed) CSTAMP(84);
                if (!bad) {
                    const uint8_t *un = w1 + j * ubytes;
                    for (int k = k0; k < k1; ++k) {
                        const uint8_t *recs[2] = {un + (int64_t)k * a.rec, un + (int64_t)(a.kc_h + k) * a.rec};
                        row_mma<FMT, 2, kXEnt>(recs, xc + (int64_t)k * CB * kXEnt, xsel, lane, acc);
                        if (first_routed && k == k0) CSTAMP(85);
                    }
                }
                if (first_routed) CSTAMP(86);
                if (t4 == 0) {  // column 0: rows g and g + 8
                    float *dst = p1p + (size_t)((warp * kRowPieces + pi) * 2) * 16;
                    dst[g] = acc[0][0];
                    dst[g + 8] = acc[0][1];
                    dst[16 + g] = acc[1][0];
                    dst[16 + g + 8] = acc[1][1];
                }
            }
        });
    };

    // ---- the layers, one after another: every CTA takes the same share of each; a layer's input row is the
    //      residual row the previous layer's CTAs left, exchanged as tagged words like h
    const int nl = MULTI ? a.nl : 1;
    for (int l = 0; l < nl; ++l) {
    const RowLayer &Ly = a.layer[l];
    par = (uint32_t)l & 1u;
    if (l > 0) {
        __syncthreads();  // every reader of the previous layer's shared-memory operands is done
        if (tid == 0)
            for (int i = 0; i <= kMaxTopK; ++i) ms->slot_ready[i] = 0;
        armed_u = 0u;  // the previous layer's copies were all consumed
        armed_p2rt = false;
        routed = false;
    }
        // ---- 0. weights that depend on nothing: router rows (and the shared-gate row), the shared expert's
        //         f-tiles of this CTA, its shared down rows; issued before waiting for the previous kernel
        // the CTA's router rows (and the shared-gate row) straight into registers: thread t holds 16-byte
        // vectors t, t + 512, ... of the rows laid end to end
        const int nvec = a.H / 8, nitems = (rr1 - rr0) * nvec;
        uint4 rwv[kRowRouterRegs];
    #pragma unroll
        for (int j = 0; j < kRowRouterRegs; ++j) {
            const int it = tid + j * kRowThreads;
            rwv[j] = make_uint4(0u, 0u, 0u, 0u);
            if (it < nitems) {
                const int row = it / nvec, v = it - row * nvec;
                const uint16_t *src = rr0 + row < a.E ? Ly.router + (int64_t)(rr0 + row) * a.H : Ly.sgate;
                rwv[j] = __ldg(reinterpret_cast<const uint4 *>(src) + v);
            }
        }
        if (tid == 0)
            for (int jj = 0; jj < nu && u0 + jj < a.nft_s; ++jj)
                copy_unit(Ly.sgu + (int64_t)(2 * (u0 + jj)) * a.kc_h * a.rec, jj);
        armed_p2sh = nrg > 0;
        if (tid == 32 && armed_p2sh) {
            mbar_arrive_expect_tx(&ms->bar_p2sh, (uint32_t)(nrg * a.kc_fs * a.rec));
            for (int j = 0; j < nrg; ++j) {
                const int rg = c + j * a.ncta;
                bulk_g2s_hint(w2 + (int64_t)(j * IPR + a.K * a.kc_f) * a.rec, Ly.sdn + (int64_t)rg * a.kc_fs * a.rec,
                              (uint32_t)(a.kc_fs * a.rec), &ms->bar_p2sh, pol);
            }
        }
        if (l == 0) {
            grid_dep_wait();  // the previous kernel (which may have written x) has finished
            if (tid == 0) ms->ep = *reinterpret_cast<volatile uint32_t *>(a.epoch);  // the previous launch's last word
            if (tid == 0) {
                mbar_arrive_expect_tx(&ms->bar_x, (uint32_t)a.H * 2);
                bulk_g2s(xs, a.x, (uint32_t)a.H * 2, &ms->bar_x);
            }
        }
        STAMP(1);


    [&]() {
        // ---- 1. the activation row: statistics (spread over the CTA, one barrier), then this CTA's router
        //         logits
        if (l == 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(&ms->bar_x, 0u, a.wait_data, nullptr))) abort_warp();
        } else {
            // the residual row the previous layer left, tagged with that layer's epoch: each thread the words
            // of its own 16-byte vectors of the row (the statistics below read exactly those)
            const uint32_t Tp = ms->ep + (uint32_t)l;
            bool seen = false;
            const uint64_t t0 = global_ns();
            for (int64_t it = 0; !bad && it < a.wait.iters; ++it) {
                bool mine = true;
                for (int v = tid; v < a.H / 8; v += kRowThreads) {
                    const ulonglong2 w0 = ld_words2(a.xw + 4 * v), w1v = ld_words2(a.xw + 4 * v + 2);
                    mine &= word_tag(w0.x) == Tp && word_tag(w0.y) == Tp && word_tag(w1v.x) == Tp &&
                            word_tag(w1v.y) == Tp;
                    reinterpret_cast<uint4 *>(xs)[v] =
                        make_uint4((uint32_t)w0.x, (uint32_t)w0.y, (uint32_t)w1v.x, (uint32_t)w1v.y);
                }
                if (__all_sync(0xffffffffu, mine)) {
                    seen = true;
                    break;
                }
                if (global_ns() - t0 > a.wait.nanos) break;
            }
            if (!seen) abort_warp();
        }
        __syncwarp();  // warps left diverged (lane-0 copy issue above) run warp collectives many times slower
        STAMP(2);
        // every thread a 16-byte vector (or none), warp partials, then every thread adds the 16 partials in
        // warp order (the same sum everywhere)
        float inv = 1.f;
        int shift_x = 0;
        {
            const uint4 *xv = reinterpret_cast<const uint4 *>(xs);
            float ss = 0.f;
            uint32_t mx2 = 0u;
            for (int i = tid; i < a.H / 8; i += kRowThreads) {
                const uint4 v = xv[i];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    mx2 = __vmaxu2(mx2, w[h] & 0x7FFF7FFFu);
                    const float lo = bf16_bits_to_f32(w[h] & 0xFFFFu), hi = bf16_bits_to_f32(w[h] >> 16);
                    ss = fmaf(lo, lo, ss);
                    ss = fmaf(hi, hi, ss);
                }
            }
            uint32_t mxw = max(mx2 & 0xFFFFu, mx2 >> 16);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mxw = max(mxw, __shfl_xor_sync(0xffffffffu, mxw, o));
            ss = warp_sum(ss);
            if (lane == 0) {
                ms->sst[warp] = ss;
                ms->smx[warp] = mxw;
            }
            __syncthreads();
            float sst = 0.f;
            uint32_t mxt = 0u;
#pragma unroll
            for (int w = 0; w < NW; w += 4) {
                const float4 s4 = *reinterpret_cast<const float4 *>(ms->sst + w);
                const uint4 m4 = *reinterpret_cast<const uint4 *>(ms->smx + w);
                sst = sst + s4.x + s4.y + s4.z + s4.w;
                mxt = max(max(mxt, max(m4.x, m4.y)), max(m4.z, m4.w));
            }
            float mx = bf16_bits_to_f32(mxt);
            if (a.norm) {
                inv = 1.0f / sqrtf(sst / (float)a.H + a.eps);
                mx = bf16_bits_to_f32(f32_to_bf16_bits(mx * inv));  // max |bf16(x * inv)|: rounding is monotonic
            }
            shift_x = frag_shift(mx);
        }
        // the row as the MoE sees it: x, or bf16(RMSNorm(x)) in stack mode
        auto xval = [&](uint32_t bits) {
            const float v = bf16_bits_to_f32(bits);
            return a.norm ? bf16_bits_to_f32(f32_to_bf16_bits(v * inv)) : v;
        };
        STAMP(3);
        // logits of this CTA's router rows: each thread's vectors, warp sums per row, the warps' sums in warp order
        const int nr = rr1 - rr0;
        {
            float part[kRowMaxRouterRows] = {0.f, 0.f, 0.f, 0.f};
            const uint4 *xv = reinterpret_cast<const uint4 *>(xs);
#pragma unroll
            for (int j = 0; j < kRowRouterRegs; ++j) {
                const int it = tid + j * kRowThreads;
                if (!bad && it < nitems) {
                    const int row = it / nvec, v = it - row * nvec;
                    const uint4 xq = xv[v];
                    const uint32_t xw[4] = {xq.x, xq.y, xq.z, xq.w};
                    const uint32_t ww[4] = {rwv[j].x, rwv[j].y, rwv[j].z, rwv[j].w};
                    float d = 0.f;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        d = fmaf(xval(xw[h] & 0xFFFFu), bf16_bits_to_f32(ww[h] & 0xFFFFu), d);
                        d = fmaf(xval(xw[h] >> 16), bf16_bits_to_f32(ww[h] >> 16), d);
                    }
#pragma unroll
                    for (int r = 0; r < kRowMaxRouterRows; ++r)
                        if (r == row) part[r] += d;
                }
            }
            CSTAMP(91);
#pragma unroll
            for (int r = 0; r < kRowMaxRouterRows; ++r) {
                const float sr = warp_sum(part[r]);
                if (lane == 0 && r < nr) ms->red[warp][r] = sr;
            }
            CSTAMP(92);
            __syncthreads();
            CSTAMP(93);
            if (tid < nr) {
                float acc = 0.f;
                for (int w = 0; w < NW; ++w) acc += ms->red[w][tid];
                const int row = rr0 + tid;
                if (row < a.E && Ly.rbias) acc += Ly.rbias[row];
                ms->lgv[tid] = acc;
            }
            __syncthreads();
            CSTAMP(94);
            // into every CTA's mailbox (a poller reads only its own lines)
            for (int q = tid; q < a.ncta * nr; q += kRowThreads) {
                const int box = q / nr, r = q - box * nr;
                st_word(a.lgw + (int64_t)box * a.lsb + rr0 + r, tag_word(ms->ep + 1u + (uint32_t)l, ms->lgv[r]));
            }
            CSTAMP(95);
            __threadfence();  // push the stores out now (nothing waits on this fence but this thread)
            CSTAMP(96);
        }
        if (__syncthreads_or(bad)) {
            bad = true;
            return;
        }
        STAMP(4);

        // ---- 2. warp 0: wait for every CTA's logits and take the top-k; warps 1-15 meanwhile build the x
        //         fragments and compute their shared-expert pieces
        if (warp == 0) {
            // poll every CTA's logits (lane l: experts 8l .. 8l+7, and the shared-gate logit) until each word
            // carries this launch's epoch
            const uint32_t T = ms->ep + 1u + (uint32_t)l;
            unsigned long long wv[8], wgate = 0ull;
            bool ok = false;
            {
                const uint64_t t0 = global_ns();
                for (int64_t it = 0; it < a.wait.iters; ++it) {
                    bool mine = true;
                    const unsigned long long *box = a.lgw + (int64_t)c * a.lsb;
                    if (8 * lane + 8 <= a.E) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const ulonglong2 v = ld_words2(box + 8 * lane + 2 * q);
                            wv[2 * q] = v.x;
                            wv[2 * q + 1] = v.y;
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; ++q) wv[q] = 8 * lane + q < a.E ? ld_word(box + 8 * lane + q) : 0ull;
                    }
                    wgate = ld_word(box + a.E);
#pragma unroll
                    for (int q = 0; q < 8; ++q) mine &= 8 * lane + q >= a.E || word_tag(wv[q]) == T;
                    mine &= word_tag(wgate) == T;
                    if (__all_sync(0xffffffffu, mine)) {
                        ok = true;
                        break;
                    }
                    if (global_ns() - t0 > a.wait.nanos) break;
                }
            }
            if (!ok) abort_warp();
            __syncwarp();
            if (ok && c == 0 && lane == 0) *a.epoch = T;  // every CTA has read the old word (its logits say so)
            STAMP(5);
            // lane l holds experts 8l .. 8l+7, sorted (key descending, index ascending); each round the lanes
            // offer their heads, the largest key wins, among equal keys the lowest lane, i.e. the lower expert
            // index; lane s keeps the slot-s winner. Slot 0 is the row maximum, so w_s = exp(l_s - l_0) / sum.
            if (!bad) {
                uint32_t key[8];
                int qi[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) key[q] = 8 * lane + q < a.E ? order_key(word_value(wv[q])) : 0u;  // 0: below any logit
                const float gate_logit = word_value(wgate);
                CSTAMP(87);
#pragma unroll
                for (int q = 0; q < 8; ++q) qi[q] = q;
                sort8_desc(key, qi);
                CSTAMP(88);
                int my_e = 0;
                float my_l = 0.f;
                // lane jj < nu holding a routed f-tile unit requests it in the round that decides its slot
                const int r_l = u0 + lane - a.nft_s;
                const int su_l = lane < nu && r_l >= 0 ? r_l / a.nft : -1;
                for (int s = 0; s < a.K; ++s) {
                    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key[0]);
                    const uint32_t bal = __ballot_sync(0xffffffffu, key[0] == kmax);
                    const int wl = __ffs(bal) - 1;
                    const int q = __shfl_sync(0xffffffffu, qi[0], wl);
                    const int es = min(8 * wl + q, a.E - 1);
                    if (lane == s) {
                        my_e = es;
                        my_l = key_value(kmax);
                    }
                    if (su_l == s)
                        copy_unit(Ly.gu + (int64_t)es * a.gu_stride + (int64_t)(2 * (r_l - s * a.nft)) * a.kc_h * a.rec, lane);
                    __syncwarp();
                    const bool win = lane == wl;
#pragma unroll
                    for (int i = 0; i < 7; ++i) {
                        key[i] = win ? key[i + 1] : key[i];
                        qi[i] = win ? qi[i + 1] : qi[i];
                    }
                    key[7] = win ? 0u : key[7];
                }
                CSTAMP(89);
                // ---- 3. the routed weights of this CTA, at once, one lane per copy: lane jj the f-tile unit jj,
                //         lane s the down rows of slot s
                {
                    const uint32_t issued = __ballot_sync(0xffffffffu, su_l >= 0);
                    if (lane == 0) armed_u |= issued;
                    if (lane < a.K) ms->esl[lane] = my_e;  // the down rows follow once the gate/up bytes are in
                    routed = true;
                    __syncwarp();
                }
                const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
                const float p = lane < a.K ? __expf(my_l - l0) : 0.f;
                const float psum = warp_sum(p);
                const float my_w = __fdividef(p, psum);
                if (lane < a.K) {
                    ms->wsl[lane] = my_w;
                    if (c == 0) {
                        if (a.topk_idx) a.topk_idx[(int64_t)l * a.K + lane] = my_e;
                        if (a.topk_w) a.topk_w[(int64_t)l * a.K + lane] = my_w;
                    }
                }
                if (lane == 0) ms->wsl[a.K] = __fdividef(1.0f, 1.0f + __expf(-gate_logit));
                CSTAMP(90);
                __syncwarp();
                STAMP(7);
            }
        } else {
            // compact x fragments: entry (block b, t) = the B fragment pair of lane (0, t): row values 16b + 2t,
            // +1 and 16b + 2t + 8, +9, scaled by 2^shift_x into fp16 (exact for every bf16 value above 2^-14 of
            // the row maximum); entry 4 and blocks past the row are zero
            const float sc = pow2f(shift_x);
            const int nent = a.kc_h * CB * kXEnt;
            for (int e = tid - kWarp; e < nent; e += kRowThreads - kWarp) {
                const int b = e / kXEnt, t = e - b * kXEnt;
                uint2 v = make_uint2(0u, 0u);
                if (t < 4 && b < a.H / 16) {
                    const uint32_t w0 = *reinterpret_cast<const uint32_t *>(xs + 16 * b + 2 * t);
                    const uint32_t w1v = *reinterpret_cast<const uint32_t *>(xs + 16 * b + 2 * t + 8);
                    v = make_uint2(pack_half2(xval(w0 & 0xFFFFu) * sc, xval(w0 >> 16) * sc),
                                   pack_half2(xval(w1v & 0xFFFFu) * sc, xval(w1v >> 16) * sc));
                }
                xc[e] = v;
            }
            bar_sync(1, kRowThreads - kWarp);  // warps 1-15: the fragments are complete
            if (warp == 1) bar_arrive(2, 2 * kWarp);  // ... which warp 0 learns through barrier 2
            __syncwarp();
            run_pieces(true);
        }
        STAMP(6);

        // ---- 4. gate/up: warp 0's shared pieces, then every warp's routed pieces
        if (warp == 0) {
            bar_sync(2, 2 * kWarp);  // the fragments (built by warps 1-15)
            __syncwarp();
            run_pieces(true);
        }
        run_pieces(false);
        if (warp == 0 && routed && !bad && nrg > 0) {
            // the routed down rows, one lane per slot: requested only now, so that the gate/up bytes (on the
            // critical path) have the memory system to themselves; they are needed after the h exchange
            if (lane == 0) mbar_arrive_expect_tx(&ms->bar_p2rt, (uint32_t)(nrg * a.K * a.kc_f * a.rec));
            __syncwarp();
            if (lane < a.K) {
                const int e = ms->esl[lane];
                for (int j = 0; j < nrg; ++j) {
                    const int rg = c + j * a.ncta;
                    bulk_g2s_hint(w2 + (int64_t)(j * IPR + lane * a.kc_f) * a.rec,
                                  Ly.dn + (int64_t)e * a.dn_stride + (int64_t)rg * a.kc_f * a.rec,
                                  (uint32_t)(a.kc_f * a.rec), &ms->bar_p2rt, pol);
                }
            }
            armed_p2rt = true;
            __syncwarp();
        }
        WSTAMP(16);
        if (__syncthreads_or(bad)) {
            bad = true;
            return;
        }
        STAMP(8);
        // each unit's pieces summed in warp order -> h = silu(gate) * up, out as tagged words
        const uint32_t T = ms->ep + 1u + (uint32_t)l;
        if (tid < nu * 16) {
            const int j = tid >> 4, n = tid & 15;
            float sg = 0.f, su = 0.f;
            for (int w = 0; w < NW; ++w) {
                if ((w + 1) * a.kc_h / NW == w * a.kc_h / NW) continue;  // an empty slice
                const float *src = p1p + (size_t)((w * kRowPieces + j) * 2) * 16;
                sg += src[n];
                su += src[16 + n];
            }
            const int sh = 24 - (MB - 1) - shift_x;
            const float gv = mul_pow2(sg, sh), uv = mul_pow2(su, sh);
            const float hv = gv / (1.0f + expf(-gv)) * uv;
            const int i = u0 + j;
            const int r = i - a.nft_s;
            const int slot = r < 0 ? a.K : r / a.nft;
            const int ft = r < 0 ? i : r - slot * a.nft;
            st_word(a.hw + (int64_t)slot * a.Fmax + ft * 16 + n, tag_word(T, hv));
        }
        STAMP(9);
        if (nrg == 0) return;

        // ---- 5. each slot's h from every CTA (one warp per slot): wait until the words carry this launch's
        //         epoch (first the last word of each 16-value unit, then every word), then the compact h
        //         operands: the routing weight (slot K: the shared gate) folded in, a power-of-two scale from
        //         max |w h| (weights are positive, so that is w max |h|, rounding included) into fp16 range,
        //         split into hi + lo (22 significant bits). Up to 4 blocks per lane are kept in registers;
        //         wider experts read h a second time.
        __syncwarp();
        for (int s = warp; !bad && s <= a.K; s += NW) {
            const int nblk = (s < a.K ? a.F : a.Fs) / 16;
            const int nb = (s < a.K ? a.kc_f : a.kc_fs) * CB;  // blocks the records span (the rest zero)
            const unsigned long long *hs = a.hw + (int64_t)s * a.Fmax;
            const float wgt = ms->wsl[s];
            // lane (bq, tq) = (lane >> 2, lane & 3) takes blocks bq, bq + 8, ... and the values of lane (0, tq)
            const int bq = lane >> 2, tq = lane & 3;
            float4 hv[4];
            bool ok = false;
            const uint64_t t0 = global_ns();
            for (int64_t it = 0; it < a.wait.iters; ++it) {
                bool mine = true;
                for (int u = lane; u < nblk; u += kWarp) mine &= word_tag(ld_word(hs + 16 * u + 15)) == T;
                if (__all_sync(0xffffffffu, mine)) {
                    ok = true;
                    break;
                }
                if (global_ns() - t0 > a.wait.nanos) break;
            }
            bool seen = false;
            for (int64_t it = 0; ok && it < a.wait.iters; ++it) {
                bool mine = true;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int b = bq + 8 * q;
                    hv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (b < nblk) {
                        const ulonglong2 p = ld_words2(hs + 16 * b + 2 * tq), r2 = ld_words2(hs + 16 * b + 2 * tq + 8);
                        mine &= word_tag(p.x) == T && word_tag(p.y) == T && word_tag(r2.x) == T && word_tag(r2.y) == T;
                        hv[q] = make_float4(word_value(p.x), word_value(p.y), word_value(r2.x), word_value(r2.y));
                    }
                }
                for (int b = bq + 32; b < nblk; b += 8) {
                    const ulonglong2 p = ld_words2(hs + 16 * b + 2 * tq), r2 = ld_words2(hs + 16 * b + 2 * tq + 8);
                    mine &= word_tag(p.x) == T && word_tag(p.y) == T && word_tag(r2.x) == T && word_tag(r2.y) == T;
                }
                if (__all_sync(0xffffffffu, mine)) {
                    seen = true;
                    break;
                }
                if (global_ns() - t0 > a.wait.nanos) break;
            }
            if (!seen) {
                abort_warp();
                break;
            }
            float hm = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                hm = fmaxf(hm, fmaxf(fmaxf(fabsf(hv[q].x), fabsf(hv[q].y)), fmaxf(fabsf(hv[q].z), fabsf(hv[q].w))));
            for (int b = bq + 32; b < nblk; b += 8) {
                const ulonglong2 p = ld_words2(hs + 16 * b + 2 * tq), r2 = ld_words2(hs + 16 * b + 2 * tq + 8);
                hm = fmaxf(hm, fmaxf(fmaxf(fabsf(word_value(p.x)), fabsf(word_value(p.y))),
                                     fmaxf(fabsf(word_value(r2.x)), fabsf(word_value(r2.y)))));
            }
            hm = warp_max(hm);
            const int shift = frag_shift(wgt * hm);
            const float sc = pow2f(shift);
            uint2 *hsl = hc + (size_t)s * a.kbf * kHEnt;
            for (int b = bq; b < nb; b += 8) {
                float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (b < nblk) {
                    if (b < 32) {
                        v4 = b < 8 ? hv[0] : b < 16 ? hv[1] : b < 24 ? hv[2] : hv[3];
                    } else {
                        const ulonglong2 p = ld_words2(hs + 16 * b + 2 * tq), r2 = ld_words2(hs + 16 * b + 2 * tq + 8);
                        v4 = make_float4(word_value(p.x), word_value(p.y), word_value(r2.x), word_value(r2.y));
                    }
                }
                const float v[4] = {v4.x * wgt * sc, v4.y * wgt * sc, v4.z * wgt * sc, v4.w * wgt * sc};
                __half h[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) h[k] = __float2half_rn(v[k]);
                __half2 h01 = __halves2half2(h[0], h[1]), h23 = __halves2half2(h[2], h[3]);
                hsl[b * kHEnt + tq] = make_uint2(*reinterpret_cast<uint32_t *>(&h01), *reinterpret_cast<uint32_t *>(&h23));
                hsl[b * kHEnt + 4 + tq] = make_uint2(pack_half2(v[0] - __half2float(h[0]), v[1] - __half2float(h[1])),
                                                     pack_half2(v[2] - __half2float(h[2]), v[3] - __half2float(h[3])));
                if (tq == 0) hsl[b * kHEnt + 8] = make_uint2(0u, 0u);
            }
            if (lane == 0) ms->shift_s[s] = shift;
            __syncwarp();
            __threadfence_block();  // the operands before the flag
            if (lane == 0) reinterpret_cast<volatile int *>(ms->slot_ready)[s] = 1;
            if (s == 0) STAMP(10);
        }
        if (!bad && !__all_sync(0xffffffffu, mbar_wait(&ms->bar_p2sh, par, a.wait_data, vflags) &&
                                                 mbar_wait(&ms->bar_p2rt, par, a.wait_data, vflags)))
            abort_warp();
        __syncwarp();
        STAMP(11);
        // ---- 6. down projections: this warp's items, one piece per (row group, slot) run
        {
            int pi = 0;
            int j = it0 / IPR, rem = it0 - j * IPR;
            for (int i = it0; i < it1;) {
                const bool shs = rem >= a.K * a.kc_f;
                const int s = shs ? a.K : rem / a.kc_f;
                const int r0 = shs ? rem - a.K * a.kc_f : rem - s * a.kc_f;
                const int kcs = shs ? a.kc_fs : a.kc_f;
                const int n = min(kcs - r0, it1 - i);
                float acc[1][2] = {{0.f, 0.f}};
                if (!bad) {  // the slot's operands (built by warp s % 16)
                    bool okf = true;
                    if (lane == 0) {
                        const volatile int *f = ms->slot_ready + s;
                        okf = *f != 0;
                        const uint64_t t0 = global_ns();
                        while (!okf && !vflags[0] && global_ns() - t0 < a.wait_data.nanos) okf = *f != 0;
                    }
                    if (!__shfl_sync(0xffffffffu, (int)okf, 0)) abort_warp();
                    __threadfence_block();
                }
                __syncwarp();
                if (!bad) {
                    const uint2 *hsl = hc + (size_t)s * a.kbf * kHEnt;
                    if (pi == 0) CSTAMP(80);
                    for (int q = 0; q < n; ++q) {
                        const uint8_t *recs[1] = {w2 + (int64_t)(i + q) * a.rec};
                        row_mma<FMT, 1, kHEnt>(recs, hsl + (r0 + q) * CB * kHEnt, hsel, lane, acc);
                        if (pi == 0 && q == 0) CSTAMP(81);
                    }
                    if (pi == 0) CSTAMP(82);
                }
                // column 0 (hi, lanes t = 0) + column 4 (lo, lanes t = 2)
                const float v0 = acc[0][0] + __shfl_xor_sync(0xffffffffu, acc[0][0], 2);
                const float v1 = acc[0][1] + __shfl_xor_sync(0xffffffffu, acc[0][1], 2);
                if (t4 == 0) {
                    float *dst = p2p + (size_t)(warp * kRowPieces + pi) * 16;
                    dst[g] = v0;
                    dst[g + 8] = v1;
                }
                ++pi;
                i += n;
                rem += n;
                if (rem == IPR) {
                    rem = 0;
                    ++j;
                }
            }
        }
        WSTAMP(32);
        if (__syncthreads_or(bad)) {
            bad = true;
            return;
        }
        STAMP(12);
        // ---- 7. y for this CTA's row groups: each (row group, slot, row) partial from its pieces in warp order,
        //         then the slots summed in order (the shared expert last)
        float *const ysl = p1p;  // [row group][slot][16]; the gate/up partial tiles are dead
        for (int it = tid; it < nrg * (a.K + 1) * 16; it += kRowThreads) {
            const int n = it & 15, js = it >> 4, j = js / (a.K + 1), s = js - j * (a.K + 1);
            const int gi0 = j * IPR + s * a.kc_f;  // the shared slot starts after the K routed ones as well
            const int gi1 = gi0 + (s < a.K ? a.kc_f : a.kc_fs);
            float ps = 0.f;
            for (int w = 0; w < NW; ++w) {
                const int a0 = w * I2 / NW, a1 = (w + 1) * I2 / NW;
                if (a0 >= a1 || a1 <= gi0 || a0 >= gi1) continue;
                ps += p2p[(size_t)(w * kRowPieces + js - ms->p2g0[w]) * 16 + n];
            }
            ysl[it] = mul_pow2(ps, 24 - (MB - 1) - ms->shift_s[s]);
        }
        __syncthreads();
        if (tid < ((nrg * 16 + kWarp - 1) & ~(kWarp - 1))) {  // whole warps (the pairing shuffle)
            const int j = tid >> 4, n = tid & 15;
            const bool live = tid < nrg * 16;
            float ysum = 0.f;
            if (live) {
                float yv[kMaxTopK + 1];
#pragma unroll
                for (int s = 0; s <= kMaxTopK; ++s) yv[s] = s <= a.K ? ysl[(j * (a.K + 1) + s) * 16 + n] : 0.f;
#pragma unroll
                for (int s = 0; s <= kMaxTopK; ++s)
                    if (s <= a.K) ysum += yv[s];
            }
            const int o = (c + j * a.ncta) * 16 + n;
            const bool inrow = live && o < a.H;
            const uint32_t hb = inrow ? f32_to_bf16_bits(bf16_bits_to_f32(xs[o]) + ysum) : 0u;  // the residual row
            if (l == nl - 1) {
                if (inrow && a.y) a.y[o] = ysum;
                if (inrow && a.h_out) a.h_out[o] = (uint16_t)hb;
            } else {
                // rows 2i, 2i + 1 as word i, tagged with this layer's epoch, for the next layer
                const uint32_t hb1 = __shfl_down_sync(0xffffffffu, hb, 1);
                if (inrow && !(n & 1))
                    st_word(a.xw + o / 2, ((unsigned long long)(ms->ep + 1u + (uint32_t)l) << 32) | hb | (hb1 << 16));
            }
        }
    }();
    if (bad) break;
    }

    // No copy may still be landing in shared memory when the CTA exits (every path).
    {
        const WaitCfg drain{int64_t(1) << 40, 1000000000ull};
        if (tid == 0) {
            mbar_wait(&ms->bar_x, 0u, drain, nullptr);
            for (int j = 0; j < nu; ++j)
                if ((armed_u >> j) & 1u) mbar_wait(&ms->bar_u[j], par, drain, nullptr);
            if (armed_p2rt) mbar_wait(&ms->bar_p2rt, par, drain, nullptr);
        }
        if (tid == 32 && armed_p2sh) mbar_wait(&ms->bar_p2sh, par, drain, nullptr);
    }
    WSTAMP(48);
    __syncthreads();
    STAMP(13);
#undef STAMP
#undef WSTAMP
#undef CSTAMP
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
struct RowPlan {
    int ncta = 0, kbf = 0, rpc = 0;
    size_t smem = 0;
    int off_stage = 0, off_xc = 0, off_hc = 0, off_p1 = 0, off_p2 = 0, off_misc = 0;
    std::vector<int16_t> ub;
};

// Pieces of a warp's range [w T / NW, (w + 1) T / NW) of items grouped in runs of `run` (the last run of a
// group may be shorter when sizes differ: `group_of` gives the run index of an item).
template <class F>
static int max_pieces(int total, F group_of) {
    int mx = 0;
    for (int w = 0; w < kRowWarps; ++w) {
        const int a0 = w * total / kRowWarps, a1 = (w + 1) * total / kRowWarps;
        if (a1 > a0) mx = std::max(mx, group_of(a1 - 1) - group_of(a0) + 1);
    }
    return mx;
}

// Fills p when the one-row path can run the layer; false otherwise (the general kernel then runs it).
static bool plan_row(const bfp_moe_layer *L, const Geometry &gu, const Geometry &dn, const Geometry &sdn, int sms,
                     int smem_optin, RowPlan *p) {
    const int K = L->top_k, H = L->hidden;
    const int nft = L->ffn / 16, nft_s = L->shared_ffn / 16;
    const int kc_h = (int)gu.kc, kc_f = (int)dn.kc, kc_fs = (int)sdn.kc, rec = gu.rec, CB = gu.cb;
    const int n1 = nft_s + K * nft;
    const int ng_d = (int)dn.ng;
    if (n1 > 32767) return false;
    p->ncta = std::max(1, std::min({sms, kRowMaxCta, std::max(n1, ng_d)}));
    const int ncta = p->ncta;
    const int nrg_max = (ng_d + ncta - 1) / ncta;
    if (nrg_max > kRowMaxRg) return false;
    const int64_t u = 2 * (int64_t)kc_h * rec;
    const int IPR = K * kc_f + kc_fs;
    const int64_t P2 = (int64_t)IPR * rec;
    // f-tile ranges split evenly (whole units): the gate/up bytes of a CTA decide when its h is out, and every
    // CTA waits for the last h, while the down rows are needed only after that exchange
    p->ub.assign(ncta + 1, 0);
    for (int c = 1; c < ncta; ++c) p->ub[c] = (int16_t)((int64_t)c * n1 / ncta);
    p->ub[ncta] = (int16_t)n1;
    int64_t area = 0;
    for (int c = 0; c < ncta; ++c) {
        const int nu = p->ub[c + 1] - p->ub[c];
        if (nu * 16 > kRowThreads) return false;  // one thread per (unit, row) sums the pieces
        const int nrg = c < ng_d ? (ng_d - c + ncta - 1) / ncta : 0;
        area = std::max<int64_t>(area, nu * u + nrg * P2);
        if (nu > kRowPieces) return false;  // every warp holds one gate/up piece per unit
        if (max_pieces(nrg * IPR, [&](int i) {
                const int j = i / IPR, rem = i - j * IPR;
                return j * (K + 1) + (rem < K * kc_f ? rem / kc_f : K);
            }) > kRowPieces)
            return false;
    }
    p->rpc = (L->n_experts + 1 + ncta - 1) / ncta;
    if (p->rpc > kRowMaxRouterRows || (int64_t)p->rpc * (H / 8) > (int64_t)kRowThreads * kRowRouterRegs) return false;
    p->kbf = std::max(kc_f, kc_fs) * CB;
    size_t o = align_up((size_t)area, 128);
    p->off_stage = (int)o;
    o = align_up(o + (size_t)H * 2, 16);
    p->off_xc = (int)o;
    o = align_up(o + (size_t)kc_h * CB * kXEnt * 8, 16);
    p->off_hc = (int)o;
    o = align_up(o + (size_t)(K + 1) * p->kbf * kHEnt * 8, 16);
    p->off_p1 = (int)o;
    o = align_up(o + (size_t)kRowWarps * kRowPieces * 2 * 16 * 4, 16);
    p->off_p2 = (int)o;
    o = align_up(o + (size_t)kRowWarps * kRowPieces * 16 * 4, 16);
    p->off_misc = (int)o;
    o = align_up(o + sizeof(RowMisc), 128);
    p->smem = o;
    return (int64_t)p->smem <= (int64_t)smem_optin;
}

template <int FMT, bool MULTI>
static int launch_row_t(const RowArgs &a, size_t smem, cudaStream_t st) {
    auto kern = moe_row_kernel<FMT, MULTI>;
    int rc = set_smem_attr(reinterpret_cast<const void *>(kern), (int)smem, "cudaFuncSetAttribute(moe_row)");
    if (rc) return rc;
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.ncta);
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (launch_mode() == BFP_LAUNCH_COOPERATIVE) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    } else {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return cuda_fail(e, "launch moe_row");
    return BFP_OK;
}

#ifdef BFP_TRACE
extern "C" int bfp_debug_set_trace_row(void *buf) {
    return (int)cudaMemcpyToSymbol(g_bfp_trace, &buf, sizeof(buf));
}
#endif

int row_layers_launch(const bfp_moe_layer *Ls, int nl, const uint16_t *x, int norm, float *y, uint16_t *h_out,
                      int32_t *topk_idx, float *topk_w, uint32_t *status, uint8_t *row_ws, int fmax, cudaStream_t st) {
    if (nl < 1 || nl > kRowStackMax) return kRowNotApplicable;
    const bfp_moe_layer *L = Ls;
    for (int l = 1; l < nl; ++l) {  // one launch runs layers of one shape
        const bfp_moe_layer &M = Ls[l];
        if (M.hidden != L->hidden || M.n_experts != L->n_experts || M.ffn != L->ffn || M.top_k != L->top_k ||
            M.shared_ffn != L->shared_ffn || M.expert_fmt != L->expert_fmt || M.gate_up_stride != L->gate_up_stride ||
            M.down_stride != L->down_stride)
            return kRowNotApplicable;
    }
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    Geometry gu, dn, sdn;
    make_geometry(L->expert_fmt, 2 * (int64_t)L->ffn, L->hidden, &gu);
    make_geometry(L->expert_fmt, L->hidden, L->ffn, &dn);
    make_geometry(L->expert_fmt, L->hidden, L->shared_ffn, &sdn);
    // plans depend on the shape and the device only; a one-row launch cannot afford to recompute one
    struct Cached {
        int key[8];
        bool ok;
        RowPlan plan;
    };
    static std::mutex mu;
    static std::vector<Cached> cache;
    const int key[8] = {L->hidden, L->n_experts, L->ffn, L->top_k, L->shared_ffn, L->expert_fmt, di.sms, di.smem_optin};
    RowPlan p;
    bool ok = false, found = false;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (const Cached &x : cache)
            if (std::equal(key, key + 8, x.key)) {
                ok = x.ok;
                if (ok) p = x.plan;
                found = true;
                break;
            }
    }
    if (!found) {
        ok = plan_row(L, gu, dn, sdn, di.sms, di.smem_optin, &p);
        std::lock_guard<std::mutex> lk(mu);
        Cached x;
        std::copy(key, key + 8, x.key);
        x.ok = ok;
        x.plan = p;
        cache.push_back(x);
    }
    if (!ok) return kRowNotApplicable;
    RowArgs a;
    a.H = L->hidden;
    a.E = L->n_experts;
    a.F = L->ffn;
    a.K = L->top_k;
    a.Fs = L->shared_ffn;
    a.ncta = p.ncta;
    a.nl = nl;
    a.x = x;
    a.norm = norm;
    a.eps = 1e-6f;
    a.gu_stride = L->gate_up_stride;
    a.dn_stride = L->down_stride;
    for (int l = 0; l < nl; ++l) {
        RowLayer &w = a.layer[l];
        w.router = Ls[l].router;
        w.rbias = Ls[l].router_bias;
        w.sgate = Ls[l].shared_gate;
        w.gu = static_cast<const uint8_t *>(Ls[l].experts_gate_up);
        w.dn = static_cast<const uint8_t *>(Ls[l].experts_down);
        w.sgu = static_cast<const uint8_t *>(Ls[l].shared_gate_up);
        w.sdn = static_cast<const uint8_t *>(Ls[l].shared_down);
    }
    a.y = y;
    a.h_out = h_out;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.status = status;
    a.epoch = reinterpret_cast<uint32_t *>(row_ws);
    a.lgw = reinterpret_cast<unsigned long long *>(row_ws + row_ws_logits_off());
    a.lsb = logit_stride(L->n_experts);
    a.hw = reinterpret_cast<unsigned long long *>(row_ws + row_ws_h_off(L->n_experts, row_boxes(di.sms)));
    a.xw = reinterpret_cast<unsigned long long *>(row_ws +
                                                  row_ws_x_off(L->n_experts, L->top_k, fmax, row_boxes(di.sms)));
    a.rec = gu.rec;
    a.kc_h = (int)gu.kc;
    a.kc_f = (int)dn.kc;
    a.kc_fs = (int)sdn.kc;
    a.nft = L->ffn / 16;
    a.nft_s = L->shared_ffn / 16;
    a.ng_d = (int)dn.ng;
    a.Fmax = fmax;
    a.kbf = p.kbf;
    a.off_stage = p.off_stage;
    a.off_xc = p.off_xc;
    a.off_hc = p.off_hc;
    a.off_p1 = p.off_p1;
    a.off_p2 = p.off_p2;
    a.off_misc = p.off_misc;
    a.wait = wait_cfg();
    a.wait_data = WaitCfg{kDefaultWaitIters, kDefaultWaitNanos};
    for (int c = 0; c <= kRowMaxCta; ++c) a.ub[c] = c <= p.ncta ? p.ub[c] : p.ub[p.ncta];
    if (nl > 1)
        return L->expert_fmt == BFP_FMT_BFP4 ? launch_row_t<4, true>(a, p.smem, st) : launch_row_t<8, true>(a, p.smem, st);
    return L->expert_fmt == BFP_FMT_BFP4 ? launch_row_t<4, false>(a, p.smem, st) : launch_row_t<8, false>(a, p.smem, st);
}

}  // namespace bfp
