// MoE decode layer (moe_decode_layer) and decode stack (moe_stack_decode).
//
// What the layer computes (Qwen3.6-35B-A3B card, "Fused decode kernels": MoE
// decode through device top-k routing and batched expert streams, one
// gate/up + down expert program for several rows; 256 experts, top-8 plus a
// shared expert: qwen3.6-a3b-blackhole page):
//     l = Wr x (+bias) -> softmax -> top-k -> renormalise -> for each selected
//     expert  D (silu(G x) * (U x))  combined with the routing weights, plus
//     sigmoid(g . x) * shared(x).
//
// GB300 design: the layer is one persistent kernel, one 512-thread CTA (16
// warps) per SM (a dependent launch by default, cooperative on request).
// Nothing waits on the host between the router and the experts:
//   1. thread 0 stages the activation rows and this CTA's router rows (plus
//      the shared-gate vector as one extra row) in shared memory with 1D bulk
//      copies (the TMA engine); the warps compute the CTA's fp32 logits on the
//      tensor cores and write them to the workspace;
//   2. warps 0-7 publish them (a release increment of a grid counter), wait for
//      every CTA's, and redundantly take softmax / top-k / renormalisation, the
//      union U of the experts any row selected (no host sync, no second launch)
//      and the share of phase-2 units the CTA owns; warps 8-15 meanwhile build
//      the fp16 activation fragments;
//   3. phase 1: f-tile units (16 ffn rows of an expert's gate and up, or of the
//      shared expert). Each warp takes a contiguous, cost-balanced run of the
//      records of the CTA's units (a unit cut by a run boundary is handed from
//      one warp to its neighbour through the workspace; with few units, units
//      are split into equal parts that meet in shared memory) and streams them
//      through two shared-memory slots of its own (lane 0 refills a slot with
//      bulk copies as soon as the warp is done with it; L2 evict-first: the
//      weights are read once); it writes h = silu(gate) * up for the rows that
//      chose the expert, fp32 to the workspace, and the per-(row, slot) maxima
//      of |h|;
//   4. after a grid barrier, phase 2: down-projection units (an expert and 16
//      row groups of the hidden dimension, one per warp): the CTA turns the
//      routing-weighted h of a batch of experts into fp16 hi + lo fragments
//      (22 significant bits) in one pass, and every warp streams its row group
//      of each unit and writes per-(row, slot) partial outputs;
//   5. after a second grid barrier, each CTA sums its row groups' slots in slot
//      order (deterministic, no float atomics) into y (or the bf16 residual).
// Every expert's weights are read from HBM once per step however many rows
// chose it. All cross-CTA waits are bounded and report BFP_ETIMEOUT.
#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "bfp_launch.h"
#include "bfp_tiles.cuh"
#include "bfp_trace.h"
#include "moe_common.cuh"

namespace bfp {

using namespace dev;

int linear_launch_ex(const bfp_matrix *w, const uint16_t *x, int m, int64_t ldx, float *y, uint16_t *y_bf16,
                     int64_t ldy, uint32_t *status, void *body, size_t body_bytes, cudaStream_t st, int norm,
                     int32_t *tokens);
int linear_ws_body_bytes(const bfp_matrix *w, int m, size_t *bytes);

constexpr int kMoeWarps = 16;                // warps of the layer kernel (no producer warp)
constexpr int kMoeThreads = kMoeWarps * 32;
// Floats of one phase-1 partial tile handed between warps: 2 records (gate, up) x 2 activation
// groups x 4 accumulators x 32 lanes.
constexpr int kP1PartFloats = 2 * 2 * 4 * 32;
// Experts whose phase-2 fragments one batch sets up together.
constexpr int kP2Batch = 4;

struct MoeArgs {
    int H, E, F, K, Fs, M, ncta;
    const uint16_t *x;
    int norm;
    float eps;
    const uint16_t *router;
    const float *rbias;
    const uint16_t *sgate;
    const uint8_t *gu, *dn;
    int64_t gu_stride, dn_stride;
    const uint8_t *sgu, *sdn;
    float *y;
    uint16_t *h_out;
    int32_t *topk_idx;
    float *topk_w;
    uint32_t *status, *ctrl;  // ctrl: [0] router, [1] exit, [2] phase-1, [3] phase-2 barrier counters
    uint32_t *hmax;  // [M][K+1] max |h| bits per (row, slot), raised in phase 1
    float *logits, *hbuf, *part;
    float *p1part;   // [ncta][NW-1][kP1PartFloats]: phase-1 partial tiles handed between neighbouring warps
    int rec, kc_h, kbp_h, kc_f, kbp_f, kc_fs, kbp_fs;
    int nft, nft_s, ng_d, r2, noct, Fmax;
    int nsw, ch1, slot_bytes, frag_bytes, scr_bytes;  // per-warp slots, phase-1 chunk records, slot bytes
    int stage_off, stage_r;  // preamble stage: ring offset of the activation rows; router rows after stage_r bytes
    WaitCfg wait;       // cross-block waits (router counter, expert counters)
    WaitCfg wait_data;  // this CTA's own bulk copies and slot hand-backs
};

// Shared-memory bookkeeping of one CTA.
// Phase 2: one expert of a batch (its units, up to qend, run on fragments set up together).
struct P2Entry {
    int j, er, nr, parts, off, qend;  // union position, emask row, rows, fragment parts (1, 2, 4), word offset
};

struct MoeMisc {
    alignas(16) float esc[kMoeWarps][rec_scale_floats<4, 2>()];  // per-warp block scales (mma_records)
    uint64_t stage_full;  // the preamble stage (activation rows, router rows) landed
    int shift_x[kMaxRows];
    float inv[kMaxRows];
    float gate_w[kMaxRows];
    int32_t tk_idx[kMaxRows][kMaxTopK];
    float tk_w[kMaxRows][kMaxTopK];
    alignas(16) uint32_t bitmap[kMaxExperts / 32];  // the experts some row chose
    uint32_t emask[kMaxExperts + 1];  // rows that chose expert e (index kMaxExperts: the shared expert)
    int16_t ulist[kMaxExperts + 1];
    int8_t eslot[kMaxExperts + 1][kMaxRows];  // slot of expert e in row r's top-k (shared: K)
    float2 red[kMoeWarps];          // activation row statistics per (row, segment)
    int32_t p1cnt[kMoeWarps];         // phase 1, units split over warps: parts finished per unit
    int32_t p1flag[kMoeWarps];        // phase 1, contiguous ranges: warp w + 1 has handed over its part
    uint32_t wsum[kMoeWarps];         // routing: per-warp sums of the union scan
    P2Entry p2b[kP2Batch];            // phase 2: the experts of the current batch
    int8_t p2row[kP2Batch][kMaxRows];  // ... fragment column -> row
    int p2shift[kP2Batch][kMaxRows];   // ... fragment column -> power-of-two scale of its h
    int p2nb;
    int64_t p2q[2];                  // this CTA's phase-2 units [p2q[0], p2q[1])
    int nU;
    int flags[4];  // [0] abort
};

// Row stride (elements) of the activation rows staged in shared memory: 16 bytes of padding per row.
__host__ __device__ inline int stage_ldx(int H) { return H + 8; }

// Phase-2 unit cost, for sharing the units between CTAs: every unit streams the same bytes and unpacks
// the same weight tiles (about three MMAs' worth of issue per block); an expert used by <= 4 rows adds
// one MMA per block (hi and lo halves of its rows' h in one 8-column MMA), <= 8 rows two (hi, lo),
// more rows four (two column groups of two).
__device__ __forceinline__ int p2_cost(uint32_t rowmask) {
    const int n = __popc(rowmask);
    return n <= 4 ? 4 : (n <= 8 ? 5 : 7);
}
// Phase-1 unit g of the list [shared-expert f-tiles, routed f-tiles of union expert 0, 1, ...]:
// position in the union U (kMaxExperts for the shared expert) and f-tile.
struct P1Tile {
    int jrow, ft;
    bool sh;
};
__device__ __forceinline__ P1Tile p1_tile(int g, int nft_s, int nft) {
    P1Tile t;
    t.sh = g < nft_s;
    t.jrow = t.sh ? kMaxExperts : (g - nft_s) / nft;
    t.ft = t.sh ? g : (g - nft_s) % nft;
    return t;
}
// Per-warp streams. Warp w has nsw slots of its own in the ring; its k-th item lands in slot
// k mod nsw, and the warp itself issues item k + nsw (lane 0, one or two bulk copies) as soon as it is
// done with item k. Its items, in order:
//   phase 1: the warp's phase-1 items (parts of the CTA's units, unit u being list entry
//            g = c + u * ncta, see p1_tile), each in chunks of ch1 records of its gate row group
//            followed by the same records of its up row group;
//   phase 2: for each down-projection unit q of the CTA's range that has a row group oct * r2 + w,
//            that row group in chunks of 2 * ch1 records.
// Within a phase a warp waits for another only where a phase-1 unit is split between warps (the
// part that finishes first hands its tile over).
template <int FMT, int NGRP>
__global__ void __launch_bounds__(kMoeThreads, 1) moe_layer_kernel(const MoeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int NW = kMoeWarps;
    constexpr int NC = NW * kWarp;  // threads
    constexpr int MB = FMT == 4 ? 3 : 7;
    constexpr int CB = FMT == 4 ? 4 : 2;
    uint32_t *frag = reinterpret_cast<uint32_t *>(smem);
    float *scr = reinterpret_cast<float *>(smem + a.frag_bytes);
    MoeMisc *ms = reinterpret_cast<MoeMisc *>(smem + a.frag_bytes + a.scr_bytes);
    const size_t bar_off = align_up(a.frag_bytes + a.scr_bytes + sizeof(MoeMisc), 16);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + bar_off);  // [NW][nsw]
    uint8_t *ring = smem + align_up(bar_off + 8 * NW * a.nsw, 128);
    uint8_t *stage = ring + a.stage_off;  // preamble only: activation rows, then router rows
    volatile int *vflags = ms->flags;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int E1 = a.E + 1;
#define STAMP(i) BFP_TRACE_AT(i)
    STAMP(0);
    const int rr0 = router_row_start(c, E1, a.ncta), rr1 = router_row_start(c + 1, E1, a.ncta);
    const int64_t gb_h = (int64_t)a.kc_h * a.rec;  // bytes of one gate/up row group
    const int ch1 = a.ch1, ch2 = 2 * a.ch1;

    // Cross-block counters: the router counter ctrl[0] and the phase barriers ctrl[2], ctrl[3] count to
    // the grid size. CTA 0 zeroes each once every CTA is past its wait: ctrl[0] after the phase-1
    // barrier, ctrl[2] (and the row maxima) after the phase-2 barrier, ctrl[3] at the start of the
    // next launch (no CTA reaches it before CTA 0 has arrived at ctrl[2]). A launch that gave up
    // (BFP_ETIMEOUT) leaves them set until the workspace is initialised again.
    for (int i = tid; i < kMaxExperts; i += NC) ms->emask[i] = 0u;
    if (tid < a.M) ms->eslot[kMaxExperts][tid] = (int8_t)a.K;
    if (tid == 0) ms->emask[kMaxExperts] = (1u << a.M) - 1u;
    if (tid < kMaxExperts / 32) ms->bitmap[tid] = 0u;
    if (tid <= NW * a.nsw) {  // one barrier per thread
        mbar_init(tid < NW * a.nsw ? &full[tid] : &ms->stage_full, 1);
        mbar_fence_init();
    }
    if (tid < NW) {
        ms->p1cnt[tid] = 0;
        ms->p1flag[tid] = 0;
    }
    if (tid < 4) ms->flags[tid] = 0;
    if (tid == 0) ms->nU = 0;
    // dependent launch: the next launch may take the SMs as this one's CTAs leave; nothing here has
    // touched global memory yet, and nothing below does before the previous launch has finished
    grid_dep_launch_dependents();
    grid_dep_wait();
    if (c == 0 && tid == 0) a.ctrl[3] = 0u;
    __syncthreads();
    STAMP(13);
    const int LDXS = stage_ldx(a.H);
    if (tid == 0) {
        // preamble stage: this CTA's router rows and (the CTA holding row E) the shared-gate row,
        // then the activation rows (row stride LDXS: the padding keeps the router's fragment loads
        // free of bank conflicts); one thread issues the copies one after another (cheaper than
        // several lanes issuing at once)
        const uint32_t xb = (uint32_t)a.M * a.H * 2;
        const int re = min(rr1, a.E);
        const uint32_t rb = re > rr0 ? (uint32_t)(re - rr0) * a.H * 2 : 0u;
        const uint32_t gsb = rr1 > a.E ? (uint32_t)a.H * 2 : 0u;
        mbar_arrive_expect_tx(&ms->stage_full, xb + rb + gsb);
        if (rb) bulk_g2s(stage + a.stage_r, a.router + (int64_t)rr0 * a.H, rb, &ms->stage_full);
        if (gsb) bulk_g2s(stage + a.stage_r + rb, a.sgate, gsb, &ms->stage_full);
        for (int r = 0; r < a.M; ++r)
            bulk_g2s(stage + (size_t)r * LDXS * 2, a.x + (int64_t)r * a.H, (uint32_t)a.H * 2, &ms->stage_full);
    }
    {
        bool bad = false;
        const uint2 *frag2 = reinterpret_cast<const uint2 *>(frag);
        const int ngrp_rows = a.M > 8 ? 3 : 1;
        auto abort_all = [&]() {
            if (tid == 0) {
                vflags[0] = 1;
                raise_status(a.status, kStatusTimeout);
            }
        };
        // A warp that gives up marks the CTA aborted; the other warps' waits see the flag and stop, and
        // the CTA-wide checks turn it into an exit.
        auto abort_warp = [&]() {
            bad = true;
            if (lane == 0) {
                vflags[0] = 1;
                raise_status(a.status, kStatusTimeout);
            }
        };
        auto check_abort = [&]() {
            if (!bad && vflags[0]) bad = true;
        };
        // ---- this warp's stream of weight chunks (see the comment above the kernel). The cursor is
        //      warp-uniform (every lane computes it); lane 0 issues. The stream is a sequence of
        //      segments (a phase-1 unit: gate and up row groups; a phase-2 row group), each issued in
        //      chunks of s_ch records.
        int cu = 0, cu_slot = 0;                 // items consumed, slot of the next one
        uint32_t cu_par = 0;                     // parity of that slot's next fill
        int iss = 0, is_slot = 0;                // items issued, slot of the next one
        const uint8_t *sa = nullptr, *sb = nullptr;  // segment sources: gate (or row group), up (or none)
        int s_left = 0;                          // records of the segment not yet issued
        int s_ch = 0;                            // records per chunk
        uint32_t s_b = 0;                        // bytes of a full chunk of one source
        bool s_live = false;
        // phase 1: the CTA's units u = 0 .. nc-1 (list entries c + u * ncta), kc_h records of gate and
        // up each (nch chunks of ch1). With at least NW units (p1_sk) every warp takes a contiguous
        // run of records [C0, C1) = [w * T / NW, (w + 1) * T / NW) of the concatenated list,
        // T = nc * kc_h: a unit cut by a run boundary has two parts, the end part as the first item
        // of warp w + 1 and the start part as the last item of warp w. Otherwise each unit is split
        // into p1_S equal parts of whole chunks (p1_S > 1 only with one activation group), dealt
        // round-robin: warp w takes parts w, w + NW, ... of the list of nc * p1_S parts.
        bool p1_sk = false;
        int p1_S = 1, p1_items = 0, p1_nch = 1, p1_C0 = 0, p1_C1 = 0;
        int p1_it = 0;                           // next item (of this warp) to issue
        struct P1Item {
            int u, k0, k1;  // unit, record range [k0, k1) of its kc_h
        };
        auto p1_item = [&](int i) -> P1Item {
            P1Item t;
            if (p1_sk) {
                t.u = p1_C0 / a.kc_h + i;
                t.k0 = max(p1_C0 - t.u * a.kc_h, 0);
                t.k1 = min(p1_C1 - t.u * a.kc_h, a.kc_h);
            } else {
                const int it = warp + i * NW, part = it % p1_S;
                t.u = it / p1_S;
                t.k0 = part * p1_nch / p1_S * ch1;
                t.k1 = min((part + 1) * p1_nch / p1_S * ch1, a.kc_h);
            }
            return t;
        };
        int q2 = 0, q2end = 0, j2 = 0, oct2 = 0; // phase 2: next unit (and its expert, octet), range end
        int nUl = 0;
        uint8_t *const my_slots = ring + (size_t)warp * a.nsw * a.slot_bytes;
        uint64_t *const my_full = full + warp * a.nsw;
        // Next segment of the stream: a phase-1 unit (gate and up row groups of an f-tile), then the
        // phase-2 row groups oct * r2 + warp of the CTA's units. Once per segment (not per chunk).
        auto next_segment = [&]() {
            s_live = true;
            if (p1_it < p1_items) {
                const P1Item t = p1_item(p1_it);
                const P1Tile pt = p1_tile(c + t.u * a.ncta, a.nft_s, a.nft);
                const uint8_t *base = pt.sh ? a.sgu : a.gu + (int64_t)ms->ulist[pt.jrow] * a.gu_stride;
                const int r0 = t.k0, r1 = t.k1;
                sa = base + (int64_t)(2 * pt.ft) * gb_h + (int64_t)r0 * a.rec;
                sb = sa + gb_h;
                s_left = r1 - r0;
                s_ch = ch1;
                ++p1_it;
                return;
            }
            // units whose octet has no row group for this warp are skipped (only an expert's last octet)
            while (q2 < q2end && warp >= min(a.r2, a.ng_d - oct2 * a.r2)) {
                ++q2;
                if (++oct2 == a.noct) {
                    oct2 = 0;
                    ++j2;
                }
            }
            if (q2 >= q2end) {
                s_live = false;
                return;
            }
            const bool sh = j2 == nUl;
            s_left = sh ? a.kc_fs : a.kc_f;
            const uint8_t *base = sh ? a.sdn : a.dn + (int64_t)ms->ulist[j2] * a.dn_stride;
            sa = base + (int64_t)(oct2 * a.r2 + warp) * s_left * a.rec;
            sb = nullptr;
            s_ch = ch2;
            ++q2;
            if (++oct2 == a.noct) {
                oct2 = 0;
                ++j2;
            }
        };
        // Issues the stream's next chunk (if any) into slot is_slot; warp-uniform.
        auto issue_next = [&]() {
            if (s_left <= 0) {
                next_segment();
                if (!s_live) return;
                s_b = (uint32_t)s_ch * a.rec;
            }
            const uint32_t b = s_left >= s_ch ? s_b : (uint32_t)s_left * a.rec;
            if (lane == 0) {
                uint8_t *dst = my_slots + (size_t)is_slot * a.slot_bytes;
                uint64_t *fb = my_full + is_slot;
                const uint64_t pol = l2_evict_first();  // weights are read once per launch
                fence_proxy_async_shared();              // this warp's reads of the slot come first
                mbar_arrive_expect_tx(fb, sb ? 2 * b : b);
                bulk_g2s_hint(dst, sa, b, fb, pol);
                if (sb) bulk_g2s_hint(dst + b, sb, b, fb, pol);
            }
            __syncwarp();
            sa += b;
            if (sb) sb += b;
            s_left -= s_ch;
            ++iss;
            if (++is_slot == a.nsw) is_slot = 0;
        };
        // trace builds: per-phase durations of warp 0 accumulated in registers: [0] phase-1 data waits,
        // [1] phase-1 MMA sections, [2] phase-2 data waits, [3] phase-1 refills, [4] phase-1 chunks
        unsigned long long tacc[15] = {};  // [10] phase-1 epilogues, [11] phase-1 unit starts, [12] phase-2 epilogues  // [5..9]: phase-2 MMA, refills, setups, units, experts
        int tslot = 0;
        // Waits for the next item; a warp whose data never came stops issuing and keeps its copies
        // in the drain at exit.
        auto take_item = [&]() -> const uint8_t * {
            check_abort();
            [[maybe_unused]] const unsigned long long tw0 = BFP_TRACE_NOW();
            if (!bad && !__all_sync(0xffffffffu, mbar_wait(my_full + cu_slot, cu_par, a.wait_data, vflags)))
                abort_warp();
            __syncwarp();  // lanes leave the wait at different polls: reconverge before the MMAs
            tacc[tslot] += BFP_TRACE_NOW() - tw0;
            return my_slots + (size_t)cu_slot * a.slot_bytes;
        };
        // Done with the item: refill its slot with the item nsw further on. After an abort the
        // item counts as unconsumed, so the drain at exit waits for its copy.
        auto give_item = [&]() {
            __syncwarp();
            if (bad) return;
            issue_next();
            ++cu;
            if (++cu_slot == a.nsw) {
                cu_slot = 0;
                cu_par ^= 1u;
            }
        };

        // Grid barrier over the consumer threads of every CTA, on a workspace counter.
        // Returns false on abort (same answer in every consumer thread of the CTA).
        auto grid_barrier = [&](uint32_t *counter) -> bool {
            bar_sync(1, NC);
            bool ok = true;
            if (tid == 0) {
                // the CTA barrier orders every thread's writes before this release (cumulative at gpu scope)
                red_release_add(counter, 1u);
                ok = wait_counter(counter, (uint32_t)a.ncta, a.wait);
            }
            const bool r = !bar_or(1, NC, !ok || bad);
            __syncwarp();  // thread 0 waited alone: reconverge, or later warp collectives run many times slower
            return r;
        };

        // ---- the MoE input rows (x, or bf16(RMSNorm(h)) in stack mode, normalised in place first)
        if (!__all_sync(0xffffffffu, mbar_wait(&ms->stage_full, 0u, a.wait_data, nullptr))) bad = true;
        __syncwarp();
        STAMP(2);  // stage landed
        uint16_t *const xs = reinterpret_cast<uint16_t *>(stage);
        if (a.norm)
            act_rows_prepare<NC>(xs, LDXS, a.M, a.H, true, a.eps, ms->shift_x, ms->inv, ms->red, 1, warp, lane);

        // ---- phase-1 unit (run by one warp): f-tile of gate and up over all of k; h = silu(gate) * up
        //      for the rows in the unit's row mask, to the workspace; row maxima of |h| to hmax.
        auto run_p1_item = [&](int i) {
            [[maybe_unused]] const unsigned long long tu0 = BFP_TRACE_NOW();
            const P1Item t = p1_item(i);
            const int r0 = t.k0, r1 = t.k1;
            const P1Tile pt = p1_tile(c + t.u * a.ncta, a.nft_s, a.nft);
            const int er = pt.sh ? kMaxExperts : ms->ulist[pt.jrow];  // expert row of emask / eslot
            const uint32_t rowmask = ms->emask[er];
            const uint32_t gm = (((rowmask & 0xFFu) ? 1u : 0u) | ((rowmask & 0xFF00u) ? 2u : 0u)) & ngrp_rows;
            bool both = false;
            if constexpr (NGRP == 2) both = gm == 3u;
            const int gsel = gm == 2u ? 1 : 0;  // the one activation group holding every row otherwise
            const uint2 *fg = frag2 + (int64_t)gsel * a.kbp_h * kWarp;
            float acc[2][NGRP][4];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int gg = 0; gg < NGRP; ++gg)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[r][gg][i] = 0.f;
            float a1[2][1][4] = {};
            tacc[11] += BFP_TRACE_NOW() - tu0;
            // each chunk: n gate records, then n up records; one loop per group count, so that each
            // keeps only its own accumulators live
            if (both) {
                for (int k0 = r0; k0 < r1; k0 += ch1) {
                    const int n = min(ch1, r1 - k0);
                    const uint8_t *sp = take_item();
                    if (!bad)
                        for (int ch = 0; ch < n; ++ch) {
                            const uint8_t *recs[2] = {sp + (size_t)ch * a.rec, sp + (size_t)(n + ch) * a.rec};
                            mma_records<FMT, NGRP, 2, false>(recs, frag2, nullptr, a.kbp_h, (k0 + ch) * CB, lane,
                                                             ms->esc[warp], acc);
                        }
                    tacc[13] += 1;
                    give_item();
                }
            } else {
                for (int k0 = r0; k0 < r1; k0 += ch1) {
                    const int n = min(ch1, r1 - k0);
                    const uint8_t *sp = take_item();
                    [[maybe_unused]] const unsigned long long tm0 = BFP_TRACE_NOW();
                    if (!bad)
                        for (int ch = 0; ch < n; ++ch) {
                            const uint8_t *recs[2] = {sp + (size_t)ch * a.rec, sp + (size_t)(n + ch) * a.rec};
                            mma_records<FMT, 1, 2, false>(recs, fg, nullptr, a.kbp_h, (k0 + ch) * CB, lane,
                                                          ms->esc[warp], a1);
                        }
                    __syncwarp();
                    tacc[1] += BFP_TRACE_NOW() - tm0;
                    tacc[4] += 1;
                    [[maybe_unused]] const unsigned long long tg0 = BFP_TRACE_NOW();
                    give_item();
                    tacc[3] += BFP_TRACE_NOW() - tg0;
                }
            }
            if (bad) return;
            if (p1_sk && (t.k0 > 0 || t.k1 < a.kc_h)) {
                // a unit cut by a run boundary: the end part (first item of warp w) goes to the
                // scratch of boundary w - 1; the start part (last item of warp w) waits for the tile
                // of boundary w, adds it and writes the unit's results
                if (t.k0 > 0) {
                    float *dst = a.p1part + ((size_t)c * (NW - 1) + (warp - 1)) * kP1PartFloats;
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int gg = 0; gg < NGRP; ++gg)
#pragma unroll
                            for (int i4 = 0; i4 < 4; ++i4)
                                dst[((r * NGRP + gg) * 4 + i4) * kWarp + lane] =
                                    both ? acc[r][gg][i4] : (gg == 0 ? a1[r][0][i4] : 0.f);
                    __threadfence();  // the tile reaches L2 before the flag is seen
                    __syncwarp();
                    if (lane == 0) reinterpret_cast<volatile int *>(ms->p1flag)[warp - 1] = 1;
                    return;
                }
                bool ok = true;
                if (lane == 0) {
                    const volatile int *f = ms->p1flag + warp;
                    ok = *f != 0;
                    const uint64_t tw0 = global_ns();
                    for (int64_t k = 1; !ok && k < a.wait_data.iters; ++k) {
                        if (vflags[0] || global_ns() - tw0 > a.wait_data.nanos) break;
                        ok = *f != 0;
                    }
                }
                if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
                    abort_warp();
                    return;
                }
                __syncwarp();
                __threadfence_block();
                const float *src = a.p1part + ((size_t)c * (NW - 1) + warp) * kP1PartFloats;
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int gg = 0; gg < NGRP; ++gg)
#pragma unroll
                        for (int i4 = 0; i4 < 4; ++i4) {
                            const float v = __ldcg(src + ((r * NGRP + gg) * 4 + i4) * kWarp + lane);
                            if (both)
                                acc[r][gg][i4] += v;
                            else if (gg == 0)
                                a1[r][0][i4] += v;
                        }
            }
            if constexpr (NGRP == 1) {
                if (!p1_sk && p1_S > 1) {
                    const int it = warp + i * NW, ui = t.u;
                    // split unit: store this part's tile; the last part to finish adds the parts in
                    // order (it < NW items, each with its scratch tile) and writes the unit's results
                    float *mine = scr + (size_t)it * 256;
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int i4 = 0; i4 < 4; ++i4) mine[(r * 4 + i4) * kWarp + lane] = a1[r][0][i4];
                    __syncwarp();
                    int last = 0;
                    if (lane == 0) {
                        __threadfence_block();
                        last = atomicAdd(&ms->p1cnt[ui], 1) == p1_S - 1;
                    }
                    if (!__shfl_sync(0xffffffffu, last, 0)) return;
                    __syncwarp();
                    __threadfence_block();
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int i4 = 0; i4 < 4; ++i4) {
                            float v = 0.f;
                            for (int q = 0; q < p1_S; ++q) v += scr[(size_t)(ui * p1_S + q) * 256 + (r * 4 + i4) * kWarp + lane];
                            a1[r][0][i4] = v;
                        }
                }
            }
            [[maybe_unused]] const unsigned long long te0 = BFP_TRACE_NOW();
#pragma unroll
            for (int gg = 0; gg < NGRP; ++gg) {
                if (!both && gg > 0) continue;
                const int grp = both ? gg : gsel;
                uint32_t me = 0u, mo = 0u;  // max |h| of rows 8 grp + 2 (lane & 3) and the next one
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float va = both ? acc[0][gg][i] : a1[0][0][i];
                    const float vb = both ? acc[1][gg][i] : a1[1][0][i];
                    const int r = acc_xrow(lane, grp, i);
                    if (r < a.M && ((rowmask >> r) & 1u)) {
                        const int sh = 24 - (MB - 1) - ms->shift_x[r];
                        const float ga = mul_pow2(va, sh), ub = mul_pow2(vb, sh);
                        const float hv = ga / (1.0f + expf(-ga)) * ub;  // silu(gate) * up
                        const int f = pt.ft * 16 + acc_wrow(lane, i);
                        a.hbuf[((int64_t)r * (a.K + 1) + ms->eslot[er][r]) * a.Fmax + f] = hv;
                        const uint32_t hb = __float_as_uint(fabsf(hv));
                        if (i & 1)
                            mo = max(mo, hb);
                        else
                            me = max(me, hb);
                    }
                }
                // the eight lanes with equal lane & 3 hold the same two rows
#pragma unroll
                for (int o = 4; o < kWarp; o <<= 1) {
                    me = max(me, __shfl_xor_sync(0xffffffffu, me, o));
                    mo = max(mo, __shfl_xor_sync(0xffffffffu, mo, o));
                }
                if (lane < 4) {
                    const int re = 8 * grp + 2 * lane, ro = re + 1;
                    if (re < a.M && ((rowmask >> re) & 1u))
                        atomicMax(&a.hmax[re * (a.K + 1) + ms->eslot[er][re]], me);
                    if (ro < a.M && ((rowmask >> ro) & 1u))
                        atomicMax(&a.hmax[ro * (a.K + 1) + ms->eslot[er][ro]], mo);
                }
            }
            __syncwarp();
            tacc[10] += BFP_TRACE_NOW() - te0;
        };

        // ---- 1. router rows: fp32 logits of this CTA's router rows (and the shared-gate row) for every
        //      input row, on the tensor cores: A = the bf16 input rows (m16 x k16 per step, rows >= M
        //      zero), B = the bf16 router rows (8 per tile, n8), k split over the warps; the warps'
        //      tiles meet in the fragment area (free until the fragments are built) and are added in
        //      warp order.
        if (rr1 > rr0) {
            const uint16_t *wr = reinterpret_cast<const uint16_t *>(stage + a.stage_r);
            const int nrows = rr1 - rr0, nt = (nrows + 7) / 8;
            const int ksteps = a.H / 16;
            float *rpart = reinterpret_cast<float *>(frag);  // [nt][NW][32 lanes][4]
            if (!bad) {
                const int g = lane >> 2, t = lane & 3;
                const int ks0 = warp * ksteps / NW, ks1 = (warp + 1) * ksteps / NW;
                const bool r0v = g < a.M, r1v = g + 8 < a.M;
                const uint16_t *xa = xs + (int64_t)g * LDXS + 2 * t;
                const uint16_t *xb = xa + (int64_t)8 * LDXS;
                for (int tile = 0; tile < nt; ++tile) {
                    const int n = 8 * tile + g;  // router row of this lane's B column
                    const bool nv = n < nrows;
                    const uint16_t *wb = wr + (int64_t)n * a.H + 2 * t;
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int ks = ks0; ks < ks1; ++ks) {
                        const int kk = 16 * ks;
                        uint32_t af[4];
                        af[0] = r0v ? *reinterpret_cast<const uint32_t *>(xa + kk) : 0u;
                        af[1] = r1v ? *reinterpret_cast<const uint32_t *>(xb + kk) : 0u;
                        af[2] = r0v ? *reinterpret_cast<const uint32_t *>(xa + kk + 8) : 0u;
                        af[3] = r1v ? *reinterpret_cast<const uint32_t *>(xb + kk + 8) : 0u;
                        const uint32_t b0 = nv ? *reinterpret_cast<const uint32_t *>(wb + kk) : 0u;
                        const uint32_t b1 = nv ? *reinterpret_cast<const uint32_t *>(wb + kk + 8) : 0u;
                        mma16816_bf16(d, af, b0, b1);
                    }
                    *reinterpret_cast<float4 *>(rpart + ((size_t)(tile * NW + warp) * kWarp + lane) * 4) =
                        make_float4(d[0], d[1], d[2], d[3]);
                }
            }
            STAMP(96);  // router tiles stored
            bar_sync(1, NC);
            const int LS = logit_stride(a.E);
            for (int idx = tid; !bad && idx < nrows * a.M; idx += NC) {
                const int i = idx / a.M, r = idx % a.M;
                const int tile = i >> 3, col = i & 7;
                const int ln = 4 * (r & 7) + (col >> 1), reg = ((r >> 3) << 1) | (col & 1);  // D[r][col]
                float acc = 0.f;
                for (int w = 0; w < NW; ++w) acc += rpart[((size_t)(tile * NW + w) * kWarp + ln) * 4 + reg];
                const int row = rr0 + i;
                if (row < a.E && a.rbias) acc += a.rbias[row];
                a.logits[(int64_t)r * LS + row] = acc;
            }
        }
        if (bar_or(1, NC, bad)) {
            abort_all();
            goto done;
        }
        STAMP(97);  // logits written
        // ---- two groups of warps from here to the end of the routing:
        //      warps 0 .. NR-1: warp 0 publishes this CTA's logits (its release waits for them to reach
        //        L2); then every CTA's router rows, top-k and the union (named barrier 3);
        //      warps NR .. NW-1: the activation fragments for phase 1 (named barrier 2), which nothing
        //        needs before the first weight chunks land.
        {
            constexpr int NR = NW / 2;                     // routing warps
            constexpr int RPW = (kMaxRows + NR - 1) / NR;  // rows per routing warp
            if (warp >= NR) {
                BFP_TRACE_AT_T(110, NR * kWarp);
                constexpr int NF = NC - NR * kWarp;
                if (!a.norm)
                    act_rows_prepare<NF>(xs, LDXS, a.M, a.H, false, a.eps, ms->shift_x, ms->inv, ms->red, 2,
                                         warp - NR, lane);
                BFP_TRACE_AT_T(111, NR * kWarp);
                act_rows_frags<NF>(xs, LDXS, a.M, a.H, a.kbp_h, NGRP, ms->shift_x, frag, 2, tid - NR * kWarp,
                                   warp - NR, lane);
                STAMP(1);  // activation fragments built
                BFP_TRACE_AT_T(112, NR * kWarp);
            } else {
                bool ok = true;
                if (tid == 0) {
                    red_release_add(&a.ctrl[0], 1u);  // after the CTA barrier: every thread's logits
                    STAMP(98);
                    ok = wait_counter(&a.ctrl[0], (uint32_t)a.ncta, a.wait);
                    STAMP(99);
                }
                if (bar_or(3, NR * kWarp, !ok)) bad = true;
                __syncwarp();  // thread 0 polled alone
                STAMP(100);
                STAMP(5);  // every CTA's router rows published
                // Top-k per row, on the logits every CTA wrote before the router counter (read from
                // L2); warp w takes rows w and w + NR, as two independent chains. Lane l holds experts
                // 8l .. 8l+7 and first sorts them (key descending, index ascending among equal keys);
                // each round the lanes offer their heads, the largest key wins and among equal keys the
                // lowest lane, i.e. the lowest expert index (ties go to the lower index); lane s keeps
                // the slot-s winner. Slot 0 is the row maximum, so p_s = exp(l_s - l_0) and
                // w_s = p_s / sum of p.
                const int LS = logit_stride(a.E);
                uint32_t key[RPW][8];
                int qi[RPW][8];
                float gate_logit[RPW];
#pragma unroll
                for (int j = 0; j < RPW; ++j) {
                    const int r = warp + NR * j;
                    const float *row = a.logits + (int64_t)r * LS;
                    if (bad || r >= a.M) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) key[j][q] = 0u;
                        gate_logit[j] = 0.f;
                    } else if (8 * lane + 8 <= a.E) {
                        const float4 v0 = __ldcg(reinterpret_cast<const float4 *>(row + 8 * lane));
                        const float4 v1 = __ldcg(reinterpret_cast<const float4 *>(row + 8 * lane + 4));
                        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                        for (int q = 0; q < 8; ++q) key[j][q] = order_key(v[q]);
                        gate_logit[j] = __ldcg(row + a.E);
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int e = 8 * lane + q;
                            key[j][q] = e < a.E ? order_key(__ldcg(row + e)) : 0u;  // 0: below any logit
                        }
                        gate_logit[j] = __ldcg(row + a.E);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) qi[j][q] = q;
                    sort8_desc(key[j], qi[j]);
                }
                STAMP(102);  // logits loaded and sorted
                int my_e[RPW] = {};
                float my_l[RPW] = {};
                for (int s = 0; s < a.K; ++s) {
#pragma unroll
                    for (int j = 0; j < RPW; ++j) {
                        const uint32_t kmax = __reduce_max_sync(0xffffffffu, key[j][0]);
                        const uint32_t bal = __ballot_sync(0xffffffffu, key[j][0] == kmax);
                        const int wl = __ffs(bal) - 1;
                        const int q = __shfl_sync(0xffffffffu, qi[j][0], wl);
                        if (lane == s) {
                            my_e[j] = min(8 * wl + q, a.E - 1);  // < E: missing experts' keys are below any logit
                            my_l[j] = key_value(kmax);
                        }
                        const bool win = lane == wl;
#pragma unroll
                        for (int i = 0; i < 7; ++i) {
                            key[j][i] = win ? key[j][i + 1] : key[j][i];
                            qi[j][i] = win ? qi[j][i + 1] : qi[j][i];
                        }
                        key[j][7] = win ? 0u : key[j][7];
                    }
                }
                STAMP(103);  // rounds done
#pragma unroll
                for (int j = 0; j < RPW; ++j) {
                    const int r = warp + NR * j;
                    const float l0 = __shfl_sync(0xffffffffu, my_l[j], 0);
                    const float p = lane < a.K ? __expf(my_l[j] - l0) : 0.f;
                    float psum = p;
#pragma unroll
                    for (int o = 1; o < kWarp; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
                    if (!bad && r < a.M) {
                        if (lane < a.K) {
                            const float w = __fdividef(p, psum);
                            const int e = my_e[j];
                            ms->tk_idx[r][lane] = e;
                            ms->tk_w[r][lane] = w;
                            atomicOr(&ms->bitmap[e >> 5], 1u << (e & 31));
                            atomicOr(&ms->emask[e], 1u << r);
                            ms->eslot[e][r] = (int8_t)lane;
                            if (c == 0) {
                                if (a.topk_idx) a.topk_idx[r * a.K + lane] = e;
                                if (a.topk_w) a.topk_w[r * a.K + lane] = w;
                            }
                        }
                        if (lane == 0) ms->gate_w[r] = __fdividef(1.0f, 1.0f + __expf(-gate_logit[j]));
                    }
                }
                STAMP(27);  // top-k of warp 0's rows done
                bar_sync(3, NR * kWarp);
                STAMP(105);
                // The union U (ascending expert index, the shared expert last) and this CTA's phase-2
                // range, one routing thread per expert: an exclusive scan of (member, cost of its
                // units) over the experts gives each member its position in U and the cost of the
                // units before it; the member whose cost interval holds one of the CTA's share
                // boundaries X = total * c / ncta, total * (c + 1) / ncta writes the first unit that
                // starts at or after X.
                {
                    static_assert(NR * kWarp == kMaxExperts, "one routing thread per expert");
                    const int e = tid;
                    const bool in_u = e < a.E && ((ms->bitmap[e >> 5] >> (e & 31)) & 1u);
                    const int cu = in_u ? p2_cost(ms->emask[e]) : 0;  // cost of one unit of expert e
                    const uint32_t v = in_u ? (1u << 16) | (uint32_t)(a.noct * cu) : 0u;
                    uint32_t incl = v;
#pragma unroll
                    for (int o = 1; o < kWarp; o <<= 1) {
                        const uint32_t t2 = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += t2;
                    }
                    if (lane == kWarp - 1) ms->wsum[warp] = incl;
                    bar_sync(3, NR * kWarp);
                    uint32_t before = 0, total = 0;
#pragma unroll
                    for (int w2 = 0; w2 < NR; ++w2) {
                        const uint32_t ws2 = ms->wsum[w2];
                        before += w2 < warp ? ws2 : 0u;
                        total += ws2;
                    }
                    const uint32_t ex = before + incl - v;
                    const int pos = (int)(ex >> 16), cum = (int)(ex & 0xFFFFu);
                    const int nU = (int)(total >> 16), cost_r = (int)(total & 0xFFFFu);
                    const int cu_s = p2_cost(ms->emask[kMaxExperts]);
                    const int tot = cost_r + a.noct * cu_s;
                    if (in_u) ms->ulist[pos] = (int16_t)e;
                    if (e == 0) {
                        ms->nU = nU;
                        ms->ulist[nU] = (int16_t)a.E;
                    }
                    STAMP(106);
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int X = tot * (c + i) / a.ncta;
                        if (in_u && cum <= X && X < cum + a.noct * cu) {
                            const int o = (X - cum + cu - 1) / cu;
                            ms->p2q[i] = o < a.noct ? pos * a.noct + o : (pos + 1) * a.noct;
                        }
                        if (e == 0 && cost_r <= X && X < tot) {
                            const int o = (X - cost_r + cu_s - 1) / cu_s;
                            ms->p2q[i] = o < a.noct ? nU * a.noct + o : (nU + 1) * a.noct;
                        }
                        if (e == 0 && X >= tot) ms->p2q[i] = (nU + 1) * a.noct;
                    }
                }
            }
            // every warp: the fragments, the union and the phase-2 range are in shared memory
            if (bar_or(1, NC, bad)) {
                abort_all();
                goto done;
            }
        }
        STAMP(109);
        STAMP(6);  // top-k + union done
        // this warp's stream: its units and the CTA's phase-2 range are known now; fill its slots
        // (every warp is past its reads of the stage, which the first slots may overlap)
        nUl = ms->nU;
        {
            const int p1_total = a.nft_s + nUl * a.nft;
            const int nc = c < p1_total ? (p1_total - c + a.ncta - 1) / a.ncta : 0;  // this CTA's units
            p1_nch = (a.kc_h + ch1 - 1) / ch1;
            // every run at least one unit long (a unit has at most two parts), and room for the tiles
            p1_sk = a.p1part != nullptr && nc >= NW;
            if (p1_sk) {
                // Runs of equal cost: a record of a unit with rows in both activation groups costs 5
                // (two MMAs per block), one of a single-group unit 4. Weighted only when every run
                // still spans at least one unit of the heavier kind (so no unit has three parts).
                auto unit_wt = [&](int u) {
                    if (u >= nc) return 0;
                    if (NGRP == 1) return 4;
                    const P1Tile pt = p1_tile(c + u * a.ncta, a.nft_s, a.nft);
                    const uint32_t m = ms->emask[pt.sh ? kMaxExperts : ms->ulist[pt.jrow]];
                    return ((m & 0xFFu) && (m & 0xFF00u)) ? 5 : 4;
                };
                int W = 0;
                for (int u = lane; u < nc; u += kWarp) W += unit_wt(u);
                W = __reduce_add_sync(0xffffffffu, W);
                const int T = nc * a.kc_h;  // records
                if (NGRP == 2 && W >= 5 * NW) {
                    // record position of weight X (in record-weight units, 0 <= X <= W * kc_h): the unit
                    // holding X and the whole records of it before X
                    const int X0 = (int)((int64_t)warp * W * a.kc_h / NW);
                    const int X1 = (int)((int64_t)(warp + 1) * W * a.kc_h / NW);
                    int P0 = T, P1 = T, carry = 0;
                    for (int u0 = 0; u0 < nc; u0 += kWarp) {
                        const int u = u0 + lane, wt = unit_wt(u), span = wt * a.kc_h;
                        int incl = span;
#pragma unroll
                        for (int o = 1; o < kWarp; o <<= 1) {
                            const int t2 = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl += t2;
                        }
                        const int beg = carry + incl - span;
                        const uint32_t b0 = __ballot_sync(0xffffffffu, u < nc && beg <= X0 && X0 < beg + span);
                        const uint32_t b1 = __ballot_sync(0xffffffffu, u < nc && beg <= X1 && X1 < beg + span);
                        const int pos0 = u * a.kc_h + (X0 - beg) / max(wt, 1), pos1 = u * a.kc_h + (X1 - beg) / max(wt, 1);
                        if (b0) P0 = __shfl_sync(0xffffffffu, pos0, __ffs(b0) - 1);
                        if (b1) P1 = __shfl_sync(0xffffffffu, pos1, __ffs(b1) - 1);
                        carry += __shfl_sync(0xffffffffu, incl, kWarp - 1);
                    }
                    p1_C0 = P0;
                    p1_C1 = P1;
                } else {
                    p1_C0 = warp * T / NW;
                    p1_C1 = (warp + 1) * T / NW;
                }
                p1_items = p1_C1 > p1_C0 ? (p1_C1 - 1) / a.kc_h - p1_C0 / a.kc_h + 1 : 0;
            } else {
                if constexpr (NGRP == 1) {
                    while (nc > 0 && nc * p1_S * 2 <= NW && p1_S * 2 <= p1_nch) p1_S *= 2;
                }
                p1_items = warp < nc * p1_S ? (nc * p1_S - warp + NW - 1) / NW : 0;
            }
            p1_it = 0;
        }
        q2end = (int)ms->p2q[1];
        q2 = (int)ms->p2q[0];
        j2 = q2 / a.noct;
        oct2 = q2 % a.noct;
        for (int i = 0; i < a.nsw; ++i) issue_next();

        // ---- 4. phase 1: this warp's units of the CTA's list [shared-expert f-tiles, routed f-tiles]
        {
            for (int i = 0; i < p1_items; ++i) {
                if (i == 1) STAMP(21);  // warp 0: second item start
                run_p1_item(i);
            }
            STAMP(8);  // warp 0: phase-1 units done
            BFP_TRACE_WARP(64);  // every warp: phase-1 items done
            BFP_TRACE_WARP_SET(80, tacc[13] * 1000 + tacc[4]);  // ... its two-group and one-group chunks
            tslot = 2;
            if (!grid_barrier(&a.ctrl[2])) {  // every CTA's h and row maxima written
                abort_all();
                goto done;
            }
            STAMP(9);  // phase-1 grid barrier passed
            if (c == 0 && tid == 0) a.ctrl[0] = 0u;  // every CTA is past the router wait
        }

        // ---- 5. down projection. Per expert, the rows that chose it become the columns 0..n-1 of
        //      its h fragments (routing weight folded in, fp16 hi + lo parts): n <= 4: hi in columns
        //      c, lo in columns c + 4 of one 8-column MMA (summed at the end); n <= 8: hi and lo
        //      fragments, two MMAs; more rows: two column groups. The CTA takes its units in
        //      batches: the experts of the next units whose fragments fit in the fragment area
        //      together (at most kP2Batch) are set up in one pass, then their units run with no
        //      CTA barrier in between.
        {
            const int nU = ms->nU;
            const int q0 = (int)ms->p2q[0], q1 = (int)ms->p2q[1];
            int p2n = 0;  // phase-2 units done by this CTA (trace stamps)
            uint32_t *hfrag = frag;  // x fragments are dead once phase 1 is done
            int q = q0;
            while (q < q1) {
                [[maybe_unused]] const unsigned long long tsu0 = BFP_TRACE_NOW();
                // every warp is done with the previous batch's fragments
                if (bar_or(1, NC, bad)) {
                    abort_all();
                    goto done;
                }
                if (tid == 0) {
                    int nb = 0, qe = q, off = 0;
                    while (qe < q1 && nb < kP2Batch) {
                        const int j = qe / a.noct;
                        const bool sh = j == nU;
                        const int er = sh ? kMaxExperts : ms->ulist[j];
                        const int nr = __popc(ms->emask[er]);
                        const int kbp = sh ? a.kbp_fs : a.kbp_f;
                        const int parts = nr <= 4 ? 1 : (nr <= 8 ? 2 : 4);
                        const int words = parts * kbp * 2 * kWarp;
                        if (nb > 0 && off + words > a.frag_bytes / 4) break;  // the first one always fits
                        P2Entry &pe = ms->p2b[nb];
                        pe.j = j;
                        pe.er = er;
                        pe.nr = nr;
                        pe.parts = parts;
                        pe.off = off;
                        pe.qend = min((j + 1) * a.noct, q1);
                        off += words;
                        qe = pe.qend;
                        ++nb;
                    }
                    ms->p2nb = nb;
                }
                bar_sync(1, NC);
                __syncwarp();
                const int nb = ms->p2nb;
                // every fragment word of the batch, once: a thread takes 4 consecutive values of one
                // column in one block and writes their hi and lo words (zeros for padding columns and
                // blocks), so no separate clearing pass is needed
                {
                    int items = 0;
                    for (int bi = 0; bi < nb; ++bi) {
                        const P2Entry &pe = ms->p2b[bi];
                        const int kbp = pe.j == nU ? a.kbp_fs : a.kbp_f;
                        items += (pe.parts == 1 ? 4 : 8 * (pe.parts / 2)) * kbp * 4;
                    }
                    for (int it = tid; it < items; it += NC) {
                        int bi = 0, base = 0, cols = 0, kbp = 0;
                        for (;; ++bi) {
                            const P2Entry &pe = ms->p2b[bi];
                            kbp = pe.j == nU ? a.kbp_fs : a.kbp_f;
                            cols = pe.parts == 1 ? 4 : 8 * (pe.parts / 2);
                            if (it - base < cols * kbp * 4 || bi == nb - 1) break;
                            base += cols * kbp * 4;
                        }
                        const P2Entry &pe = ms->p2b[bi];
                        const bool sh = pe.j == nU;
                        const int rem0 = it - base, col = rem0 / (kbp * 4), rem = rem0 - col * kbp * 4;
                        const int blk = rem >> 2, qq = rem & 3;
                        const int Fe = sh ? a.Fs : a.F;
                        uint32_t *hf = hfrag + pe.off;
                        const int lo_off = (pe.parts == 4 ? 2 : 1) * kbp * 2 * kWarp;  // words
                        uint32_t hw2[2] = {0u, 0u}, lw2[2] = {0u, 0u};
                        if (col < pe.nr && blk < Fe / 16) {
                            const uint32_t rowmask = ms->emask[pe.er];
                            const int r = (int)__fns(rowmask, 0, col + 1);
                            const int slot = ms->eslot[pe.er][r];
                            const float w = sh ? ms->gate_w[r] : ms->tk_w[r][slot];
                            const uint32_t hm = __ldcg(&a.hmax[r * (a.K + 1) + slot]);
                            const float4 v4 = __ldcg(reinterpret_cast<const float4 *>(
                                                         a.hbuf + ((int64_t)r * (a.K + 1) + slot) * a.Fmax) +
                                                     rem);
                            // routing weight folded into h; per-row power-of-two scale into fp16 range
                            // from the phase-1 maximum (weights are positive, so max |w h| = w max |h|,
                            // rounding included)
                            const int shift = frag_shift(w * __uint_as_float(hm));
                            const float sc = pow2f(shift);
                            const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                            for (int pr = 0; pr < 2; ++pr) {
                                const float v0 = vv[2 * pr] * w * sc, v1 = vv[2 * pr + 1] * w * sc;
                                const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
                                __half2 hh = __halves2half2(h0, h1);
                                hw2[pr] = *reinterpret_cast<uint32_t *>(&hh);
                                lw2[pr] = pack_half2(v0 - __half2float(h0), v1 - __half2float(h1));
                            }
                            if (blk == 0 && qq == 0) {
                                ms->p2row[bi][col] = (int8_t)r;
                                ms->p2shift[bi][col] = shift;
                            }
                        }
#pragma unroll
                        for (int pr = 0; pr < 2; ++pr) {
                            hf[frag_word(col, blk, 2 * qq + pr, kbp)] = hw2[pr];
                            if (pe.parts == 1)
                                hf[frag_word(col + 4, blk, 2 * qq + pr, kbp)] = lw2[pr];
                            else
                                hf[lo_off + frag_word(col, blk, 2 * qq + pr, kbp)] = lw2[pr];
                        }
                    }
                }
                bar_sync(1, NC);
                if (p2n == 0) STAMP(10);  // first batch's h fragments ready
                tacc[7] += BFP_TRACE_NOW() - tsu0;
                tacc[9] += nb;
                for (int bi = 0; bi < nb; ++bi) {
                    const P2Entry &pe = ms->p2b[bi];
                    const int j = pe.j;
                    const bool sh = j == nU;
                    const int kc = sh ? a.kc_fs : a.kc_f, kbp = sh ? a.kbp_fs : a.kbp_f;
                    const int er = pe.er, nr = pe.nr;
                    const bool packed = pe.parts == 1;
                    const uint32_t *hfb = hfrag + pe.off;
                    for (; q < pe.qend; ++q) {
                        const int oct = q - j * a.noct;
                        tacc[8] += 1;
                        const int rg0 = oct * a.r2, nrg = min(a.r2, a.ng_d - rg0);
                        const bool mine = warp < nrg;
                        if (p2n == 0) STAMP(16);  // first phase-2 unit: start
                        float acc[1][NGRP][4];
#pragma unroll
                        for (int g = 0; g < NGRP; ++g)
#pragma unroll
                            for (int i = 0; i < 4; ++i) acc[0][g][i] = 0.f;
                        if (mine) {
                            // this warp's row group rg0 + warp of the unit, in chunks of ch2 records
                            const uint2 *hi2 = reinterpret_cast<const uint2 *>(hfb);
                            const uint2 *lo2 = hi2 + (pe.parts == 4 ? 2 : 1) * kbp * kWarp;
                            const bool both = NGRP == 2 && pe.parts == 4;
                            float a1[1][1][4] = {};
                            // one chunk loop per path (the path is fixed per expert)
                            if (both) {
                                for (int k0 = 0; k0 < kc; k0 += ch2) {
                                    const int n = min(ch2, kc - k0);
                                    const uint8_t *rb = take_item();
                                    if (p2n == 0) STAMP(17);  // ... its first data landed (warp 0)
                                    [[maybe_unused]] const unsigned long long tm0 = BFP_TRACE_NOW();
                                    if (!bad)
                                        for (int ch = 0; ch < n; ch += 2) {
                                            if (ch + 1 < n)
                                                mma_records_k<FMT, NGRP, 2, true>(rb + (size_t)ch * a.rec, a.rec, hi2, lo2, kbp,
                                                                                  (k0 + ch) * CB, lane, ms->esc[warp], acc[0]);
                                            else
                                                mma_records_k<FMT, NGRP, 1, true>(rb + (size_t)ch * a.rec, a.rec, hi2, lo2, kbp,
                                                                                  (k0 + ch) * CB, lane, ms->esc[warp], acc[0]);
                                        }
                                    __syncwarp();
                                    tacc[5] += BFP_TRACE_NOW() - tm0;
                                    [[maybe_unused]] const unsigned long long tg0 = BFP_TRACE_NOW();
                                    give_item();
                                    tacc[6] += BFP_TRACE_NOW() - tg0;
                                }
                            } else if (packed) {
                                // columns of group 0 only: hi in columns c, lo in columns c + 4
                                for (int k0 = 0; k0 < kc; k0 += ch2) {
                                    const int n = min(ch2, kc - k0);
                                    const uint8_t *rb = take_item();
                                    if (p2n == 0) STAMP(17);
                                    [[maybe_unused]] const unsigned long long tm0 = BFP_TRACE_NOW();
                                    if (!bad)
                                        for (int ch = 0; ch < n; ch += 2) {
                                            if (ch + 1 < n)
                                                mma_records_k<FMT, 1, 2, false>(rb + (size_t)ch * a.rec, a.rec, hi2, nullptr, kbp,
                                                                                (k0 + ch) * CB, lane, ms->esc[warp], a1[0]);
                                            else
                                                mma_records_k<FMT, 1, 1, false>(rb + (size_t)ch * a.rec, a.rec, hi2, nullptr, kbp,
                                                                                (k0 + ch) * CB, lane, ms->esc[warp], a1[0]);
                                        }
                                    __syncwarp();
                                    tacc[5] += BFP_TRACE_NOW() - tm0;
                                    [[maybe_unused]] const unsigned long long tg0 = BFP_TRACE_NOW();
                                    give_item();
                                    tacc[6] += BFP_TRACE_NOW() - tg0;
                                }
                            } else {
                                for (int k0 = 0; k0 < kc; k0 += ch2) {
                                    const int n = min(ch2, kc - k0);
                                    const uint8_t *rb = take_item();
                                    if (p2n == 0) STAMP(17);
                                    [[maybe_unused]] const unsigned long long tm0 = BFP_TRACE_NOW();
                                    if (!bad)
                                        for (int ch = 0; ch < n; ch += 2) {
                                            if (ch + 1 < n)
                                                mma_records_k<FMT, 1, 2, true>(rb + (size_t)ch * a.rec, a.rec, hi2, lo2, kbp,
                                                                               (k0 + ch) * CB, lane, ms->esc[warp], a1[0]);
                                            else
                                                mma_records_k<FMT, 1, 1, true>(rb + (size_t)ch * a.rec, a.rec, hi2, lo2, kbp,
                                                                               (k0 + ch) * CB, lane, ms->esc[warp], a1[0]);
                                        }
                                    __syncwarp();
                                    tacc[5] += BFP_TRACE_NOW() - tm0;
                                    [[maybe_unused]] const unsigned long long tg0 = BFP_TRACE_NOW();
                                    give_item();
                                    tacc[6] += BFP_TRACE_NOW() - tg0;
                                }
                            }
                            if (!both) {
#pragma unroll
                                for (int i = 0; i < 4; ++i) acc[0][0][i] = a1[0][0][i];
                            }
                        }
                        if (p2n == 0) STAMP(18);  // ... warp 0's MMAs done
                        if (p2n == 1) STAMP(29);
                        [[maybe_unused]] const unsigned long long tp0 = BFP_TRACE_NOW();
                        if (!bad && mine) {
                            const int rg = rg0 + warp;
                            if (packed) {  // column c + 4 holds the lo half of column c: lanes t and t ^ 2
#pragma unroll
                                for (int i = 0; i < 4; ++i) acc[0][0][i] += __shfl_xor_sync(0xffffffffu, acc[0][0][i], 2);
                            }
#pragma unroll
                            for (int g = 0; g < NGRP; ++g)
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int col = acc_xrow(lane, g, i);
                                    if (col < nr && (!packed || col < 4)) {
                                        const int r = ms->p2row[bi][col];
                                        const int s = ms->eslot[er][r];
                                        const int n = rg * 16 + acc_wrow(lane, i);
                                        a.part[((int64_t)r * (a.K + 1) + s) * a.H + n] =
                                            mul_pow2(acc[0][g][i], 24 - (MB - 1) - ms->p2shift[bi][col]);
                                    }
                                }
                        }
                        __syncwarp();
                        tacc[12] += BFP_TRACE_NOW() - tp0;
                        if (p2n == 0) STAMP(19);  // ... partial outputs stored
                        if (p2n == 1) STAMP(31);
                        ++p2n;
                    }
                }
            }
            STAMP(11);  // down projections done
            BFP_TRACE_SET(40, tacc[0]);
            BFP_TRACE_SET(41, tacc[1]);
            BFP_TRACE_SET(42, tacc[2]);
            BFP_TRACE_SET(44, tacc[3]);
            BFP_TRACE_SET(43, tacc[4] * 1000);
            BFP_TRACE_SET(45, tacc[5]);
            BFP_TRACE_SET(46, tacc[6]);
            BFP_TRACE_SET(47, tacc[7]);
            BFP_TRACE_SET(35, tacc[8] * 1000);
            BFP_TRACE_SET(36, tacc[9] * 1000);
            BFP_TRACE_SET(37, tacc[10]);
            BFP_TRACE_SET(38, tacc[11]);
            BFP_TRACE_SET(39, tacc[12]);
            if (!grid_barrier(&a.ctrl[3])) {  // every (row, slot) partial written
                abort_all();
                goto done;
            }
            STAMP(12);
            if (c == 0) {  // every CTA is past the phase-1 wait and done reading the row maxima
                if (tid == 0) a.ctrl[2] = 0u;
                for (int i = tid; i < a.M * (a.K + 1); i += NC) a.hmax[i] = 0u;
            }
            // ---- 6. combine: y_r = sum over slots (in slot order) + shared, for this CTA's row groups
            const int g0 = (int)((int64_t)c * a.ng_d / a.ncta), g1 = (int)((int64_t)(c + 1) * a.ng_d / a.ncta);
            for (int i = tid; i < (g1 - g0) * a.M * 16; i += NC) {
                const int rgl = i / (a.M * 16), rem = i - rgl * a.M * 16;
                const int r = rem >> 4, n = (g0 + rgl) * 16 + (rem & 15);
                float pv[kMaxTopK + 1];
#pragma unroll
                for (int s2 = 0; s2 <= kMaxTopK; ++s2)
                    pv[s2] = s2 <= a.K ? __ldcg(&a.part[((int64_t)r * (a.K + 1) + s2) * a.H + n]) : 0.f;
                float sum = 0.f;
#pragma unroll
                for (int s2 = 0; s2 <= kMaxTopK; ++s2)
                    if (s2 <= a.K) sum += pv[s2];
                if (a.y) a.y[(int64_t)r * a.H + n] = sum;
                if (a.h_out) {
                    const float hin = bf16_bits_to_f32(a.x[(int64_t)r * a.H + n]);
                    a.h_out[(int64_t)r * a.H + n] = f32_to_bf16_bits(hin + sum);
                }
            }
        }
    done:
        // No copy may still be landing in shared memory when the CTA exits (every path): this warp's
        // issued but unconsumed items, the stage, the consumers' own copies.
        {
            WaitCfg drain{int64_t(1) << 40, 1000000000ull};
            int sl = cu_slot;
            uint32_t par = cu_par;
            for (int k = cu; k < iss; ++k) {
                if (lane == 0) mbar_wait(my_full + sl, par, drain, nullptr);
                if (++sl == a.nsw) {
                    sl = 0;
                    par ^= 1u;
                }
            }
            if (tid == 0) {
                mbar_wait(&ms->stage_full, 0u, drain, nullptr);
            }
        }
    }
    __syncthreads();
    STAMP(30);
#undef STAMP
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
struct MoePlan {
    Geometry gu, dn, sgu, sdn;
    int ngrp, ncta, nsw, ch1, slot_bytes, frag_bytes, scr_bytes, r2, noct, Fmax, stage_off, stage_r, row_boxes;
    size_t smem;
    size_t off_ctrl, off_hmax, off_logits, off_hbuf, off_part, off_row, off_p1part;
    size_t ws_core;   // bytes the layer cannot run without
    size_t ws_bytes;  // plus the phase-1 handoff tiles (moe_workspace_size)
};

static int validate_layer(const bfp_moe_layer *L, int m) {
    if (!L) return fail(BFP_EINVAL, "null layer");
    if (m < 1 || m > kMaxRows) return fail(BFP_ESHAPE, "m must be in [1, 16]");
    if (L->expert_fmt != BFP_FMT_BFP4 && L->expert_fmt != BFP_FMT_BFP8) return fail(BFP_EINVAL, "bad expert_fmt");
    if (L->hidden < 16 || L->hidden % 16 || L->ffn < 16 || L->ffn % 16 || L->shared_ffn < 16 || L->shared_ffn % 16)
        return fail(BFP_ESHAPE, "hidden, ffn, shared_ffn must be positive multiples of 16");
    if (L->top_k < 1 || L->top_k > kMaxTopK || L->n_experts < L->top_k || L->n_experts > kMaxExperts)
        return fail(BFP_ESHAPE, "need 1 <= top_k <= 8 and top_k <= n_experts <= 256");
    if (L->hidden > 16384 || L->ffn > 16384 || L->shared_ffn > 16384) return fail(BFP_ESHAPE, "dimension too large");
    if (!L->router || !L->shared_gate || !L->experts_gate_up || !L->experts_down || !L->shared_gate_up ||
        !L->shared_down)
        return fail(BFP_EINVAL, "null weight pointer in layer");
    const void *ptrs[] = {L->router, L->shared_gate, L->experts_gate_up, L->experts_down, L->shared_gate_up,
                          L->shared_down};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(BFP_EALIGN, "layer weights must be 16-byte aligned");
    if (L->router_bias && ((uintptr_t)L->router_bias & 3u)) return fail(BFP_EALIGN, "router_bias misaligned");
    return BFP_OK;
}

static int plan_moe(const bfp_moe_layer *L, int m, MoePlan *p) {
    int rc = validate_layer(L, m);
    if (rc) return rc;
    DeviceInfo di;
    rc = device_info(&di);
    if (rc) return rc;
    const int fmt = L->expert_fmt;
    make_geometry(fmt, 2 * (int64_t)L->ffn, L->hidden, &p->gu);
    make_geometry(fmt, L->hidden, L->ffn, &p->dn);
    make_geometry(fmt, 2 * (int64_t)L->shared_ffn, L->hidden, &p->sgu);
    make_geometry(fmt, L->hidden, L->shared_ffn, &p->sdn);
    if (L->gate_up_stride < p->gu.bytes() || L->gate_up_stride % 16 || L->down_stride < p->dn.bytes() ||
        L->down_stride % 16)
        return fail(BFP_EINVAL, "expert strides must cover the packed matrices and be multiples of 16");
    p->ngrp = m > 8 ? 2 : 1;
    const int kbp_h = (int)(p->gu.kc * p->gu.cb), kbp_f = (int)(p->dn.kc * p->dn.cb),
              kbp_fs = (int)(p->sdn.kc * p->sdn.cb);
    p->Fmax = std::max(L->ffn, L->shared_ffn);
    p->frag_bytes = (int)std::max<int64_t>((int64_t)p->ngrp * kbp_h * 256,
                                           (int64_t)2 * p->ngrp * std::max(kbp_f, kbp_fs) * 256);
    const int nft = L->ffn / 16, nft_s = L->shared_ffn / 16;
    // grid: enough CTAs for the phase-1 units of the worst-case union, at most one per SM
    const int64_t worst_units = nft_s + (int64_t)std::min(L->n_experts, m * L->top_k) * nft;
    p->ncta = (int)std::max<int64_t>(1, std::min<int64_t>(di.sms, worst_units));
    const int rows_per_cta = (L->n_experts + 1 + p->ncta - 1) / p->ncta;  // router rows (+ gate row) per CTA
    // the router's per-warp partial tiles use the fragment area before the fragments are built
    p->frag_bytes = (int)std::max<int64_t>(p->frag_bytes, (int64_t)(rows_per_cta + 7) / 8 * kMoeWarps * kWarp * 16);
    // scratch (one activation group): the tiles of phase-1 units split over warps, one 256-float
    // tile per warp
    p->scr_bytes = p->ngrp == 1 ? kMoeWarps * 256 * 4 : 0;
    // phase 2: units of up to one row group per consumer warp
    p->r2 = (int)std::min<int64_t>(kMoeWarps, p->dn.ng);
    p->noct = (int)((p->dn.ng + p->r2 - 1) / p->r2);
    // the routing scan packs the phase-2 cost of the union into 16 bits
    if ((int64_t)p->noct * 7 * (kMaxExperts + 1) >= 65536) return fail(BFP_ESHAPE, "hidden size too large");
    // per-warp slots: a phase-1 chunk is ch1 records of a gate row group and the same of its up row
    // group, a phase-2 chunk 2 * ch1 records of one row group
    p->ch1 = (int)std::min<int64_t>(4, p->gu.kc);
    p->slot_bytes = 2 * p->ch1 * p->gu.rec;
    // the preamble stage (activation rows, then the CTA's router rows) takes the ring's last bytes
    p->stage_r = (int)align_up((size_t)m * stage_ldx(L->hidden) * 2, 16);
    const size_t stage_bytes = align_up((size_t)p->stage_r + (size_t)rows_per_cta * L->hidden * 2, 128);
    const size_t base = align_up((size_t)p->frag_bytes + p->scr_bytes + sizeof(MoeMisc), 16);
    const int64_t avail = (int64_t)di.smem_optin - (int64_t)base - 128;
    const int64_t per_slot_row = (int64_t)kMoeWarps * (p->slot_bytes + 8);  // one slot per warp + barrier
    p->nsw = (int)std::min<int64_t>(8, avail / per_slot_row);
    if (p->nsw < 2) return fail(BFP_ESHAPE, "layer too large for shared memory");
    const size_t ring = (size_t)kMoeWarps * p->nsw * p->slot_bytes;
    if (ring < stage_bytes) return fail(BFP_ESHAPE, "activation rows do not fit in shared memory");
    p->stage_off = (int)(ring - stage_bytes);
    p->smem = align_up(base + 8 * (size_t)kMoeWarps * p->nsw, 128) + ring;
    // workspace
    size_t o = kWsHeader;
    p->off_ctrl = o;
    o += 32;  // counters: [0..3] this kernel, [4..5] the one-row kernel (moe_row.cu)
    p->off_hmax = o;
    o = align_up(o + 4 * (size_t)m * (L->top_k + 1), 256);
    p->off_logits = o;
    o = align_up(o + 4 * (size_t)m * logit_stride(L->n_experts), 256);
    p->off_hbuf = o;
    o = align_up(o + 4 * (size_t)m * (L->top_k + 1) * p->Fmax, 256);
    p->off_part = o;
    o = align_up(o + 4 * (size_t)m * (L->top_k + 1) * L->hidden, 256);
    p->off_row = o;  // the one-row kernel's exchange area (moe_row.cu): epoch word, tagged logits and h
    p->row_boxes = row_boxes(di.sms);
    o = align_up(o + row_ws_bytes(L->n_experts, L->top_k, p->Fmax, L->hidden, p->row_boxes), 256);
    p->ws_core = o;
    p->off_p1part = o;
    o = align_up(o + 4 * (size_t)p->ncta * (kMoeWarps - 1) * kP1PartFloats, 256);
    p->ws_bytes = o;
    return BFP_OK;
}

template <int FMT, int NGRP>
static int launch_moe_t(const MoeArgs &a, const MoePlan &p, cudaStream_t st) {
    auto kern = moe_layer_kernel<FMT, NGRP>;
    int rc = set_smem_attr(reinterpret_cast<const void *>(kern), (int)p.smem, "cudaFuncSetAttribute(moe_layer)");
    if (rc) return rc;
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ncta);
    cfg.blockDim = dim3(kMoeThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (launch_mode() == BFP_LAUNCH_COOPERATIVE) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    } else {  // one CTA per SM takes the whole GPU: the CTAs are resident together once it is free
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return cuda_fail(e, "launch moe_layer");
    return BFP_OK;
}

#ifdef BFP_TRACE
extern "C" int bfp_debug_set_trace(void *buf) {
    return (int)cudaMemcpyToSymbol(g_bfp_trace, &buf, sizeof(buf));
}
#endif

static int moe_launch(const bfp_moe_layer *L, const uint16_t *x, int m, int norm, float *y, uint16_t *h_out,
                      int32_t *topk_idx, float *topk_w, void *ws, size_t ws_bytes, cudaStream_t st) {
    MoePlan p;
    int rc = plan_moe(L, m, &p);
    if (rc) return rc;
    if (!x) return fail(BFP_EINVAL, "null x");
    if (!y && !h_out) return fail(BFP_EINVAL, "no output");
    if (!aligned16(x) || (y && !aligned16(y)) || (h_out && !aligned16(h_out)) || !aligned16(ws) ||
        (topk_idx && ((uintptr_t)topk_idx & 3u)) || (topk_w && ((uintptr_t)topk_w & 3u)))
        return fail(BFP_EALIGN, "device pointers must be 16-byte aligned");
    // a workspace of ws_core bytes runs the layer without the phase-1 handoff tiles (whole units per warp)
    if (!ws || ws_bytes < p.ws_core) return fail(BFP_EWORKSPACE, "workspace smaller than moe_workspace_size");
    uint8_t *w = static_cast<uint8_t *>(ws);
    MoeArgs a;
    a.H = L->hidden;
    a.E = L->n_experts;
    a.F = L->ffn;
    a.K = L->top_k;
    a.Fs = L->shared_ffn;
    a.M = m;
    a.ncta = p.ncta;
    a.x = x;
    a.norm = norm;
    a.eps = 1e-6f;
    a.router = L->router;
    a.rbias = L->router_bias;
    a.sgate = L->shared_gate;
    a.gu = static_cast<const uint8_t *>(L->experts_gate_up);
    a.dn = static_cast<const uint8_t *>(L->experts_down);
    a.gu_stride = L->gate_up_stride;
    a.dn_stride = L->down_stride;
    a.sgu = static_cast<const uint8_t *>(L->shared_gate_up);
    a.sdn = static_cast<const uint8_t *>(L->shared_down);
    a.y = y;
    a.h_out = h_out;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.status = reinterpret_cast<uint32_t *>(w);
    a.ctrl = reinterpret_cast<uint32_t *>(w + p.off_ctrl);
    a.hmax = reinterpret_cast<uint32_t *>(w + p.off_hmax);
    a.logits = reinterpret_cast<float *>(w + p.off_logits);
    a.hbuf = reinterpret_cast<float *>(w + p.off_hbuf);
    a.part = reinterpret_cast<float *>(w + p.off_part);
    a.p1part = ws_bytes >= p.ws_bytes ? reinterpret_cast<float *>(w + p.off_p1part) : nullptr;
    a.rec = p.gu.rec;
    a.kc_h = (int)p.gu.kc;
    a.kbp_h = (int)(p.gu.kc * p.gu.cb);
    a.kc_f = (int)p.dn.kc;
    a.kbp_f = (int)(p.dn.kc * p.dn.cb);
    a.kc_fs = (int)p.sdn.kc;
    a.kbp_fs = (int)(p.sdn.kc * p.sdn.cb);
    a.nft = L->ffn / 16;
    a.nft_s = L->shared_ffn / 16;
    a.ng_d = (int)p.dn.ng;
    a.r2 = p.r2;
    a.noct = p.noct;
    a.Fmax = p.Fmax;
    a.nsw = p.nsw;
    a.ch1 = p.ch1;
    a.slot_bytes = p.slot_bytes;
    a.stage_off = p.stage_off;
    a.stage_r = p.stage_r;
    a.frag_bytes = p.frag_bytes;
    a.scr_bytes = p.scr_bytes;
    a.wait = wait_cfg();
    a.wait_data = WaitCfg{kDefaultWaitIters, kDefaultWaitNanos};
    if (m == 1 && row_path()) {  // one row: the latency path (moe_row.cu), when the layer's shape fits it
        rc = row_layers_launch(L, 1, x, norm, y, h_out, topk_idx, topk_w, a.status, w + p.off_row, a.Fmax, st);
        if (rc != kRowNotApplicable) return rc;
    }
    if (L->expert_fmt == BFP_FMT_BFP4)
        return p.ngrp == 1 ? launch_moe_t<4, 1>(a, p, st) : launch_moe_t<4, 2>(a, p, st);
    return p.ngrp == 1 ? launch_moe_t<8, 1>(a, p, st) : launch_moe_t<8, 2>(a, p, st);
}

}  // namespace bfp

using namespace bfp;

extern "C" {

int moe_workspace_size(const bfp_moe_layer *layer, int m, size_t *bytes) {
    if (!bytes) return fail(BFP_EINVAL, "bytes is null");
    MoePlan p;
    int rc = plan_moe(layer, m, &p);
    if (rc) return rc;
    *bytes = p.ws_bytes;
    return BFP_OK;
}

int moe_decode_layer(const bfp_moe_layer *layer, const uint16_t *x, int m, float *y, int32_t *topk_idx,
                     float *topk_w, void *ws, size_t ws_bytes, bfp_stream_t stream) {
    if (!y) return fail(BFP_EINVAL, "null y");
    return moe_launch(layer, x, m, 0, y, nullptr, topk_idx, topk_w, ws, ws_bytes,
                      reinterpret_cast<cudaStream_t>(stream));
}

// Stack workspace: [moe workspace (its header holds the shared status word)]
//                  [linear workspace body][two bf16 h buffers]
static int stack_layout(const bfp_moe_layer *layers, int n_layers, const bfp_matrix *lm_head, int m, size_t *moe_b,
                        size_t *lin_b, size_t *h_b) {
    if (!layers || n_layers < 1) return fail(BFP_EINVAL, "need at least one layer");
    size_t mb = 0;
    for (int l = 0; l < n_layers; ++l) {
        MoePlan p;
        int rc = plan_moe(&layers[l], m, &p);
        if (rc) return rc;
        if (layers[l].hidden != layers[0].hidden) return fail(BFP_ESHAPE, "layers differ in hidden size");
        mb = std::max(mb, p.ws_bytes);
    }
    if (!lm_head || lm_head->k != layers[0].hidden) return fail(BFP_ESHAPE, "lm_head.k must equal hidden");
    size_t lb = 0;
    int rc = linear_ws_body_bytes(lm_head, m, &lb);
    if (rc) return rc;
    *moe_b = align_up(mb, 256);
    *lin_b = align_up(lb, 256);
    *h_b = align_up((size_t)m * layers[0].hidden * 2, 256);
    return BFP_OK;
}

int moe_stack_workspace_size(const bfp_moe_layer *layers, int n_layers, const bfp_matrix *lm_head, int m,
                             size_t *bytes) {
    if (!bytes) return fail(BFP_EINVAL, "bytes is null");
    size_t a, b, c;
    int rc = stack_layout(layers, n_layers, lm_head, m, &a, &b, &c);
    if (rc) return rc;
    *bytes = a + b + c;
    return BFP_OK;
}

// The stack, then the LM head: fp32 logits (nullable when tokens are asked for) and, with tokens, the greedy
// next token of every row from the LM head's own epilogue.
static int stack_run(const bfp_moe_layer *layers, int n_layers, const bfp_matrix *lm_head, uint16_t *h, int m,
                     float *logits, int32_t *tokens, int32_t *topk_idx, void *ws, size_t ws_bytes, cudaStream_t st) {
    size_t mb, lb, hb;
    int rc = stack_layout(layers, n_layers, lm_head, m, &mb, &lb, &hb);
    if (rc) return rc;
    if (!h || (!logits && !tokens)) return fail(BFP_EINVAL, "null h, or neither logits nor tokens");
    if (!ws || ws_bytes < mb + lb + hb) return fail(BFP_EWORKSPACE, "workspace smaller than moe_stack_workspace_size");
    if (!aligned16(h) || (logits && !aligned16(logits)) || !aligned16(ws))
        return fail(BFP_EALIGN, "pointers must be 16-byte aligned");
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint16_t *hb2 = reinterpret_cast<uint16_t *>(w + mb + lb);
    uint16_t *cur = h, *nxt = hb2;
    int32_t *idx = topk_idx;  // layer l's selection follows the layers before it, m * top_k entries each
    int l0 = 0;               // layers done
    if (m == 1 && row_path()) {
        // one row: the layers in as few launches as possible (each runs up to 48 layers of one shape, the
        // residual row passing between them inside the launch), h updated in place
        MoePlan p;
        rc = plan_moe(&layers[0], 1, &p);
        if (rc) return rc;
        while (l0 < n_layers) {
            const int nl = std::min(48, n_layers - l0);
            rc = row_layers_launch(&layers[l0], nl, h, 1, nullptr, h, idx, nullptr, reinterpret_cast<uint32_t *>(w),
                                   w + p.off_row, p.Fmax, st);
            if (rc == kRowNotApplicable) break;  // the remaining layers one launch each
            if (rc) return rc;
            if (idx) idx += (int64_t)nl * layers[l0].top_k;
            l0 += nl;
        }
    }
    for (int l = l0; l < n_layers; ++l) {
        rc = moe_launch(&layers[l], cur, m, 1, nullptr, nxt, idx, nullptr, ws, mb, st);
        if (rc) return rc;
        if (idx) idx += (int64_t)m * layers[l].top_k;
        std::swap(cur, nxt);
    }
    if (cur != h) {
        cudaError_t e = cudaMemcpyAsync(h, cur, (size_t)m * layers[0].hidden * 2, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e, "copy final h");
    }
    return linear_launch_ex(lm_head, h, m, layers[0].hidden, logits, nullptr, lm_head->n,
                            reinterpret_cast<uint32_t *>(w), w + mb, lb, st, 1, tokens);
}

int moe_stack_decode(const bfp_moe_layer *layers, int n_layers, const bfp_matrix *lm_head, uint16_t *h, int m,
                     float *logits, int32_t *topk_idx, void *ws, size_t ws_bytes, bfp_stream_t stream) {
    if (!logits) return fail(BFP_EINVAL, "null logits");
    return stack_run(layers, n_layers, lm_head, h, m, logits, nullptr, topk_idx, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

int moe_stack_decode_greedy(const bfp_moe_layer *layers, int n_layers, const bfp_matrix *lm_head, uint16_t *h, int m,
                            float *logits, int32_t *tokens, int32_t *topk_idx, void *ws, size_t ws_bytes,
                            bfp_stream_t stream) {
    if (!tokens) return fail(BFP_EINVAL, "null tokens");
    if ((uintptr_t)tokens & 3u) return fail(BFP_EALIGN, "tokens must be 4-byte aligned");
    return stack_run(layers, n_layers, lm_head, h, m, logits, tokens, topk_idx, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ----------------------------------------------------------------------------
// moe_decode_layer_static: the same layer for callers that cannot allocate
// device memory. Its scratch is one file-scope device array of a fixed size,
// shared by every call on a device and kept for the life of the process.
// ----------------------------------------------------------------------------
namespace bfp {

constexpr size_t kStaticScratchBytes = size_t(2) << 20;  // 2 MiB: a full-size layer at 16 rows needs about 1.85 MB
static __device__ __align__(256) uint8_t g_moe_static_scratch[kStaticScratchBytes];

// Device address of the scratch array on the current device. The array's name
// in host code is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current; the array
// is zeroed at the same time. Both steps are synchronous: the first call on a
// device must not happen inside a stream capture.
static int static_scratch(void **out) {
    static std::mutex mu;
    static std::vector<void *> addr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(mu);
    if ((int)addr.size() <= dev) addr.resize(dev + 1, nullptr);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_moe_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        e = cudaMemset(p, 0, kStaticScratchBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(static scratch)");
        addr[dev] = p;
    }
    *out = addr[dev];
    return BFP_OK;
}

}  // namespace bfp

extern "C" int moe_decode_layer_static(const bfp_moe_layer *layer, const uint16_t *x, int m, float *y,
                                       int32_t *topk_idx, float *topk_w, bfp_stream_t stream) {
    if (!y) return fail(BFP_EINVAL, "null y");
    MoePlan p;
    int rc = plan_moe(layer, m, &p);
    if (rc) return rc;
    if (p.ws_core > kStaticScratchBytes)
        return fail(BFP_EWORKSPACE, "this layer needs " + std::to_string(p.ws_core) +
                                        " bytes of scratch; the built-in scratch holds " +
                                        std::to_string(kStaticScratchBytes) +
                                        " (use moe_decode_layer with a caller-allocated workspace)");
    void *ws = nullptr;
    rc = static_scratch(&ws);
    if (rc) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // The status word and the cross-block counters must start at zero: clear them on the stream.
    cudaError_t e = cudaMemsetAsync(ws, 0, p.off_logits, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static scratch counters)");
    if (m == 1) {  // the one-row kernel's epoch word and tagged words start over too
        e = cudaMemsetAsync(static_cast<uint8_t *>(ws) + p.off_row, 0,
                            row_ws_bytes(layer->n_experts, layer->top_k, p.Fmax, layer->hidden, p.row_boxes), st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static scratch, one-row area)");
    }
    return moe_launch(layer, x, m, 0, y, nullptr, topk_idx, topk_w, ws, kStaticScratchBytes, st);
}
