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
// GB300 design: the layer is one persistent cooperative kernel, one CTA per SM
// (8 consumer warps + 1 producer warp). Nothing waits on the host between the
// router and the experts. Each CTA walks a fixed list of "units", each a
// contiguous span of packed weights streamed into a shared-memory ring by
// cp.async.bulk (TMA, 1D) on mbarriers:
//   1. its rows of the router (and the shared-gate vector as one extra row):
//      fp32 logits to the workspace, then a release increment of a counter;
//   2. its shared-expert gate/up f-tiles (known before routing, so their bytes
//      stream while the router counter fills);
//   3. after the router counter reaches the grid size, every CTA redundantly
//      takes softmax / top-k / renormalisation and deduplicates the union U of
//      experts selected by any row (so no host sync, no second launch);
//   4. routed gate/up f-tiles (expert in U, 16 ffn rows): h = silu(a) * b for
//      every row that chose the expert, fp32 to the workspace, then a release
//      increment of that expert's counter;
//   5. down-projection units (expert, 8 row groups of the hidden dimension):
//      wait for the expert's counter, multiply by the routing weight, split h
//      into fp16 hi + lo fragments (22 significant bits), write per-(row, slot)
//      partial outputs; the last of the |U|+1 arrivals for a row group sums
//      the slots in slot order (deterministic, no float atomics).
// Every expert's weights are read from HBM once per step however many rows
// chose it. All cross-CTA waits are bounded and report BFP_ETIMEOUT.
#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "bfp_launch.h"
#include "bfp_tiles.cuh"

namespace bfp {

using namespace dev;

int linear_launch_ex(const bfp_matrix *w, const uint16_t *x, int m, int64_t ldx, float *y, uint16_t *y_bf16,
                     int64_t ldy, uint32_t *status, void *body, size_t body_bytes, cudaStream_t st, int norm);
int linear_ws_body_bytes(const bfp_matrix *w, int m, size_t *bytes);

constexpr int kMaxRows = 16;
constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 256;

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
    uint32_t *status, *ctrl, *done1, *rgcnt;
    float *logits, *hbuf, *part;
    int rec, kc_h, kbp_h, kc_f, kbp_f, kc_fs, kbp_fs;
    int nft, nft_s, ng_d, r2, noct, Fmax;
    int nslot, slot_bytes, frag_bytes, scr_bytes;
    WaitCfg wait;       // cross-block waits (router counter, expert counters)
    WaitCfg wait_data;  // this CTA's own bulk copies and slot hand-backs
};

// Shared-memory bookkeeping of one CTA.
struct MoeMisc {
    int shift_x[kMaxRows];
    float inv[kMaxRows];
    int shift_h[kMaxRows];
    float gate_w[kMaxRows];
    float hw[kMaxRows];  // combine weight of the current phase-2 expert per row
    int32_t tk_idx[kMaxRows][kMaxTopK];
    float tk_w[kMaxRows][kMaxTopK];
    uint32_t bitmap[kMaxExperts / 32];
    uint32_t umask[kMaxExperts + 1];
    int16_t pos[kMaxExperts];
    int16_t ulist[kMaxExperts + 1];
    int8_t uslot[kMaxExperts + 1][kMaxRows];
    uint32_t maxbits[kMaxRows];
    int nU;
    int flags[4];  // [0] abort
};

__host__ __device__ inline int router_row_start(int c, int rows, int ncta) { return (int)((int64_t)c * rows / ncta); }

// Ordered 32-bit key of a float: larger float <=> larger unsigned key.
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int FMT, int NGRP>
__global__ void __launch_bounds__(kThreads, 1) moe_layer_kernel(const MoeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int NW = kConsumerWarps;
    constexpr int NC = NW * kWarp;  // consumer threads
    constexpr int MB = FMT == 4 ? 3 : 7;
    constexpr int CB = FMT == 4 ? 4 : 2;
    uint32_t *frag = reinterpret_cast<uint32_t *>(smem);
    float *scr = reinterpret_cast<float *>(smem + a.frag_bytes);
    MoeMisc *ms = reinterpret_cast<MoeMisc *>(smem + a.frag_bytes + a.scr_bytes);
    const size_t bar_off = align_up(a.frag_bytes + a.scr_bytes + sizeof(MoeMisc), 16);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + bar_off);
    uint64_t *empty = full + a.nslot;
    uint8_t *ring = smem + align_up(bar_off + 16 * a.nslot, 128);
    volatile int *vflags = ms->flags;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int E1 = a.E + 1;  // router rows + the shared-gate row
    const int rr0 = router_row_start(c, E1, a.ncta), rr1 = router_row_start(c + 1, E1, a.ncta);
    const int64_t gb_h = (int64_t)a.kc_h * a.rec;  // bytes of one gate/up row group
    const int nft_total_pre = a.nft_s;              // phase-1 units known before routing

    if (tid == 0) {
        for (int i = 0; i < a.nslot; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
        }
        for (int i = 0; i < 4; ++i) ms->flags[i] = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == NW) {
        // ==================================================================== producer
        // Lane 0 issues every copy; the whole warp meets the consumers at the
        // routing hand-off (named barrier 2) at one convergent point.
        int64_t u = 0;
        bool bad = false;
        auto issue = [&](int nspan, const uint8_t *const *src, const uint32_t *bytes) -> bool {
            const int slot = (int)(u % a.nslot);
            const int64_t use = u / a.nslot;
            if (use > 0 && !mbar_wait(&empty[slot], (uint32_t)((use - 1) & 1), a.wait_data, vflags)) return false;
            if (vflags[0]) return false;
            uint32_t total = 0;
            for (int i = 0; i < nspan; ++i) total += bytes[i];
            mbar_arrive_expect_tx(&full[slot], total);
            uint8_t *dst = ring + (size_t)slot * a.slot_bytes;
            for (int i = 0; i < nspan; ++i) {
                bulk_g2s(dst, src[i], bytes[i], &full[slot]);
                dst += bytes[i];
            }
            ++u;
            return true;
        };
        if (lane == 0) {
            // 1. router rows
            if (rr1 > rr0) {
                const uint8_t *src[2];
                uint32_t bytes[2];
                int ns = 0;
                const int re = min(rr1, a.E);
                if (re > rr0) {
                    src[ns] = reinterpret_cast<const uint8_t *>(a.router + (int64_t)rr0 * a.H);
                    bytes[ns++] = (uint32_t)(re - rr0) * a.H * 2;
                }
                if (rr1 > a.E) {
                    src[ns] = reinterpret_cast<const uint8_t *>(a.sgate);
                    bytes[ns++] = (uint32_t)a.H * 2;
                }
                bad = !issue(ns, src, bytes);
            }
            // 2. shared-expert gate/up f-tiles
            for (int g = c; !bad && g < nft_total_pre; g += a.ncta) {
                const uint8_t *src[1] = {a.sgu + (int64_t)2 * g * gb_h};
                const uint32_t bytes[1] = {(uint32_t)(2 * gb_h)};
                bad = !issue(1, src, bytes);
            }
        }
        // 3. wait for the consumers' routing decision
        __syncwarp();
        bar_sync(2, kThreads);
        if (lane == 0) {
            const int nU = ms->nU;
            if (vflags[0]) bad = true;
            // 4. routed gate/up f-tiles
            const int p1 = a.nft_s + nU * a.nft;
            int g = c;
            while (g < a.nft_s) g += a.ncta;
            for (; !bad && g < p1; g += a.ncta) {
                const int i = g - a.nft_s;
                const int e = ms->ulist[i / a.nft], ft = i % a.nft;
                const uint8_t *src[1] = {a.gu + (int64_t)e * a.gu_stride + (int64_t)2 * ft * gb_h};
                const uint32_t bytes[1] = {(uint32_t)(2 * gb_h)};
                bad = !issue(1, src, bytes);
            }
            // 5. down-projection units
            const int64_t p2 = (int64_t)(nU + 1) * a.noct;
            const int64_t q0 = (int64_t)c * p2 / a.ncta, q1 = (int64_t)(c + 1) * p2 / a.ncta;
            for (int64_t q = q0; !bad && q < q1; ++q) {
                const int j = (int)(q / a.noct), oct = (int)(q % a.noct);
                const bool sh = j == nU;
                const int kc = sh ? a.kc_fs : a.kc_f;
                const int64_t gb_f = (int64_t)kc * a.rec;
                const int rg0 = oct * a.r2, nrg = min(a.r2, a.ng_d - rg0);
                const uint8_t *base = sh ? a.sdn : a.dn + (int64_t)ms->ulist[j] * a.dn_stride;
                const uint8_t *src[1] = {base + rg0 * gb_f};
                const uint32_t bytes[1] = {(uint32_t)(nrg * gb_f)};
                bad = !issue(1, src, bytes);
            }
            // No copy may still be landing in shared memory when the CTA exits.
            WaitCfg drain{int64_t(1) << 40, 1000000000ull};
            for (int64_t sl = 0; sl < min64(u, a.nslot); ++sl) {
                const int64_t last_use = (u - 1 - sl) / a.nslot;
                mbar_wait(&full[sl], (uint32_t)(last_use & 1), drain, nullptr);
            }
            if (bad && !vflags[0]) {
                raise_status(a.status, kStatusTimeout);
                vflags[0] = 1;
            }
        }
        __syncwarp();
    } else {
        // =================================================================== consumers
        bool dispatched = false;
        bool bad = false;
        int64_t u = 0;
        const uint2 *frag2 = reinterpret_cast<const uint2 *>(frag);
        const int ngrp_rows = a.M > 8 ? 3 : 1;
        auto abort_all = [&]() {
            if (tid == 0) {
                vflags[0] = 1;
                raise_status(a.status, kStatusTimeout);
            }
        };
        auto wait_slot = [&](int64_t uu) -> int {
            const int slot = (int)(uu % a.nslot);
            if (!bad)
                bad = !__all_sync(0xffffffffu,
                                  mbar_wait(&full[slot], (uint32_t)((uu / a.nslot) & 1), a.wait_data, nullptr));
            return slot;
        };
        // A warp whose data never arrived keeps the slot, so the producer cannot
        // start a second copy into memory that a first copy may still be filling.
        auto release_slot = [&](int slot) {
            __syncwarp();
            if (lane == 0 && !bad) mbar_arrive(&empty[slot]);
        };

        // ---- activation fragments (MoE input: x, or bf16(RMSNorm(h)) in stack mode)
        build_act_frags<NC>(a.x, a.H, a.M, a.H, a.kbp_h, NGRP, a.norm != 0, a.eps, frag, ms->shift_x, ms->inv, tid, warp,
                        lane);

        // ---- phase-1 unit: one f-tile (16 ffn rows) of gate and up; h = silu(gate) * up for the
        //      rows in rowmask, slot table row jrow. Returns false on abort (same answer in all warps).
        auto run_phase1 = [&](int eid, int ft, uint32_t rowmask, int jrow) -> bool {
            const int slot = wait_slot(u);
            const uint8_t *slotp = ring + (size_t)slot * a.slot_bytes;
            const uint32_t gm = (((rowmask & 0xFFu) ? 1u : 0u) | ((rowmask & 0xFF00u) ? 2u : 0u)) & ngrp_rows;
            float acc[2][NGRP][4];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int g = 0; g < NGRP; ++g)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[r][g][i] = 0.f;
            if (!bad) {
                for (int ch = warp; ch < a.kc_h; ch += NW) {
                    const uint8_t *recs[2] = {slotp + (size_t)ch * a.rec, slotp + gb_h + (size_t)ch * a.rec};
                    mma_records<FMT, NGRP, 2, false>(recs, frag2, nullptr, a.kbp_h, ch * CB, lane, gm, acc);
                }
            }
            release_slot(slot);
            ++u;
            constexpr int TILE = NGRP * 128;
            float *mine = scr + warp * 2 * TILE;
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int g = 0; g < NGRP; ++g)
#pragma unroll
                    for (int i = 0; i < 4; ++i) mine[r * TILE + (g * 4 + i) * kWarp + lane] = acc[r][g][i];
            if (bar_or(1, NC, bad)) return false;
            if (tid < TILE) {
                float va = 0.f, vb = 0.f;
                for (int w = 0; w < NW; ++w) {
                    va += scr[w * 2 * TILE + tid];
                    vb += scr[w * 2 * TILE + TILE + tid];
                }
                const int grp = tid >> 7, i = (tid >> 5) & 3, ln = tid & 31;
                const int r = acc_xrow(ln, grp, i);
                const int f = ft * 16 + acc_wrow(ln, i);
                if (r < a.M && ((rowmask >> r) & 1u)) {
                    const int sh = 24 - (MB - 1) - ms->shift_x[r];
                    const float ga = scalbnf(va, sh), ub = scalbnf(vb, sh);
                    const float hv = ga / (1.0f + expf(-ga)) * ub;  // silu(gate) * up
                    const int s = ms->uslot[jrow][r];
                    a.hbuf[((int64_t)r * (a.K + 1) + s) * a.Fmax + f] = hv;
                }
            }
            __threadfence();
            bar_sync(1, NC);
            if (tid == 0) red_release_add(&a.done1[eid], 1u);
            return true;
        };

        // ---- 1. router rows
        if (rr1 > rr0) {
            const int slot = wait_slot(u);
            const uint16_t *wr = reinterpret_cast<const uint16_t *>(ring + (size_t)slot * a.slot_bytes);
            const int nrows = rr1 - rr0;
            if (!bad) {
                for (int p = warp; p < nrows * a.M; p += NW) {
                    const int i = p / a.M, r = p % a.M;
                    const uint16_t *xr = a.x + (int64_t)r * a.H;
                    const uint16_t *w = wr + (int64_t)i * a.H;
                    const float inv = ms->inv[r];
                    float acc = 0.f;
                    for (int j = lane * 8; j < a.H; j += 8 * kWarp) {
                        const uint4 wv = *reinterpret_cast<const uint4 *>(w + j);
                        const uint4 xv = *reinterpret_cast<const uint4 *>(xr + j);
                        const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w}, xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            float x0 = bf16_bits_to_f32(xa[q] & 0xFFFFu), x1 = bf16_bits_to_f32(xa[q] >> 16);
                            if (a.norm) {
                                x0 = __bfloat162float(__float2bfloat16_rn(x0 * inv));
                                x1 = __bfloat162float(__float2bfloat16_rn(x1 * inv));
                            }
                            acc = fmaf(bf16_bits_to_f32(wa[q] & 0xFFFFu), x0, acc);
                            acc = fmaf(bf16_bits_to_f32(wa[q] >> 16), x1, acc);
                        }
                    }
                    acc = warp_sum(acc);
                    if (lane == 0) {
                        const int row = rr0 + i;
                        if (row < a.E && a.rbias) acc += a.rbias[row];
                        a.logits[(int64_t)r * E1 + row] = acc;
                    }
                }
            }
            release_slot(slot);
            ++u;
        }
        __threadfence();
        if (bar_or(1, NC, bad)) {
            abort_all();
            goto done;
        }
        if (tid == 0) red_release_add(&a.ctrl[0], 1u);

        // ---- 2. shared-expert gate/up f-tiles (all rows use the shared expert)
        for (int g = c; g < a.nft_s; g += a.ncta) {
            if (tid == 0) {
                ms->umask[kMaxExperts] = (a.M >= 32 ? 0xFFFFFFFFu : ((1u << a.M) - 1u));
                for (int r = 0; r < a.M; ++r) ms->uslot[kMaxExperts][r] = (int8_t)a.K;
            }
            bar_sync(1, NC);
            if (!run_phase1(a.E, g, ms->umask[kMaxExperts], kMaxExperts)) {
                abort_all();
                goto done;
            }
        }

        // ---- 3. routing: wait for every CTA's router rows, then top-k and the expert union
        {
            bool ok = true;
            if (tid == 0) ok = wait_counter(&a.ctrl[0], (uint32_t)a.ncta, a.wait);
            if (bar_or(1, NC, !ok)) {
                abort_all();
                goto done;
            }
            float *lg = scr;  // M x E1 logits (the phase-1 scratch is free here)
            for (int i = tid; i < a.M * E1; i += NC) lg[i] = __ldcg(&a.logits[i]);
            bar_sync(1, NC);
            for (int r = warp; r < a.M; r += NW) {
                float v[8];
                float p[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int e = lane + 32 * q;
                    v[q] = e < a.E ? lg[r * E1 + e] : -INFINITY;
                }
                float mx = -INFINITY;
#pragma unroll
                for (int q = 0; q < 8; ++q) mx = fmaxf(mx, v[q]);
                mx = warp_max(mx);
#pragma unroll
                for (int q = 0; q < 8; ++q) p[q] = (lane + 32 * q < a.E) ? expf(v[q] - mx) : 0.f;
                uint32_t taken = 0;
                float psum = 0.f;
                for (int s = 0; s < a.K; ++s) {
                    int bq = -1;
                    float bv = 0.f;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const bool ok2 = lane + 32 * q < a.E && !((taken >> q) & 1u);
                        if (ok2 && (bq < 0 || v[q] > bv)) {
                            bq = q;
                            bv = v[q];
                        }
                    }
                    const uint32_t key = bq >= 0 ? order_key(bv) : 0u;
                    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
                    const uint32_t cand = (bq >= 0 && key == kmax) ? (uint32_t)(lane + 32 * bq) : 0xFFFFFFFFu;
                    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
                    const int owner = (int)(win & 31u), wq = (int)(win >> 5);
                    float pw = 0.f;
                    if (lane == owner) {
                        taken |= 1u << wq;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            if (q == wq) pw = p[q];
                    }
                    pw = __shfl_sync(0xffffffffu, pw, owner);
                    psum += pw;
                    if (lane == 0) {
                        ms->tk_idx[r][s] = (int32_t)win;
                        ms->tk_w[r][s] = pw;
                    }
                }
                if (lane == 0) {
                    for (int s = 0; s < a.K; ++s) ms->tk_w[r][s] = ms->tk_w[r][s] / psum;
                    ms->gate_w[r] = 1.0f / (1.0f + expf(-lg[r * E1 + a.E]));
                }
            }
            if (tid < kMaxExperts / 32) ms->bitmap[tid] = 0u;
            for (int i = tid; i <= kMaxExperts; i += NC) ms->umask[i] = 0u;
            bar_sync(1, NC);
            if (c == 0) {
                for (int i = tid; i < a.M * a.K; i += NC) {
                    const int r = i / a.K, s = i % a.K;
                    if (a.topk_idx) a.topk_idx[i] = ms->tk_idx[r][s];
                    if (a.topk_w) a.topk_w[i] = ms->tk_w[r][s];
                }
            }
            for (int i = tid; i < a.M * a.K; i += NC) {
                const int e = ms->tk_idx[i / a.K][i % a.K];
                atomicOr(&ms->bitmap[e >> 5], 1u << (e & 31));
            }
            bar_sync(1, NC);
            if (warp == 0) {
                int base = 0;
                for (int wd = 0; wd < kMaxExperts / 32; ++wd) {
                    const uint32_t word = ms->bitmap[wd];
                    const int pre = __popc(word & ((1u << lane) - 1u));
                    if ((word >> lane) & 1u) {
                        const int e = 32 * wd + lane;
                        ms->pos[e] = (int16_t)(base + pre);
                        ms->ulist[base + pre] = (int16_t)e;
                    }
                    base += __popc(word);
                }
                if (lane == 0) {
                    ms->nU = base;
                    ms->ulist[base] = (int16_t)a.E;
                }
            }
            bar_sync(1, NC);
            const int nU = ms->nU;
            for (int i = tid; i < a.M * a.K; i += NC) {
                const int r = i / a.K, s = i % a.K;
                const int j = ms->pos[ms->tk_idx[r][s]];
                atomicOr(&ms->umask[j], 1u << r);
                ms->uslot[j][r] = (int8_t)s;
            }
            if (tid < a.M) ms->uslot[nU][tid] = (int8_t)a.K;
            if (tid == 0) ms->umask[nU] = (1u << a.M) - 1u;
            bar_sync(1, NC);
        }
        bar_arrive(2, kThreads);
        dispatched = true;

        // ---- 4. routed gate/up f-tiles
        {
            const int nU = ms->nU;
            const int p1 = a.nft_s + nU * a.nft;
            int g = c;
            while (g < a.nft_s) g += a.ncta;
            for (; g < p1; g += a.ncta) {
                const int i = g - a.nft_s;
                const int j = i / a.nft, ft = i % a.nft;
                if (!run_phase1(ms->ulist[j], ft, ms->umask[j], j)) {
                    abort_all();
                    goto done;
                }
            }
        }

        // ---- 5. down projection + combine
        {
            const int nU = ms->nU;
            const int64_t p2 = (int64_t)(nU + 1) * a.noct;
            const int64_t q0 = (int64_t)c * p2 / a.ncta, q1 = (int64_t)(c + 1) * p2 / a.ncta;
            int cur = -1;
            uint32_t *hfrag = frag;  // x fragments are dead once phase 1 is done
            for (int64_t q = q0; q < q1; ++q) {
                const int j = (int)(q / a.noct), oct = (int)(q % a.noct);
                const bool sh = j == nU;
                const int eid = sh ? a.E : ms->ulist[j];
                const int Fe = sh ? a.Fs : a.F;
                const int kc = sh ? a.kc_fs : a.kc_f, kbp = sh ? a.kbp_fs : a.kbp_f;
                const uint32_t rowmask = ms->umask[j];
                if (j != cur) {
                    // h of this expert complete? (all its f-tiles, from whichever CTAs ran them)
                    bool ok = true;
                    if (tid == 0) ok = wait_counter(&a.done1[eid], (uint32_t)(sh ? a.nft_s : a.nft), a.wait);
                    if (bar_or(1, NC, !ok)) {
                        abort_all();
                        goto done;
                    }
                    if (tid < a.M) {
                        ms->maxbits[tid] = 0u;
                        ms->hw[tid] = ((rowmask >> tid) & 1u) ? (sh ? ms->gate_w[tid] : ms->tk_w[tid][ms->uslot[j][tid]]) : 0.f;
                    }
                    const int words = 2 * NGRP * kbp * kWarp * 2;
                    for (int i = tid; i < words / 4; i += NC) reinterpret_cast<uint4 *>(hfrag)[i] = make_uint4(0, 0, 0, 0);
                    bar_sync(1, NC);
                    // routing weight folded into h; per-row power-of-two scale into fp16 range
                    for (int i = tid; i < a.M * Fe; i += NC) {
                        const int r = i / Fe, f = i % Fe;
                        if ((rowmask >> r) & 1u) {
                            const float v = __ldcg(&a.hbuf[((int64_t)r * (a.K + 1) + ms->uslot[j][r]) * a.Fmax + f]) * ms->hw[r];
                            atomicMax(&ms->maxbits[r], __float_as_uint(fabsf(v)));
                        }
                    }
                    bar_sync(1, NC);
                    if (tid < a.M) ms->shift_h[tid] = frag_shift(__uint_as_float(ms->maxbits[tid]));
                    bar_sync(1, NC);
                    const int fb = Fe / 16;
                    const int lo_off = NGRP * kbp * kWarp * 2;  // words
                    for (int i = tid; i < a.M * fb * 8; i += NC) {
                        const int r = i / (fb * 8), rem = i % (fb * 8), b = rem >> 3, jj = rem & 7;
                        if (!((rowmask >> r) & 1u)) continue;
                        const float *hp = a.hbuf + ((int64_t)r * (a.K + 1) + ms->uslot[j][r]) * a.Fmax + 16 * b + 2 * jj;
                        const float w = ms->hw[r];
                        const int shh = ms->shift_h[r];
                        const float v0 = scalbnf(__ldcg(hp) * w, shh), v1 = scalbnf(__ldcg(hp + 1) * w, shh);
                        const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
                        const float r0 = v0 - __half2float(h0), r1 = v1 - __half2float(h1);
                        const int wi = frag_word(r, b, jj, kbp);
                        __half2 hh = __halves2half2(h0, h1);
                        hfrag[wi] = *reinterpret_cast<uint32_t *>(&hh);
                        hfrag[lo_off + wi] = pack_half2(r0, r1);
                    }
                    bar_sync(1, NC);
                    cur = j;
                }
                const int slot = wait_slot(u);
                const uint8_t *slotp = ring + (size_t)slot * a.slot_bytes;
                const int rg0 = oct * a.r2, nrg = min(a.r2, a.ng_d - rg0);
                const uint32_t gm = (((rowmask & 0xFFu) ? 1u : 0u) | ((rowmask & 0xFF00u) ? 2u : 0u)) & ngrp_rows;
                float acc[1][NGRP][4];
#pragma unroll
                for (int g = 0; g < NGRP; ++g)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[0][g][i] = 0.f;
                const bool mine = warp < nrg;
                if (!bad && mine) {
                    const uint8_t *rb = slotp + (size_t)warp * kc * a.rec;
                    const uint2 *hi2 = reinterpret_cast<const uint2 *>(hfrag);
                    const uint2 *lo2 = hi2 + NGRP * kbp * kWarp;
                    for (int ch = 0; ch < kc; ++ch) {
                        const uint8_t *recs[1] = {rb + (size_t)ch * a.rec};
                        mma_records<FMT, NGRP, 1, true>(recs, hi2, lo2, kbp, ch * CB, lane, gm, acc);
                    }
                }
                release_slot(slot);
                ++u;
                if (!bad && mine) {
                    const int rg = rg0 + warp;
#pragma unroll
                    for (int g = 0; g < NGRP; ++g)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = acc_xrow(lane, g, i);
                            if (r < a.M && ((rowmask >> r) & 1u)) {
                                const int s = ms->uslot[j][r];
                                const int n = rg * 16 + acc_wrow(lane, i);
                                a.part[((int64_t)r * (a.K + 1) + s) * a.H + n] =
                                    scalbnf(acc[0][g][i], 24 - (MB - 1) - ms->shift_h[r]);
                            }
                        }
                    __threadfence();
                    __syncwarp();
                    uint32_t old = 0;
                    if (lane == 0) old = atom_add_acq_rel(&a.rgcnt[rg], 1u);
                    old = __shfl_sync(0xffffffffu, old, 0);
                    if (old == (uint32_t)nU) {  // last of the nU + 1 experts for this row group
                        __threadfence();
                        for (int i = lane; i < a.M * 16; i += kWarp) {
                            const int r = i >> 4, n = rg * 16 + (i & 15);
                            float sum = 0.f;
                            for (int s = 0; s <= a.K; ++s) sum += __ldcg(&a.part[((int64_t)r * (a.K + 1) + s) * a.H + n]);
                            if (a.y) a.y[(int64_t)r * a.H + n] = sum;
                            if (a.h_out) {
                                const float hin = bf16_bits_to_f32(a.x[(int64_t)r * a.H + n]);
                                a.h_out[(int64_t)r * a.H + n] = f32_to_bf16_bits(hin + sum);
                            }
                        }
                        if (lane == 0) atomicExch(&a.rgcnt[rg], 0u);
                    }
                }
                if (bar_or(1, NC, bad)) {
                    abort_all();
                    goto done;
                }
            }
        }
    done:
        if (!dispatched) bar_arrive(2, kThreads);
    }
    __syncthreads();
    // ---- the last CTA out resets the cross-block counters for the next launch
    if (tid == 0) {
        __threadfence();
        const uint32_t old = atom_add_acq_rel(&a.ctrl[1], 1u);
        if (old == (uint32_t)(a.ncta - 1)) {
            for (int i = 0; i <= a.E; ++i) a.done1[i] = 0u;
            for (int i = 0; i < a.ng_d; ++i) a.rgcnt[i] = 0u;
            a.ctrl[0] = 0u;
            __threadfence();
            atomicExch(&a.ctrl[1], 0u);
        }
    }
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
struct MoePlan {
    Geometry gu, dn, sgu, sdn;
    int ngrp, ncta, nslot, slot_bytes, frag_bytes, scr_bytes, r2, noct, Fmax;
    size_t smem;
    size_t off_ctrl, off_done1, off_rgcnt, off_logits, off_hbuf, off_part, ws_bytes;
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
    p->scr_bytes = (int)align_up(std::max<size_t>((size_t)kConsumerWarps * 2 * p->ngrp * 128 * 4,
                                                  (size_t)m * (L->n_experts + 1) * 4),
                                 128);
    const int64_t gbh = p->gu.group_bytes();
    const int64_t gbf = std::max(p->dn.group_bytes(), p->sdn.group_bytes());
    p->r2 = (int)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(kConsumerWarps, 2 * gbh / gbf), p->dn.ng));
    p->noct = (int)((p->dn.ng + p->r2 - 1) / p->r2);
    const int nft = L->ffn / 16, nft_s = L->shared_ffn / 16;
    // grid: enough CTAs for the phase-1 units of the worst-case union, at most one per SM
    const int64_t worst_units = nft_s + (int64_t)std::min(L->n_experts, m * L->top_k) * nft;
    p->ncta = (int)std::max<int64_t>(1, std::min<int64_t>(di.sms, worst_units));
    const int rows_per_cta = (L->n_experts + 1 + p->ncta - 1) / p->ncta;
    int64_t slot = std::max<int64_t>(2 * gbh, (int64_t)p->r2 * gbf);
    slot = std::max<int64_t>(slot, (int64_t)rows_per_cta * L->hidden * 2);
    slot = (int64_t)align_up((size_t)slot, 128);
    const size_t fixed = align_up(align_up((size_t)p->frag_bytes + p->scr_bytes + sizeof(MoeMisc), 16) + 16 * 8, 128);
    if ((int64_t)di.smem_optin < (int64_t)fixed + 2 * slot) return fail(BFP_ESHAPE, "layer too large for shared memory");
    p->nslot = (int)std::min<int64_t>(8, ((int64_t)di.smem_optin - (int64_t)fixed) / slot);
    p->slot_bytes = (int)slot;
    p->smem = fixed + (size_t)p->nslot * slot;
    // workspace
    size_t o = kWsHeader;
    p->off_ctrl = o;
    o += 16;
    p->off_done1 = o;
    o = align_up(o + 4 * (size_t)(L->n_experts + 1), 16);
    p->off_rgcnt = o;
    o = align_up(o + 4 * (size_t)p->dn.ng, 256);
    p->off_logits = o;
    o = align_up(o + 4 * (size_t)m * (L->n_experts + 1), 256);
    p->off_hbuf = o;
    o = align_up(o + 4 * (size_t)m * (L->top_k + 1) * p->Fmax, 256);
    p->off_part = o;
    o = align_up(o + 4 * (size_t)m * (L->top_k + 1) * L->hidden, 256);
    p->ws_bytes = o;
    return BFP_OK;
}

template <int FMT, int NGRP>
static int launch_moe_t(const MoeArgs &a, const MoePlan &p, cudaStream_t st) {
    auto kern = moe_layer_kernel<FMT, NGRP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(moe_layer)");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ncta);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return cuda_fail(e, "launch moe_layer (cooperative)");
    return BFP_OK;
}

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
    if (!ws || ws_bytes < p.ws_bytes) return fail(BFP_EWORKSPACE, "workspace smaller than moe_workspace_size");
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
    a.done1 = reinterpret_cast<uint32_t *>(w + p.off_done1);
    a.rgcnt = reinterpret_cast<uint32_t *>(w + p.off_rgcnt);
    a.logits = reinterpret_cast<float *>(w + p.off_logits);
    a.hbuf = reinterpret_cast<float *>(w + p.off_hbuf);
    a.part = reinterpret_cast<float *>(w + p.off_part);
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
    a.nslot = p.nslot;
    a.slot_bytes = p.slot_bytes;
    a.frag_bytes = p.frag_bytes;
    a.scr_bytes = p.scr_bytes;
    a.wait = wait_cfg();
    a.wait_data = WaitCfg{kDefaultWaitIters, kDefaultWaitNanos};
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

int moe_stack_decode(const bfp_moe_layer *layers, int n_layers, const bfp_matrix *lm_head, uint16_t *h, int m,
                     float *logits, void *ws, size_t ws_bytes, bfp_stream_t stream) {
    size_t mb, lb, hb;
    int rc = stack_layout(layers, n_layers, lm_head, m, &mb, &lb, &hb);
    if (rc) return rc;
    if (!h || !logits) return fail(BFP_EINVAL, "null h or logits");
    if (!ws || ws_bytes < mb + lb + hb) return fail(BFP_EWORKSPACE, "workspace smaller than moe_stack_workspace_size");
    if (!aligned16(h) || !aligned16(logits) || !aligned16(ws)) return fail(BFP_EALIGN, "pointers must be 16-byte aligned");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint16_t *hb2 = reinterpret_cast<uint16_t *>(w + mb + lb);
    uint16_t *cur = h, *nxt = hb2;
    for (int l = 0; l < n_layers; ++l) {
        rc = moe_launch(&layers[l], cur, m, 1, nullptr, nxt, nullptr, nullptr, ws, mb, st);
        if (rc) return rc;
        std::swap(cur, nxt);
    }
    if (cur != h) {
        cudaError_t e = cudaMemcpyAsync(h, cur, (size_t)m * layers[0].hidden * 2, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e, "copy final h");
    }
    return linear_launch_ex(lm_head, h, m, layers[0].hidden, logits, nullptr, lm_head->n,
                            reinterpret_cast<uint32_t *>(w), w + mb, lb, st, 1);
}

}  // extern "C"

// ----------------------------------------------------------------------------
// moe_decode_layer_static: the same layer for callers that cannot allocate
// device memory. Its scratch is one file-scope device array of a fixed size,
// shared by every call on a device and kept for the life of the process.
// ----------------------------------------------------------------------------
namespace bfp {

constexpr size_t kStaticScratchBytes = size_t(2) << 20;  // 2 MiB: a full-size layer at 16 rows needs ~1.5 MiB
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
    if (p.ws_bytes > kStaticScratchBytes)
        return fail(BFP_EWORKSPACE, "this layer needs " + std::to_string(p.ws_bytes) +
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
    return moe_launch(layer, x, m, 0, y, nullptr, topk_idx, topk_w, ws, kStaticScratchBytes, st);
}
