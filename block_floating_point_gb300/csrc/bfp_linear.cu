// Dense BFP decode projection (bfp_linear), device decode (bfp_unpack_device)
// and the workspace entry points.
//
// Dense projections and the LM head are BFP8 (Qwen3.6-35B-A3B card, "Precision
// as served"); every row of a decode step multiplies against one pass over the
// weights (Qwen3.8-27B s27v6 card, "Multi-user decode").
//
// GB300 design: the weight stream is the whole cost (1.0625 or 0.5625 bytes
// per weight, read once). A grid of one 512-thread CTA per SM gives every CTA
// the same number of whole 16-row groups. Each row group is cut into S parts
// along k (S > 1 only when the CTA has fewer row groups than warps), and each
// of the 16 warps takes whole parts: it streams the part's tile records
// through two shared-memory slots of its own with 1D bulk copies (the TMA
// engine; lane 0 refills a slot as soon as the warp is done with it),
// unpacks each 16-value block into an fp16 A fragment and runs one mma.sync
// k16 step per block. The parts of a split row group meet in shared memory:
// the last one to finish adds them in order (results do not depend on
// timing) and writes the outputs. Nothing crosses CTAs.
#include <algorithm>
#include <mutex>
#include <vector>

#include "bfp_launch.h"
#include "bfp_tc.h"
#include "bfp_tiles.cuh"

namespace bfp {

using namespace dev;

// ----------------------------------------------------------------------------
// Device info (cached per device)
// ----------------------------------------------------------------------------
int device_info(DeviceInfo *out) {
    static std::mutex mu;
    static std::vector<DeviceInfo> cache;
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(mu);
    if ((int)cache.size() <= d) cache.resize(d + 1);
    if (cache[d].device != d) {
        DeviceInfo info;
        info.device = d;
        e = cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, d);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        e = cudaDeviceGetAttribute(&info.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(smem opt-in)");
        cache[d] = info;
    }
    *out = cache[d];
    return BFP_OK;
}


int set_smem_attr(const void *kernel, int smem, const char *what) {
    struct Entry {
        const void *k;
        int device, smem;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry &x : done)
        if (x.k == kernel && x.device == d && x.smem >= smem) return BFP_OK;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail(e, what);
    for (Entry &x : done)
        if (x.k == kernel && x.device == d) {
            x.smem = smem;
            return BFP_OK;
        }
    done.push_back(Entry{kernel, d, smem});
    return BFP_OK;
}

// ----------------------------------------------------------------------------
// bfp_linear kernel
// ----------------------------------------------------------------------------
constexpr int kLinWarps = 16;
constexpr int kLinThreads = kLinWarps * 32;
constexpr int kLinMaxRows = 32;
constexpr int kLinInplaceRegs = 8;  // fragment pairs per thread and group when four groups are built in place

struct LinearArgs {
    const uint8_t *w;
    int64_t n;
    int ng, k, kc, kbp, rec;
    const uint16_t *x;
    int64_t ldx;
    int m, norm;
    float eps;
    float *y;
    uint16_t *yb;
    int64_t ldy;
    uint32_t *status;
    int ncta, S, chw, nsw, slot_bytes, frag_bytes, scr_bytes, stage_off;
    int ldxs;  // row stride of the staged activation rows (elements)
    WaitCfg wait;
    // greedy next token (nullable): tokens[r] = the index of row r's largest output; gcount and gpart (the
    // workspace body) take the CTAs' keys, the last CTA to finish reduces them
    int32_t *tokens;
    uint32_t *gcount;
    unsigned long long *gpart;  // [ncta][kLinMaxRows]
};

// Shared-memory bookkeeping of one CTA.
struct LinMisc {
    alignas(16) float esc[kLinWarps][rec_scale_floats<4, 1>()];  // per-warp block scales (mma_records)
    uint64_t stage_full;                                          // the activation rows landed
    int shift[32];
    float inv[32];
    float2 red[kLinWarps];  // activation row statistics per (row, segment)
    int cnt[kLinWarps];     // parts finished per row group of a split
    int flags[4];        // [0] abort, [1] this CTA reduces the greedy keys
    unsigned long long gbest[kLinWarps][kLinMaxRows];  // greedy: each warp's best key per row
};

// Greedy key of output (value v, index i): an order-preserving image of v (with -0 folded into +0) above the
// complement of i, so the unsigned maximum is the largest value and, among equal values, the lowest index.
// NaN outputs are given key 0 by the caller (never chosen; a row with nothing else gives index 0).
__device__ __forceinline__ unsigned long long lin_greedy_key(float v, int64_t i) {
    v += 0.0f;
    const uint32_t u = __float_as_uint(v);
    const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)k << 32) | (0xFFFFFFFFu - (uint32_t)i);
}
__device__ __forceinline__ unsigned long long lin_umax(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

template <int FMT, int NGRP>
__global__ void __launch_bounds__(kLinThreads, 1) bfp_linear_kernel(const __grid_constant__ LinearArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int NW = kLinWarps;
    constexpr int NC = NW * kWarp;
    constexpr int MB = FMT == 4 ? 3 : 7;
    constexpr int CB = FMT == 4 ? 4 : 2;
    uint32_t *frag = reinterpret_cast<uint32_t *>(smem);
    LinMisc *lm = reinterpret_cast<LinMisc *>(smem + a.frag_bytes + a.scr_bytes);
    const size_t bar_off = align_up(a.frag_bytes + a.scr_bytes + sizeof(LinMisc), 16);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + bar_off);  // [NW][nsw]
    uint8_t *ring = smem + align_up(bar_off + 8 * NW * a.nsw, 128);
    // the activation rows, before the streams start: in the ring's tail, or (four activation groups) in the
    // fragment area itself, turned into fragments in place
    uint8_t *stage = NGRP == 4 ? smem : ring + a.stage_off;
    volatile int *flags = lm->flags;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int rg0 = (int)((int64_t)c * a.ng / a.ncta), rg1 = (int)((int64_t)(c + 1) * a.ng / a.ncta);
    const int S = a.S, items = (rg1 - rg0) * S;

    if (tid <= NW * a.nsw) {  // one barrier per thread
        mbar_init(tid < NW * a.nsw ? &full[tid] : &lm->stage_full, 1);
        mbar_fence_init();
    }
    if (tid < NW) lm->cnt[tid] = 0;
    if (tid < 4) lm->flags[tid] = 0;
    // dependent launch: the next kernel may take the SMs as this grid's CTAs leave; no global memory
    // is touched before the previous kernel on the stream has finished (grid_dep_wait below)
    grid_dep_launch_dependents();
    __syncthreads();
    bool bad = false;
    // ---- this warp's stream: items it = warp, warp + NW, ...; item it = part it % S of row group
    //      rg0 + it / S, i.e. records [part * kc / S, (part + 1) * kc / S) of the group, in chunks
    //      of chw records through the warp's nsw slots (lane 0 issues, every lane keeps the cursor)
    uint8_t *const my_slots = ring + (size_t)warp * a.nsw * a.slot_bytes;
    uint64_t *const my_full = full + warp * a.nsw;
    int iss = 0, is_slot = 0, cu = 0, cu_slot = 0;
    uint32_t cu_par = 0;
    int it_iss = warp;  // next item to issue
    const uint8_t *src = nullptr;
    int s_left = 0;
    auto issue_next = [&]() {
        if (bad) return;
        if (s_left <= 0) {
            if (it_iss >= items) return;
            const int rg = rg0 + it_iss / S, part = it_iss % S;
            const int r0 = part * a.kc / S, r1 = (part + 1) * a.kc / S;
            src = a.w + ((int64_t)rg * a.kc + r0) * a.rec;
            s_left = r1 - r0;
            it_iss += NW;
        }
        const uint32_t b = (uint32_t)min(a.chw, s_left) * a.rec;
        if (lane == 0) {
            uint64_t *fb = my_full + is_slot;
            const uint64_t pol = l2_evict_first();  // the weights are read once per launch
            fence_proxy_async_shared();              // this warp's reads of the slot come first
            mbar_arrive_expect_tx(fb, b);
            bulk_g2s_hint(my_slots + (size_t)is_slot * a.slot_bytes, src, b, fb, pol);
        }
        src += b;
        s_left -= a.chw;
        ++iss;
        if (++is_slot == a.nsw) is_slot = 0;
    };
    auto take_item = [&]() -> const uint8_t * {
        if (!bad && flags[0]) bad = true;
        if (!bad && !__all_sync(0xffffffffu, mbar_wait(my_full + cu_slot, cu_par, a.wait, flags))) {
            bad = true;
            if (lane == 0) {
                flags[0] = 1;
                raise_status(a.status, kStatusTimeout);
            }
        }
        return my_slots + (size_t)cu_slot * a.slot_bytes;
    };
    auto give_item = [&]() {  // a slot whose data never came is kept (the drain below waits for it)
        __syncwarp();
        if (bad) return;
        issue_next();
        ++cu;
        if (++cu_slot == a.nsw) {
            cu_slot = 0;
            cu_par ^= 1u;
        }
    };
    // The weights do not depend on the activations: a warp whose slots lie below the stage starts
    // its stream before the rows land. The rows' copies are requested first, so that they do not
    // queue behind the CTA's weight chunks (measured after an L2 flush: 16 rows landed 1.6 us after
    // the CTA started instead of 3.1 us).
    const bool early = NGRP == 4 || (size_t)(warp + 1) * a.nsw * a.slot_bytes <= (size_t)a.stage_off;
    grid_dep_wait();
    if (tid == 0) {  // the activation rows, one copy per row (rows are ldx apart in global memory)
        mbar_arrive_expect_tx(&lm->stage_full, (uint32_t)a.m * a.k * 2);
        for (int r = 0; r < a.m; ++r)
            bulk_g2s(stage + (size_t)r * a.ldxs * 2, a.x + (int64_t)r * a.ldx, (uint32_t)a.k * 2, &lm->stage_full);
    }
    __syncthreads();
    if (early)
        for (int i = 0; i < a.nsw; ++i) issue_next();
    if (!__all_sync(0xffffffffu, mbar_wait(&lm->stage_full, 0u, a.wait, nullptr))) bad = true;
    uint16_t *const xs = reinterpret_cast<uint16_t *>(stage);
    // (inlined: 0.3-0.5 us less than the calls at 1 and 16 rows)
    if constexpr (NGRP == 4) {
        act_rows_prepare_body<NC>(xs, a.ldxs, a.m, a.k, a.norm != 0, a.eps, lm->shift, lm->inv, lm->red, 1, warp,
                                  lane);
        act_rows_frags_inplace_body<NC>(xs, a.ldxs, a.m, a.k, a.kbp, lm->shift, frag, 1, tid);
    } else {
        act_rows_stats_frags_body<NC>(xs, a.ldxs, a.m, a.k, a.kbp, NGRP, a.norm != 0, a.eps, lm->shift, frag, 1,
                                      warp, lane);
    }
    // every warp is past its reads of the stage (the barrier ending act_rows_frags): the rest
    // of the streams may start
    if (!early)
        for (int i = 0; i < a.nsw; ++i) issue_next();

    const uint2 *frag2 = reinterpret_cast<const uint2 *>(frag);
    unsigned long long gk[NGRP][2];  // greedy: this lane's best keys, rows 8 g + 2 (lane & 3) + j
#pragma unroll
    for (int g = 0; g < NGRP; ++g) gk[g][0] = gk[g][1] = 0ull;
    for (int it = warp; it < items; it += NW) {
        const int rg = rg0 + it / S, part = it % S;
        const int r0 = part * a.kc / S, r1 = (part + 1) * a.kc / S;
        float acc[1][NGRP][4];
#pragma unroll
        for (int g = 0; g < NGRP; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[0][g][i] = 0.f;
        for (int k0 = r0; k0 < r1; k0 += a.chw) {
            const int n = min(a.chw, r1 - k0);
            const uint8_t *sp = take_item();
            if (!bad)
                for (int ch = 0; ch < n; ++ch) {
                    const uint8_t *recs[1] = {sp + (size_t)ch * a.rec};
                    mma_records<FMT, NGRP, 1, false>(recs, frag2, nullptr, a.kbp, (k0 + ch) * CB, lane, lm->esc[warp],
                                                     acc);
                }
            give_item();
        }
        if (bad) continue;
        if (S > 1) {
            // part of a split row group: store the tile; the last part to finish adds the parts in
            // order and writes the outputs. Items < NW then (item it is warp it's only one), so a warp's
            // own slots are free once its item is done and hold its tile.
            auto part_tile = [&](int w) {
                return reinterpret_cast<float *>(ring + (size_t)w * a.nsw * a.slot_bytes);
            };
            float *mine = part_tile(it);
#pragma unroll
            for (int g = 0; g < NGRP; ++g)
#pragma unroll
                for (int i = 0; i < 4; ++i) mine[(g * 4 + i) * kWarp + lane] = acc[0][g][i];
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                last = atomicAdd(&lm->cnt[it / S], 1) == S - 1;
            }
            if (!__shfl_sync(0xffffffffu, last, 0)) continue;
            __threadfence_block();
#pragma unroll
            for (int g = 0; g < NGRP; ++g)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float v = 0.f;
                    for (int q = 0; q < S; ++q) v += part_tile((it / S) * S + q)[(g * 4 + i) * kWarp + lane];
                    acc[0][g][i] = v;
                }
        }
#pragma unroll
        for (int g = 0; g < NGRP; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = acc_xrow(lane, g, i);
                const int64_t nrow = (int64_t)rg * 16 + acc_wrow(lane, i);
                if (r < a.m && nrow < a.n) {
                    const float v = mul_pow2(acc[0][g][i], 24 - (MB - 1) - lm->shift[r]);
                    if (a.y) a.y[(int64_t)r * a.ldy + nrow] = v;
                    if (a.yb) a.yb[(int64_t)r * a.ldy + nrow] = f32_to_bf16_bits(v);
                    if (v == v) gk[g][i & 1] = lin_umax(gk[g][i & 1], lin_greedy_key(v, nrow));
                }
            }
    }
    // greedy next token: each warp's best key per row (lanes of equal lane & 3 hold the same rows), the
    // CTA's best per row to the workspace, and the last CTA to finish reduces every CTA's keys
    if (a.tokens) {
#pragma unroll
        for (int g = 0; g < NGRP; ++g)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
#pragma unroll
                for (int o = 4; o < kWarp; o <<= 1) gk[g][j] = lin_umax(gk[g][j], __shfl_xor_sync(0xffffffffu, gk[g][j], o));
            }
        if (lane < 4) {
#pragma unroll
            for (int g = 0; g < NGRP; ++g) {
                lm->gbest[warp][8 * g + 2 * lane] = gk[g][0];
                lm->gbest[warp][8 * g + 2 * lane + 1] = gk[g][1];
            }
        }
        __syncthreads();
        if (tid < a.m) {
            unsigned long long b = 0ull;
            for (int w = 0; w < NW; ++w) b = lin_umax(b, lm->gbest[w][tid]);
            __stcg(a.gpart + (int64_t)c * kLinMaxRows + tid, b);
            __threadfence();  // the key reaches L2 before the count
        }
        __syncthreads();
        if (tid == 0) lm->flags[1] = atomicAdd(a.gcount, 1u) == (uint32_t)(a.ncta - 1);
        __syncthreads();
        if (lm->flags[1]) {
            // 16 threads per row, each over every 16th CTA's key (independent loads in flight), then a
            // reduction over the 16 lanes
            __threadfence();
            const int r = tid >> 4, q0 = tid & 15;
            unsigned long long b = 0ull;
            if (r < a.m) {
#pragma unroll 4
                for (int q = q0; q < a.ncta; q += 16) b = lin_umax(b, __ldcg(a.gpart + (int64_t)q * kLinMaxRows + r));
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) b = lin_umax(b, __shfl_xor_sync(0xffffffffu, b, o));
            if (r < a.m && q0 == 0)
                a.tokens[r] = b == 0ull ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)(b & 0xFFFFFFFFull));
            if (tid == 0) *a.gcount = 0u;  // every CTA has counted: ready for the next call
        }
    }
    // No copy may still be landing in shared memory when the CTA exits (every path).
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
        if (tid == 0) mbar_wait(&lm->stage_full, 0u, drain, nullptr);
    }
    __syncthreads();
}

// ----------------------------------------------------------------------------
// bfp_unpack_device: every block through the A-fragment unpack and one MMA
// against unit columns, then scaled by 2^(24 + E - 127 - (mb - 1)).
// ----------------------------------------------------------------------------
template <int FMT>
__global__ void bfp_unpack_kernel(const uint8_t *w, int64_t n, int k, int kc, int rec, int64_t nrec, float *out) {
    constexpr int MB = FMT == 4 ? 3 : 7;
    constexpr int CB = FMT == 4 ? 4 : 2;
    const int64_t q = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (q >= nrec) return;
    const int64_t rg = q / kc;
    const int c = (int)(q - rg * kc);
    const uint8_t *rp = w + q * rec;
    const int g = lane >> 2, t = lane & 3;
    const uint4 wq = *reinterpret_cast<const uint4 *>(rp + 16 * lane);
    const uint32_t one = 0x3C00u;  // fp16 1.0
    const uint32_t id = ((2 * t == g) ? one : 0u) | ((2 * t + 1 == g) ? one << 16 : 0u);
    const int kb = k / 16;
    for (int b = 0; b < CB; ++b) {
        const int blk = c * CB + b;
        if (blk >= kb) break;
        uint32_t a[4];
        uint32_t ew;
        int eb0, eb1;
        if (FMT == 4) {
            const uint32_t ws[4] = {wq.x, wq.y, wq.z, wq.w};
            unpack_bfp4(ws[b], a);
            ew = *reinterpret_cast<const uint32_t *>(rp + 512 + 8 * g + 4 * (b >> 1));
            eb0 = 2 * (b & 1);
        } else {
            if (b == 0)
                unpack_bfp8(wq.x, wq.y, a);
            else
                unpack_bfp8(wq.z, wq.w, a);
            ew = *reinterpret_cast<const uint32_t *>(rp + 512 + 4 * g);
            eb0 = 2 * b;
        }
        eb1 = eb0 + 1;
        float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(lo, a, id, 0u);  // columns 0..7 of the block
        mma16816(hi, a, 0u, id);  // columns 8..15
        const int E0 = (ew >> (8 * eb0)) & 0xFF, E1 = (ew >> (8 * eb1)) & 0xFF;
        const int64_t row0 = rg * 16 + g, row1 = row0 + 8;
        const int col = blk * 16 + 2 * t;
        if (row0 < n) {
            float *o = out + row0 * k + col;
            o[0] = scalbnf(lo[0], 24 + E0 - 127 - (MB - 1));
            o[1] = scalbnf(lo[1], 24 + E0 - 127 - (MB - 1));
            o[8] = scalbnf(hi[0], 24 + E0 - 127 - (MB - 1));
            o[9] = scalbnf(hi[1], 24 + E0 - 127 - (MB - 1));
        }
        if (row1 < n) {
            float *o = out + row1 * k + col;
            o[0] = scalbnf(lo[2], 24 + E1 - 127 - (MB - 1));
            o[1] = scalbnf(lo[3], 24 + E1 - 127 - (MB - 1));
            o[8] = scalbnf(hi[2], 24 + E1 - 127 - (MB - 1));
            o[9] = scalbnf(hi[3], 24 + E1 - 127 - (MB - 1));
        }
    }
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
struct LinearPlan {
    int ngrp, ncta, S, chw, nsw, slot_bytes, frag_bytes, scr_bytes, stage_off, ldxs;
    size_t smem;
    size_t ws_bytes;  // workspace after its header (none: nothing crosses CTAs)
};

static int plan_linear(const Geometry &g, int m, LinearPlan *p) {
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    p->ngrp = m > 16 ? 4 : (m > 8 ? 2 : 1);
    const int kbp = (int)(g.kc * g.cb);
    p->frag_bytes = p->ngrp * kbp * 32 * 8;
    // four groups: the fragments are built in place from the staged rows, group by group, each thread
    // holding its share of a group (kLinInplaceRegs fragment pairs) in registers
    if (p->ngrp == 4 && (int64_t)kbp * 32 > (int64_t)kLinThreads * kLinInplaceRegs)
        return fail(BFP_ESHAPE, "more than 16 rows needs k <= 2048");
    // grid: the same number of whole row groups per CTA (at most one CTA per SM)
    const int64_t per = (g.ng + di.sms - 1) / di.sms;
    p->ncta = (int)((g.ng + per - 1) / per);
    // parts per row group: every warp gets one when a CTA has fewer row groups than warps
    p->S = 1;
    while (per * p->S * 2 <= kLinWarps && p->S * 2 <= g.kc) p->S *= 2;
    p->scr_bytes = 0;  // the parts of a split row group meet in their warps' own slots
    p->ldxs = (int)g.k;
    if (p->ngrp == 4) {
        // rows staged in the fragment area: a stride of 8 mod 64 elements (4 mod 32 words) puts the 8 rows
        // a warp reads at once in different banks, and at least 16 kbp elements makes a group's staged
        // rows (8 ldxs elements) at least as long as its fragments (kbp * 256 bytes), so the groups can be
        // built in place from the first one up; the area grows by what the rows need beyond the fragments
        p->ldxs = (int)std::max<int64_t>(g.k, (int64_t)kbp * 16);
        p->ldxs += (8 - p->ldxs % 64 + 64) % 64;
        const int64_t rows_bytes = (int64_t)m * p->ldxs * 2;
        if (rows_bytes > p->frag_bytes) p->scr_bytes = (int)align_up((size_t)(rows_bytes - p->frag_bytes), 16);
    }
    const size_t stage = p->ngrp == 4 ? 0 : align_up((size_t)m * g.k * 2, 128);
    const size_t base = align_up((size_t)p->frag_bytes + p->scr_bytes + sizeof(LinMisc), 16);
    const int64_t avail = (int64_t)di.smem_optin - (int64_t)base - 128;
    // chunks of up to 8 records, smaller when two slots per warp would not fit
    p->nsw = 0;
    for (int chw : {8, 6, 4, 2, 1}) {
        p->chw = (int)std::min<int64_t>(chw, g.kc);
        p->slot_bytes = p->chw * g.rec;
        p->nsw = (int)std::min<int64_t>(4, avail / ((int64_t)kLinWarps * (p->slot_bytes + 8)));
        if (p->nsw >= 2 && (int64_t)p->nsw * p->slot_bytes >= (int64_t)p->ngrp * 128 * 4) break;
        p->nsw = 0;
    }
    if (p->nsw < 2) return fail(BFP_ESHAPE, "k too large for the activation fragments in shared memory");
    const size_t ring = (size_t)kLinWarps * p->nsw * p->slot_bytes;
    if (ring < stage) return fail(BFP_ESHAPE, "activation rows do not fit in shared memory");
    p->stage_off = (int)(ring - stage);
    p->smem = align_up(base + 8 * (size_t)kLinWarps * p->nsw, 128) + ring;
    p->ws_bytes = 256 + (size_t)p->ncta * kLinMaxRows * 8;  // greedy token: count, then one key per (CTA, row)
    return BFP_OK;
}

template <int FMT, int NGRP>
static int launch_linear_t(const LinearArgs &a, const LinearPlan &p, cudaStream_t st) {
    auto kern = bfp_linear_kernel<FMT, NGRP>;
    int rc = set_smem_attr(reinterpret_cast<const void *>(kern), (int)p.smem, "cudaFuncSetAttribute(bfp_linear)");
    if (rc) return rc;
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ncta);
    cfg.blockDim = dim3(kLinThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // no waits between CTAs
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return cuda_fail(e, "launch bfp_linear");
    return BFP_OK;
}

// Shared by bfp_linear and the decode stack's LM head (norm = RMS-normalise x first).
// status: the workspace status word; body: the rest of the workspace (unused by this kernel).
int linear_launch_ex(const bfp_matrix *w, const uint16_t *x, int m, int64_t ldx, float *y, uint16_t *y_bf16,
                     int64_t ldy, uint32_t *status, void *body, size_t body_bytes, cudaStream_t st, int norm,
                     int32_t *tokens) {
    Geometry g;
    int rc = check_matrix(w, &g, true);
    if (rc) return rc;
    if (m < 1 || m > 32) return fail(BFP_ESHAPE, "m must be in [1, 32]");
    if (!x || (!y && !y_bf16 && !tokens)) return fail(BFP_EINVAL, "null x or no output");
    if (tokens && ((uintptr_t)tokens & 3u)) return fail(BFP_EALIGN, "tokens must be 4-byte aligned");
    if (ldx < g.k || ldx % 8 != 0) return fail(BFP_EALIGN, "ldx must be >= k and a multiple of 8");
    if ((y || y_bf16) && ldy < g.n) return fail(BFP_EINVAL, "ldy < n");
    if (!aligned16(x) || (y && !aligned16(y)) || (y_bf16 && !aligned16(y_bf16)))
        return fail(BFP_EALIGN, "device pointers must be 16-byte aligned");
    LinearPlan p;
    rc = plan_linear(g, m, &p);
    if (rc) return rc;
    if (body_bytes < p.ws_bytes) return fail(BFP_EWORKSPACE, "workspace smaller than bfp_linear_workspace_size");
    // the tcgen05 kernel when asked for (bfp_set_linear_path(2)) and the shape fits it
    if (!tokens && !norm && linear_path() == 2) {
        rc = linear_tc_launch(g, static_cast<const uint8_t *>(w->data), x, m, ldx, y, y_bf16, ldy, status, st);
        if (rc != kTcNotApplicable) return rc;
    }
    LinearArgs a;
    a.w = static_cast<const uint8_t *>(w->data);
    a.n = g.n;
    a.ng = (int)g.ng;
    a.k = (int)g.k;
    a.kc = (int)g.kc;
    a.kbp = (int)(g.kc * g.cb);
    a.rec = g.rec;
    a.x = x;
    a.ldx = ldx;
    a.m = m;
    a.norm = norm;
    a.eps = 1e-6f;
    a.y = y;
    a.yb = y_bf16;
    a.ldy = ldy;
    a.status = status;
    a.ncta = p.ncta;
    a.S = p.S;
    a.chw = p.chw;
    a.nsw = p.nsw;
    a.slot_bytes = p.slot_bytes;
    a.frag_bytes = p.frag_bytes;
    a.scr_bytes = p.scr_bytes;
    a.stage_off = p.stage_off;
    a.ldxs = p.ldxs;
    a.wait = WaitCfg{kDefaultWaitIters, kDefaultWaitNanos};  // only this CTA's own copies are waited on
    a.tokens = tokens;
    a.gcount = static_cast<uint32_t *>(body);
    a.gpart = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(body) + 256);
    if (g.fmt == BFP_FMT_BFP4)
        return p.ngrp == 1 ? launch_linear_t<4, 1>(a, p, st)
                           : p.ngrp == 2 ? launch_linear_t<4, 2>(a, p, st) : launch_linear_t<4, 4>(a, p, st);
    return p.ngrp == 1 ? launch_linear_t<8, 1>(a, p, st)
                       : p.ngrp == 2 ? launch_linear_t<8, 2>(a, p, st) : launch_linear_t<8, 4>(a, p, st);
}

// Bytes of the workspace after its header (the kernel keeps everything in shared memory: none).
int linear_ws_body_bytes(const bfp_matrix *w, int m, size_t *bytes) {
    Geometry g;
    int rc = check_matrix(w, &g, false);
    if (rc) return rc;
    if (m < 1 || m > 32) return fail(BFP_ESHAPE, "m must be in [1, 32]");
    LinearPlan p;
    rc = plan_linear(g, m, &p);
    if (rc) return rc;
    *bytes = p.ws_bytes;
    return BFP_OK;
}

}  // namespace bfp

using namespace bfp;

extern "C" {

int bfp_unpack_device(const bfp_matrix *w, float *out, bfp_stream_t stream) {
    Geometry g;
    int rc = check_matrix(w, &g, true);
    if (rc) return rc;
    if (!out) return fail(BFP_EINVAL, "null output");
    if (!aligned16(out)) return fail(BFP_EALIGN, "out not 16-byte aligned");
    const int64_t nrec = g.ng * g.kc;
    const int wpb = 8;
    const int64_t blocks = (nrec + wpb - 1) / wpb;
    if (blocks > 0x7FFFFFFF) return fail(BFP_ESHAPE, "matrix too large for bfp_unpack_device");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t *src = static_cast<const uint8_t *>(w->data);
    if (g.fmt == BFP_FMT_BFP4)
        bfp_unpack_kernel<4><<<(unsigned)blocks, wpb * 32, 0, st>>>(src, g.n, (int)g.k, (int)g.kc, g.rec, nrec, out);
    else
        bfp_unpack_kernel<8><<<(unsigned)blocks, wpb * 32, 0, st>>>(src, g.n, (int)g.k, (int)g.kc, g.rec, nrec, out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch bfp_unpack_device");
    return BFP_OK;
}

int bfp_linear_workspace_size(const bfp_matrix *w, int m, size_t *bytes) {
    if (!bytes) return fail(BFP_EINVAL, "bytes is null");
    size_t body = 0;
    int rc = linear_ws_body_bytes(w, m, &body);
    if (rc) return rc;
    *bytes = kWsHeader + body;
    return BFP_OK;
}

int bfp_linear(const bfp_matrix *w, const uint16_t *x, int m, int64_t ldx, float *y, uint16_t *y_bf16, int64_t ldy,
               void *ws, size_t ws_bytes, bfp_stream_t stream) {
    if (!ws || ws_bytes < kWsHeader) return fail(BFP_EWORKSPACE, "workspace null or smaller than its header");
    return linear_launch_ex(w, x, m, ldx, y, y_bf16, ldy, static_cast<uint32_t *>(ws),
                            static_cast<uint8_t *>(ws) + kWsHeader, ws_bytes - kWsHeader,
                            reinterpret_cast<cudaStream_t>(stream), 0, nullptr);
}

int bfp_linear_greedy(const bfp_matrix *w, const uint16_t *x, int m, int64_t ldx, float *y, int64_t ldy,
                      int32_t *tokens, void *ws, size_t ws_bytes, bfp_stream_t stream) {
    if (!tokens) return fail(BFP_EINVAL, "null tokens");
    if (!ws || ws_bytes < kWsHeader) return fail(BFP_EWORKSPACE, "workspace null or smaller than its header");
    return linear_launch_ex(w, x, m, ldx, y, nullptr, ldy, static_cast<uint32_t *>(ws),
                            static_cast<uint8_t *>(ws) + kWsHeader, ws_bytes - kWsHeader,
                            reinterpret_cast<cudaStream_t>(stream), 0, tokens);
}

int bfp_workspace_init(void *ws, size_t ws_bytes, bfp_stream_t stream) {
    if (!ws || ws_bytes < kWsHeader) return fail(BFP_EWORKSPACE, "workspace null or smaller than its header");
    cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
    return BFP_OK;
}

int bfp_workspace_status(const void *ws, int *status, bfp_stream_t stream) {
    if (!ws || !status) return fail(BFP_EINVAL, "null argument");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t word = 0;
    e = cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read workspace status");
    *status = word == 0 ? BFP_OK : -(int)word;
    return BFP_OK;
}

}  // extern "C"
