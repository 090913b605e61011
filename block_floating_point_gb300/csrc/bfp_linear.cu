// Dense BFP decode projection (bfp_linear), device decode (bfp_unpack_device)
// and the workspace entry points.
//
// Dense projections and the LM head are BFP8 (Qwen3.6-35B-A3B card, "Precision
// as served"); every row of a decode step multiplies against one pass over the
// weights (Qwen3.8-27B s27v6 card, "Multi-user decode").
//
// GB300 design: the weight stream is the whole cost (1.0625 or 0.5625 bytes
// per weight, read once). A persistent grid of one 288-thread CTA per SM walks
// an equal share of the matrix's tile records (stream-K: shares may start and
// end inside a row group). One producer warp streams the share into a ring of
// shared-memory slots with 1D bulk copies (cp.async.bulk, the TMA engine)
// completing on mbarriers; eight consumer warps unpack each 16-value block
// into an fp16 A fragment and run one mma.sync k16 step per block. A row group
// split between CTAs is finished by whichever CTA arrives last (fixed-order
// sum of the partials, so results do not depend on timing).
#include <algorithm>
#include <mutex>
#include <vector>

#include "bfp_launch.h"
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


// ----------------------------------------------------------------------------
// bfp_linear kernel
// ----------------------------------------------------------------------------
struct LinearArgs {
    const uint8_t *w;
    int64_t n, ng;
    int k, kc, kbp, rec;
    const uint16_t *x;
    int64_t ldx;
    int m, norm;
    float eps;
    float *y;
    uint16_t *yb;
    int64_t ldy;
    uint32_t *status, *cnt;
    float *part;
    int ncta, nslot, slot_recs, slot_bytes, frag_bytes;
    WaitCfg wait;
};

// CTA c's share of the record line [0, R): [floor(cR/ncta), floor((c+1)R/ncta)).
__device__ __forceinline__ int64_t share_start(int64_t c, int64_t R, int ncta) { return c * R / ncta; }
__device__ __forceinline__ int cta_of(int64_t q, int64_t R, int ncta) {
    int c = (int)(q * ncta / R);
    while (c + 1 < ncta && share_start(c + 1, R, ncta) <= q) ++c;
    while (c > 0 && share_start(c, R, ncta) > q) --c;
    return c;
}

constexpr int kLinEsc = 256;                                                 // offset of the per-warp scale scratch
constexpr int kLinMisc = kLinEsc + kConsumerWarps * rec_scale_floats<4, 1>() * 4;  // shift[16], inv[16], flags, scales

template <int FMT, int NGRP>
__global__ void __launch_bounds__(kThreads, 1) bfp_linear_kernel(const LinearArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int NW = kConsumerWarps;
    constexpr int TILE = NGRP * 128;  // accumulator values per 16-row group
    constexpr int MB = FMT == 4 ? 3 : 7;
    constexpr int CB = FMT == 4 ? 4 : 2;
    uint32_t *frag = reinterpret_cast<uint32_t *>(smem);
    float *scr = reinterpret_cast<float *>(smem + a.frag_bytes);
    int *shift = reinterpret_cast<int *>(scr + NW * TILE);
    float *inv = reinterpret_cast<float *>(shift + 16);
    volatile int *flags = reinterpret_cast<volatile int *>(inv + 16);
    float *esc = reinterpret_cast<float *>(smem + a.frag_bytes + NW * TILE * 4 + kLinEsc) +
                 (threadIdx.x >> 5) * rec_scale_floats<4, 1>();  // this warp's scale scratch
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.frag_bytes + NW * TILE * 4 + kLinMisc);
    uint64_t *empty = full + a.nslot;
    uint8_t *ring = smem + align_up(a.frag_bytes + NW * TILE * 4 + kLinMisc + 16 * a.nslot, 128);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int64_t R = a.ng * a.kc;
    const int64_t s = share_start(c, R, a.ncta), e = share_start(c + 1, R, a.ncta);

    if (tid == 0) {
        for (int i = 0; i < a.nslot; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
        }
        flags[0] = 0;
        flags[1] = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == NW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int64_t u = 0;
            bool bad = false;
            // the activation rows first, 8 rows per slot (the fragments are built from them)
            for (int r0 = 0; r0 < a.m; r0 += 8) {
                const int slot = (int)(u % a.nslot);
                const int nr = min(8, a.m - r0);
                mbar_arrive_expect_tx(&full[slot], (uint32_t)nr * a.k * 2);
                for (int r = 0; r < nr; ++r)  // one copy per row: rows are ldx apart in global memory
                    bulk_g2s(ring + (size_t)slot * a.slot_bytes + (size_t)r * a.k * 2, a.x + (int64_t)(r0 + r) * a.ldx,
                             (uint32_t)a.k * 2, &full[slot]);
                ++u;
            }
            for (int64_t pos = s; pos < e;) {
                const int64_t rg = pos / a.kc;
                const int c0 = (int)(pos - rg * a.kc);
                const int len = (int)min64(min64(e - pos, a.kc - c0), a.slot_recs);
                const int slot = (int)(u % a.nslot);
                const int64_t use = u / a.nslot;
                if (use > 0 && !mbar_wait(&empty[slot], (uint32_t)((use - 1) & 1), a.wait, flags)) {
                    bad = true;
                    break;
                }
                if (flags[0]) break;
                const uint32_t bytes = (uint32_t)len * a.rec;
                mbar_arrive_expect_tx(&full[slot], bytes);
                bulk_g2s_hint(ring + (size_t)slot * a.slot_bytes, a.w + (rg * a.kc + c0) * a.rec, bytes, &full[slot],
                              l2_evict_first());  // the weights are read once per launch
                pos += len;
                ++u;
            }
            // No copy may still be landing in shared memory when the CTA exits.
            WaitCfg drain{int64_t(1) << 40, 1000000000ull};
            for (int64_t sl = 0; sl < min64(u, a.nslot); ++sl) {
                const int64_t last_use = (u - 1 - sl) / a.nslot;
                mbar_wait(&full[sl], (uint32_t)(last_use & 1), drain, nullptr);
            }
            if (bad) {
                raise_status(a.status, kStatusTimeout);
                flags[0] = 1;
            }
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------------- consumers
        bool bad = false;
        int64_t u = 0;
        {
            // activation rows staged by the producer in slots 0 .. nx-1
            const int nx = (a.m + 7) / 8;
            for (int i = 0; i < nx; ++i)
                if (!bad) bad = !__all_sync(0xffffffffu, mbar_wait(&full[i], 0u, a.wait, nullptr));
            build_act_frags<NW * kWarp>(reinterpret_cast<const uint16_t *>(ring), a.k, 8, a.slot_bytes / 2, a.m, a.k,
                                        a.kbp, NGRP, a.norm != 0, a.eps, frag, shift, inv, tid, warp, lane);
            __syncwarp();
            for (int i = 0; i < nx; ++i)
                if (lane == 0 && !bad) mbar_arrive(&empty[i]);
            u = nx;
        }
        const uint2 *frag2 = reinterpret_cast<const uint2 *>(frag);
        float acc[1][NGRP][4];
#pragma unroll
        for (int g = 0; g < NGRP; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[0][g][i] = 0.f;
        const int64_t rg_first = s / a.kc;
        for (int64_t pos = s; pos < e;) {
            const int64_t rg = pos / a.kc;
            const int c0 = (int)(pos - rg * a.kc);
            const int len = (int)min64(min64(e - pos, a.kc - c0), a.slot_recs);
            const int slot = (int)(u % a.nslot);
            const int64_t use = u / a.nslot;
            if (!bad) bad = !__all_sync(0xffffffffu, mbar_wait(&full[slot], (uint32_t)(use & 1), a.wait, nullptr));
            if (!bad) {
                const uint8_t *base = ring + (size_t)slot * a.slot_bytes;
                for (int i = warp; i < len; i += NW) {
                    const uint8_t *recs[1] = {base + (size_t)i * a.rec};
                    mma_records<FMT, NGRP, 1, false>(recs, frag2, nullptr, a.kbp, (c0 + i) * CB, lane, esc, acc);
                }
            }
            __syncwarp();
            if (lane == 0 && !bad) mbar_arrive(&empty[slot]);  // a slot whose data never came is kept
            pos += len;
            ++u;
            if (c0 + len < a.kc && pos < e) continue;  // row group continues in the next slot
            // ---- end of this CTA's part of row group rg: reduce over warps
            float *mine = scr + warp * TILE;
#pragma unroll
            for (int g = 0; g < NGRP; ++g)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    mine[(g * 4 + i) * kWarp + lane] = acc[0][g][i];
                    acc[0][g][i] = 0.f;
                }
            if (bar_or(1, NW * kWarp, bad)) {
                if (tid == 0) {
                    flags[0] = 1;
                    raise_status(a.status, kStatusTimeout);
                }
                break;
            }
            const bool partial = rg * a.kc < s || (rg + 1) * a.kc > e;
            float v = 0.f;
            int r = 0;
            int64_t nrow = 0;
            const bool have = tid < TILE;
            if (have) {
                for (int w = 0; w < NW; ++w) v += scr[w * TILE + tid];
                const int grp = tid >> 7, i = (tid >> 5) & 3, ln = tid & 31;
                nrow = rg * 16 + acc_wrow(ln, i);
                r = acc_xrow(ln, grp, i);
                if (r < a.m) v = mul_pow2(v, 24 - (MB - 1) - shift[r]);
            }
            auto store = [&](float val) {
                if (have && r < a.m && nrow < a.n) {
                    if (a.y) a.y[(int64_t)r * a.ldy + nrow] = val;
                    if (a.yb) a.yb[(int64_t)r * a.ldy + nrow] = f32_to_bf16_bits(val);
                }
            };
            if (!partial) {
                store(v);
                bar_sync(1, NW * kWarp);
            } else {
                const int slotp = 2 * c + (rg == rg_first ? 0 : 1);
                if (have) a.part[(size_t)slotp * TILE + tid] = v;
                bar_sync(1, NW * kWarp);
                const int cf = cta_of(rg * a.kc, R, a.ncta), cl = cta_of((rg + 1) * a.kc - 1, R, a.ncta);
                if (tid == 0) {
                    __threadfence();  // every thread's partial store, ordered by the barrier, before the count
                    const uint32_t old = atom_add_acq_rel(&a.cnt[rg], 1u);
                    flags[1] = (old == (uint32_t)(cl - cf)) ? 1 : 0;
                }
                bar_sync(1, NW * kWarp);
                if (flags[1]) {
                    float sum = 0.f;
                    if (have) {
                        for (int cc = cf; cc <= cl; ++cc) {
                            const int sp = 2 * cc + (rg == share_start(cc, R, a.ncta) / a.kc ? 0 : 1);
                            sum += __ldcg(&a.part[(size_t)sp * TILE + tid]);
                        }
                    }
                    store(sum);
                    if (tid == 0) atomicExch(&a.cnt[rg], 0u);
                }
                bar_sync(1, NW * kWarp);
            }
        }
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
    int ngrp, ncta, nslot, slot_recs, slot_bytes, frag_bytes;
    size_t smem;
    size_t ws_cnt_off, ws_part_off, ws_bytes;
};

static int plan_linear(const Geometry &g, int m, LinearPlan *p) {
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    p->ngrp = m > 8 ? 2 : 1;
    const int kbp = (int)(g.kc * g.cb);
    p->frag_bytes = p->ngrp * kbp * 32 * 8;
    const size_t fixed =
        align_up((size_t)p->frag_bytes + kConsumerWarps * p->ngrp * 128 * 4 + kLinMisc + 16 * 8, 128);
    const int64_t R = g.ng * g.kc;
    p->ncta = (int)std::min<int64_t>(di.sms, R);
    const int64_t per_cta = (R + p->ncta - 1) / p->ncta;
    int recs = (int)std::min<int64_t>(std::min<int64_t>(g.kc, std::max<int64_t>(1, 36864 / g.rec)), per_cta);
    if (recs < 1) recs = 1;
    const size_t xrows = (size_t)std::min(m, 8) * g.k * 2;  // staged activation rows per slot
    for (;;) {
        const size_t slot = align_up(std::max((size_t)recs * g.rec, xrows), 16);
        const size_t avail = di.smem_optin > (int)fixed ? di.smem_optin - fixed : 0;
        int nslot = (int)std::min<size_t>(8, avail / slot);
        if (nslot >= 2) {
            p->slot_recs = recs;
            p->slot_bytes = (int)slot;
            p->nslot = nslot;
            p->smem = fixed + (size_t)nslot * slot;
            break;
        }
        if (recs == 1) return fail(BFP_ESHAPE, "k too large for the activation fragments in shared memory");
        recs = std::max(1, recs / 2);
    }
    p->ws_cnt_off = 0;
    p->ws_part_off = align_up((size_t)g.ng * 4, 256);
    p->ws_bytes = p->ws_part_off + (size_t)2 * p->ncta * p->ngrp * 128 * 4;
    return BFP_OK;
}

template <int FMT, int NGRP>
static int launch_linear_t(const LinearArgs &a, const LinearPlan &p, cudaStream_t st) {
    auto kern = bfp_linear_kernel<FMT, NGRP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bfp_linear)");
    kern<<<p.ncta, kThreads, p.smem, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch bfp_linear");
    return BFP_OK;
}

// Shared by bfp_linear and the decode stack's LM head (norm = RMS-normalise x first).
// status: the workspace status word; body: the kernel's counters and partials.
int linear_launch_ex(const bfp_matrix *w, const uint16_t *x, int m, int64_t ldx, float *y, uint16_t *y_bf16,
                     int64_t ldy, uint32_t *status, void *body, size_t body_bytes, cudaStream_t st, int norm) {
    Geometry g;
    int rc = check_matrix(w, &g, true);
    if (rc) return rc;
    if (m < 1 || m > 16) return fail(BFP_ESHAPE, "m must be in [1, 16]");
    if (!x || (!y && !y_bf16)) return fail(BFP_EINVAL, "null x or no output");
    if (ldx < g.k || ldx % 8 != 0) return fail(BFP_EALIGN, "ldx must be >= k and a multiple of 8");
    if (ldy < g.n) return fail(BFP_EINVAL, "ldy < n");
    if (!aligned16(x) || (y && !aligned16(y)) || (y_bf16 && !aligned16(y_bf16)) || !aligned16(body))
        return fail(BFP_EALIGN, "device pointers must be 16-byte aligned");
    LinearPlan p;
    rc = plan_linear(g, m, &p);
    if (rc) return rc;
    if (!body || body_bytes < p.ws_bytes) return fail(BFP_EWORKSPACE, "workspace smaller than bfp_linear_workspace_size");
    LinearArgs a;
    a.w = static_cast<const uint8_t *>(w->data);
    a.n = g.n;
    a.ng = g.ng;
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
    uint8_t *wsb = static_cast<uint8_t *>(body);
    a.status = status;
    a.cnt = reinterpret_cast<uint32_t *>(wsb + p.ws_cnt_off);
    a.part = reinterpret_cast<float *>(wsb + p.ws_part_off);
    a.ncta = p.ncta;
    a.nslot = p.nslot;
    a.slot_recs = p.slot_recs;
    a.slot_bytes = p.slot_bytes;
    a.frag_bytes = p.frag_bytes;
    a.wait = WaitCfg{kDefaultWaitIters, kDefaultWaitNanos};  // only this CTA's own copies are waited on
    if (g.fmt == BFP_FMT_BFP4)
        return p.ngrp == 1 ? launch_linear_t<4, 1>(a, p, st) : launch_linear_t<4, 2>(a, p, st);
    return p.ngrp == 1 ? launch_linear_t<8, 1>(a, p, st) : launch_linear_t<8, 2>(a, p, st);
}

// Bytes of the kernel's counters and partials (the workspace after its header).
int linear_ws_body_bytes(const bfp_matrix *w, int m, size_t *bytes) {
    Geometry g;
    int rc = check_matrix(w, &g, false);
    if (rc) return rc;
    if (m < 1 || m > 16) return fail(BFP_ESHAPE, "m must be in [1, 16]");
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
                            reinterpret_cast<cudaStream_t>(stream), 0);
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
