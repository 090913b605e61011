// BFP KV cache: encode on append (bfp_kv_append) and decode attention over the
// cache for one query token (bfp_attn_decode).
//
// The qwen3.6-a3b-blackhole page (QWEN36_KV_DTYPE row) stores the attention KV
// cache as BFP8 (20.0 -> 10.6 KiB per token) and decode attention re-reads the
// whole cache every step; the Qwen3.8-27B s27v6 card ("Changes in s27",
// bfp8_v4r) keeps K in BFP8 and stores V Hadamard-rotated as BFP4. Here each
// token's K (and V) vector of one KV head is cut into 16-value blocks along the
// head dimension, each with one exponent byte; the rotation is the Sylvester
// Hadamard matrix H_d applied to V in fp32 by the fast transform before
// encoding, and undone once on the attention output (H_d H_d = d I).
//
// Attention: the context is split into chunks of kChunk tokens; CTA (s, h)
// takes KV head h and a contiguous range of chunks, streams each chunk's K and
// V fields into shared memory with bulk copies (two stages), and keeps a
// running softmax (max, sum, weighted V sum) for the G query heads of the
// group. A second launch merges the CTAs' partial results per query head and,
// for rotated V, applies H_d / d.
#include <cuda_runtime.h>

#include <algorithm>

#include "bfp_launch.h"

namespace bfp {

using namespace dev;

namespace {

constexpr int kChunk = 64;         // tokens per shared-memory stage
constexpr int kAttnThreads = 256;  // 8 warps
constexpr int kMaxGroup = 8;       // query heads per KV head

__host__ __device__ constexpr int row_code_bytes(int fmt, int d) { return fmt == BFP_FMT_BFP8 ? d : d / 2; }

// 2^e for e in [-149, 127], exact (subnormal below -126).
__device__ __forceinline__ float exact_pow2(int e) {
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << (e + 149));
}

// Round-to-nearest-even magnitude of fp32 bits u on a block with exponent field E (the plain BFP rule:
// significand shifted right by (24 - mb) + (E - e), saturated; exponent field 0 gives 0).
__device__ __forceinline__ uint32_t bfp_code(uint32_t u, int E, int mb) {
    const int e = (int)((u >> 23) & 0xFFu);
    uint32_t mag = 0;
    if (e != 0) {
        const uint64_t sig = (uint64_t)((u & 0x7FFFFFu) | 0x800000u);
        const int sh = (24 - mb) + (E - e);
        if (sh < 40) {
            const uint64_t bias = ((uint64_t)1 << (sh - 1)) - 1u + ((sig >> sh) & 1u);
            mag = (uint32_t)((sig + bias) >> sh);
        }
        const uint32_t top = (1u << mb) - 1u;
        if (mag > top) mag = top;
    }
    const uint32_t s = mag ? (u >> 31) : 0u;
    return (s << mb) | mag;
}

struct KvArgs {
    int kvh, d, k_fmt, v_fmt, rot;
    int64_t cap;
    uint8_t *kc, *ke, *vc, *ve;
};

// One warp per (token, KV head, K or V) row: load d bf16 values (VPL per lane, contiguous), rotate V
// if asked (fp32 fast Walsh-Hadamard transform, stages h = 1, 2, 4, ...), encode 16-value blocks.
template <int VPL>
__global__ void __launch_bounds__(128) kv_append_kernel(const KvArgs a, const uint16_t *k, const uint16_t *v,
                                                        int64_t pos, int n_new) {
    grid_dep_launch_dependents();
    grid_dep_wait();
    constexpr int D = VPL * kWarp;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int64_t nrows = (int64_t)n_new * a.kvh * 2;
    if (row >= nrows) return;
    const int which = (int)(row & 1);  // 0: K, 1: V
    const int64_t rest = row >> 1;
    const int64_t tok = rest / a.kvh;
    const int h = (int)(rest % a.kvh);
    const uint16_t *src = (which ? v : k) + (tok * a.kvh + h) * D + lane * VPL;
    float x[VPL];
#pragma unroll
    for (int t = 0; t < VPL; ++t) x[t] = __uint_as_float((uint32_t)src[t] << 16);
    if (which && a.rot) {
#pragma unroll
        for (int hh = 1; hh < VPL; hh <<= 1)
#pragma unroll
            for (int t = 0; t < VPL; ++t)
                if (!(t & hh)) {
                    const float p = x[t], q = x[t + hh];
                    x[t] = p + q;
                    x[t + hh] = p - q;
                }
#pragma unroll
        for (int lh = 1; lh < kWarp; lh <<= 1) {
            const bool upper = (lane & lh) != 0;
#pragma unroll
            for (int t = 0; t < VPL; ++t) {
                const float o = __shfl_xor_sync(0xffffffffu, x[t], lh);
                x[t] = upper ? o - x[t] : x[t] + o;
            }
        }
    }
    const int fmt = which ? a.v_fmt : a.k_fmt;
    const int mb = fmt == BFP_FMT_BFP8 ? 7 : 3;
    uint32_t u[VPL];
    int E = 0;
#pragma unroll
    for (int t = 0; t < VPL; ++t) {
        u[t] = __float_as_uint(x[t]);
        E = max(E, (int)((u[t] >> 23) & 0xFFu));
    }
    constexpr int L = 16 / VPL;  // lanes per block
#pragma unroll
    for (int o = 1; o < L; o <<= 1) E = max(E, __shfl_xor_sync(0xffffffffu, E, o));
    const int64_t slot = (int64_t)h * a.cap + pos + tok;
    uint8_t *codes = (which ? a.vc : a.kc) + slot * row_code_bytes(fmt, D);
    uint8_t *exps = (which ? a.ve : a.ke) + slot * (D / 16);
    if ((lane % L) == 0) exps[lane / L] = (uint8_t)E;
    if (fmt == BFP_FMT_BFP8) {
        uint8_t c[VPL];
#pragma unroll
        for (int t = 0; t < VPL; ++t) c[t] = (uint8_t)bfp_code(u[t], E, mb);
#pragma unroll
        for (int t = 0; t < VPL; ++t) codes[lane * VPL + t] = c[t];
    } else {
#pragma unroll
        for (int t = 0; t < VPL; t += 2)
            codes[(lane * VPL + t) / 2] = (uint8_t)(bfp_code(u[t], E, mb) | (bfp_code(u[t + 1], E, mb) << 4));
    }
}

struct AttnArgs {
    int kvh, G, S, nchunk;
    int64_t cap, n_ctx;
    float scale;
    const uint8_t *kc, *ke, *vc, *ve;
    const uint16_t *q;
    float *part;  // [kvh][S][G][D + 2]: o (D values), m, l
    uint32_t *status;
    WaitCfg wait;
};

// Decoded value of code c (sign << mb | magnitude) times 2^(E - 127 - (mb - 1)).
template <int MB>
__device__ __forceinline__ float code_value(uint32_t c, float scale) {
    const float m = (float)(c & ((1u << MB) - 1u));
    return ((c >> MB) & 1u) ? -m * scale : m * scale;
}

template <int VPL, int KF, int VF>
__global__ void __launch_bounds__(kAttnThreads) attn_partial_kernel(const AttnArgs a) {
    constexpr int D = VPL * kWarp;
    constexpr int KMB = KF == BFP_FMT_BFP8 ? 7 : 3, VMB = VF == BFP_FMT_BFP8 ? 7 : 3;
    constexpr int KROW = row_code_bytes(KF, D), VROW = row_code_bytes(VF, D), EROW = D / 16;
    constexpr int SK = kChunk * KROW, SKE = kChunk * EROW, SV = kChunk * VROW;
    constexpr int STAGE = SK + 2 * SKE + SV;
    constexpr int NTG = kAttnThreads / D;  // token groups of the V pass
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(16) float pw[kChunk][kMaxGroup];  // softmax weights of the chunk, [token][head]
    __shared__ float alpha_s[kMaxGroup], m_s[kMaxGroup], l_s[kMaxGroup];
    __shared__ uint64_t full[2];
    __shared__ int abort_s;
    __shared__ float red[NTG > 1 ? NTG - 1 : 1][kMaxGroup][NTG > 1 ? D : 1];  // token groups 1.. of the V pass
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y, s = blockIdx.x, G = a.G;
    const int c0 = (int)((int64_t)a.nchunk * s / a.S), c1 = (int)((int64_t)a.nchunk * (s + 1) / a.S);
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_fence_init();
        abort_s = 0;
    }
    if (tid < kMaxGroup) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.f;
    }
    grid_dep_launch_dependents();
    grid_dep_wait();
    __syncthreads();
    const uint8_t *kc = a.kc + (int64_t)h * a.cap * KROW, *ke = a.ke + (int64_t)h * a.cap * EROW;
    const uint8_t *vc = a.vc + (int64_t)h * a.cap * VROW, *ve = a.ve + (int64_t)h * a.cap * EROW;
    auto issue = [&](int ci) {  // thread 0: chunk ci into stage (ci - c0) & 1
        const int st = (ci - c0) & 1;
        uint8_t *dst = smem + st * STAGE;
        const int64_t t0 = (int64_t)ci * kChunk;
        mbar_arrive_expect_tx(&full[st], STAGE);
        bulk_g2s(dst, kc + t0 * KROW, SK, &full[st]);
        bulk_g2s(dst + SK, ke + t0 * EROW, SKE, &full[st]);
        bulk_g2s(dst + SK + SKE, vc + t0 * VROW, SV, &full[st]);
        bulk_g2s(dst + SK + SKE + SV, ve + t0 * EROW, SKE, &full[st]);
    };
    if (tid == 0) {
        if (c0 < c1) issue(c0);
        if (c0 + 1 < c1) issue(c0 + 1);
    }
    // this lane's slice of the G query vectors (scores pass: lanes split the head dimension)
    float qr[kMaxGroup][VPL];
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g)
#pragma unroll
        for (int t = 0; t < VPL; ++t)
            qr[g][t] = g < G ? __uint_as_float((uint32_t)a.q[((int64_t)h * G + g) * D + lane * VPL + t] << 16) : 0.f;
    const int col = tid % D, tg = tid / D;
    float acc[kMaxGroup];
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) acc[g] = 0.f;

    for (int ci = c0; ci < c1; ++ci) {
        const int st = (ci - c0) & 1;
        const uint32_t par = (uint32_t)(((ci - c0) >> 1) & 1);
        if (tid == 0 && !mbar_wait(&full[st], par, a.wait, nullptr)) {
            abort_s = 1;
            raise_status(a.status, kStatusTimeout);
            // chunks ci and ci + 1 are the copies in flight: give them a bounded time to land before
            // the CTA leaves
            mbar_wait(&full[st], par, a.wait, nullptr);
            if (ci + 1 < c1) mbar_wait(&full[st ^ 1], (uint32_t)(((ci + 1 - c0) >> 1) & 1), a.wait, nullptr);
        }
        __syncthreads();
        if (abort_s) return;
        const uint8_t *sk = smem + st * STAGE, *ske = sk + SK, *sv = ske + SKE, *sve = sv + SV;
        const int64_t tb = (int64_t)ci * kChunk;
        const int nv = (int)min64((int64_t)kChunk, a.n_ctx - tb);
        // ---- scores: warp w takes tokens w, w + 8, ...; the G dot products are reduced together
        for (int i = warp; i < kChunk; i += kAttnThreads / kWarp) {
            float dot[kMaxGroup];
            if (i < nv) {
                const float bs = exact_pow2((int)ske[i * EROW + lane * VPL / 16] - 127 - (KMB - 1));
                float kv[VPL];
                if (KF == BFP_FMT_BFP8) {
#pragma unroll
                    for (int t = 0; t < VPL; ++t) kv[t] = code_value<KMB>(sk[i * KROW + lane * VPL + t], bs);
                } else {
#pragma unroll
                    for (int t = 0; t < VPL; t += 2) {
                        const uint32_t b = sk[i * KROW + (lane * VPL + t) / 2];
                        kv[t] = code_value<KMB>(b & 15u, bs);
                        kv[t + 1] = code_value<KMB>(b >> 4, bs);
                    }
                }
#pragma unroll
                for (int g = 0; g < kMaxGroup; ++g) {
                    float sacc = 0.f;
#pragma unroll
                    for (int t = 0; t < VPL; ++t) sacc = fmaf(kv[t], qr[g][t], sacc);
                    dot[g] = sacc;
                }
            } else {
#pragma unroll
                for (int g = 0; g < kMaxGroup; ++g) dot[g] = 0.f;
            }
            // 8 values over 32 lanes: halve the set at each of the first three steps
            float r4[4], r2[2];
            const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float send = b4 ? dot[j] : dot[j + 4], keep = b4 ? dot[j + 4] : dot[j];
                r4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float send = b3 ? r4[j] : r4[j + 2], keep = b3 ? r4[j + 2] : r4[j];
                r2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
            float r1;
            {
                const float send = b2 ? r2[0] : r2[1], keep = b2 ? r2[1] : r2[0];
                r1 = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
            r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
            r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
            if ((lane & 3) == 0) pw[i][lane >> 2] = i < nv ? r1 * a.scale : -INFINITY;
        }
        __syncthreads();
        // ---- running softmax: warp g updates head g over the chunk's scores
        if (warp < G) {
            const int g = warp;
            float mx = -INFINITY;
            for (int i = lane; i < kChunk; i += kWarp) mx = fmaxf(mx, pw[i][g]);
            mx = warp_max(mx);
            const float m_old = m_s[g], m_new = fmaxf(m_old, mx);
            float sum = 0.f;
            for (int i = lane; i < kChunk; i += kWarp) {
                const float p = i < nv ? __expf(pw[i][g] - m_new) : 0.f;
                pw[i][g] = p;
                sum += p;
            }
            sum = warp_sum(sum);
            if (lane == 0) {
                const float al = __expf(m_old - m_new);  // 0 on the first chunk (m_old = -inf)
                alpha_s[g] = al;
                l_s[g] = l_s[g] * al + sum;
                m_s[g] = m_new;
            }
        }
        __syncthreads();
        // ---- weighted V sum: thread (col, tg) takes column col of tokens tg, tg + NTG, ...
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) acc[g] *= g < G ? alpha_s[g] : 0.f;
        for (int i = tg; i < nv; i += NTG) {
            const float bs = exact_pow2((int)sve[i * EROW + col / 16] - 127 - (VMB - 1));
            float val;
            if (VF == BFP_FMT_BFP8) {
                val = code_value<VMB>(sv[i * VROW + col], bs);
            } else {
                const uint32_t b = sv[i * VROW + col / 2];
                val = code_value<VMB>((col & 1) ? (b >> 4) : (b & 15u), bs);
            }
            const float4 p0 = *reinterpret_cast<const float4 *>(&pw[i][0]);
            const float4 p1 = *reinterpret_cast<const float4 *>(&pw[i][4]);
            acc[0] = fmaf(p0.x, val, acc[0]);
            acc[1] = fmaf(p0.y, val, acc[1]);
            acc[2] = fmaf(p0.z, val, acc[2]);
            acc[3] = fmaf(p0.w, val, acc[3]);
            acc[4] = fmaf(p1.x, val, acc[4]);
            acc[5] = fmaf(p1.y, val, acc[5]);
            acc[6] = fmaf(p1.z, val, acc[6]);
            acc[7] = fmaf(p1.w, val, acc[7]);
        }
        __syncthreads();  // the stage is free again
        if (tid == 0 && ci + 2 < c1) {
            fence_proxy_async_shared();
            issue(ci + 2);
        }
    }
    // ---- partial results: o for each head (token groups added in order), then m and l
    if constexpr (NTG > 1) {
        if (tg > 0)
#pragma unroll
            for (int g = 0; g < kMaxGroup; ++g) red[tg - 1][g][col] = acc[g];
        __syncthreads();
        if (tg == 0)
            for (int j = 1; j < NTG; ++j)
#pragma unroll
                for (int g = 0; g < kMaxGroup; ++g) acc[g] += red[j - 1][g][col];
    }
    float *base = a.part + (((int64_t)h * a.S + s) * G) * (D + 2);
    if (tg == 0)
        for (int g = 0; g < G; ++g) base[(int64_t)g * (D + 2) + col] = acc[g];
    if (tid < G) {
        base[(int64_t)tid * (D + 2) + D] = m_s[tid];
        base[(int64_t)tid * (D + 2) + D + 1] = l_s[tid];
    }
}

// One CTA per query head: merge the S partial results; rotate back (H_d / d) when V is stored rotated.
template <int D>
__global__ void __launch_bounds__(D) attn_merge_kernel(const float *part, int kvh, int G, int S, int rot, float *out) {
    __shared__ float x[D];
    grid_dep_wait();
    const int j = blockIdx.x, h = j / G, g = j % G, col = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, part[(((int64_t)h * S + s) * G + g) * (D + 2) + D]);
    float L = 0.f, o = 0.f;
    for (int s = 0; s < S; ++s) {
        const float *p = part + (((int64_t)h * S + s) * G + g) * (D + 2);
        const float w = p[D] == -INFINITY ? 0.f : __expf(p[D] - M);  // a split with no tokens has m = -inf
        L = fmaf(p[D + 1], w, L);
        o = fmaf(p[col], w, o);
    }
    float y = o / L;
    if (rot) {
        x[col] = y;
        __syncthreads();
        for (int hh = 1; hh < D; hh <<= 1) {
            const float a = x[col & ~hh], b = x[col | hh];
            __syncthreads();
            x[col] = (col & hh) ? a - b : a + b;
            __syncthreads();
        }
        y = x[col] * (1.0f / D);
    }
    out[(int64_t)j * D + col] = y;
}

int check_cache(const bfp_kv_cache *c) {
    if (!c) return fail(BFP_EINVAL, "null cache");
    if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256)
        return fail(BFP_ESHAPE, "head_dim must be 64, 128 or 256");
    if (c->kv_heads < 1 || c->kv_heads > 64) return fail(BFP_ESHAPE, "kv_heads must be in 1..64");
    for (int f : {c->k_fmt, c->v_fmt})
        if (f != BFP_FMT_BFP4 && f != BFP_FMT_BFP8) return fail(BFP_EINVAL, "k_fmt and v_fmt must be BFP4 or BFP8");
    if (c->v_rotated != 0 && c->v_rotated != 1) return fail(BFP_EINVAL, "v_rotated must be 0 or 1");
    if (c->reserved != 0) return fail(BFP_EINVAL, "reserved must be 0");
    if (c->capacity < kChunk || c->capacity % kChunk != 0 || c->capacity > (int64_t(1) << 31))
        return fail(BFP_ESHAPE, "capacity must be a positive multiple of 64 tokens, at most 2^31");
    if (!c->k_codes || !c->k_exps || !c->v_codes || !c->v_exps) return fail(BFP_EINVAL, "null cache array");
    if (!aligned16(c->k_codes) || !aligned16(c->k_exps) || !aligned16(c->v_codes) || !aligned16(c->v_exps))
        return fail(BFP_EALIGN, "cache arrays must be 16-byte aligned");
    return BFP_OK;
}

int attn_split(const bfp_kv_cache *c, int64_t n_ctx, int *S) {
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    const int64_t nchunk = (n_ctx + kChunk - 1) / kChunk;
    // about two CTAs per SM over all KV heads, at least two chunks per CTA
    int64_t s = std::max<int64_t>(1, (int64_t)2 * di.sms / c->kv_heads);
    s = std::min<int64_t>(s, std::max<int64_t>(1, nchunk / 2));
    *S = (int)s;
    return BFP_OK;
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int VPL, int KF, int VF>
int launch_partial(const AttnArgs &a, cudaStream_t st) {
    constexpr int D = VPL * kWarp;
    constexpr int STAGE = kChunk * (row_code_bytes(KF, D) + row_code_bytes(VF, D) + 2 * (D / 16));
    auto kern = attn_partial_kernel<VPL, KF, VF>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * STAGE);
    if (e != cudaSuccess) return cuda_fail(e, "attention shared memory");
    e = launch_pdl(kern, dim3(a.S, a.kvh), dim3(kAttnThreads), (size_t)2 * STAGE, st, a);
    if (e != cudaSuccess) return cuda_fail(e, "launch attention");
    return BFP_OK;
}

template <int VPL>
int launch_partial_d(const AttnArgs &a, int kf, int vf, cudaStream_t st) {
    if (kf == BFP_FMT_BFP8 && vf == BFP_FMT_BFP8) return launch_partial<VPL, BFP_FMT_BFP8, BFP_FMT_BFP8>(a, st);
    if (kf == BFP_FMT_BFP8 && vf == BFP_FMT_BFP4) return launch_partial<VPL, BFP_FMT_BFP8, BFP_FMT_BFP4>(a, st);
    if (kf == BFP_FMT_BFP4 && vf == BFP_FMT_BFP8) return launch_partial<VPL, BFP_FMT_BFP4, BFP_FMT_BFP8>(a, st);
    return launch_partial<VPL, BFP_FMT_BFP4, BFP_FMT_BFP4>(a, st);
}

}  // namespace

}  // namespace bfp

using namespace bfp;

extern "C" {

int bfp_kv_cache_size(int fmt, int kv_heads, int head_dim, int64_t capacity, size_t *code_bytes, size_t *exp_bytes) {
    if (!code_bytes || !exp_bytes) return fail(BFP_EINVAL, "null output");
    if (fmt != BFP_FMT_BFP4 && fmt != BFP_FMT_BFP8) return fail(BFP_EINVAL, "fmt must be BFP4 or BFP8");
    if ((head_dim != 64 && head_dim != 128 && head_dim != 256) || kv_heads < 1 || kv_heads > 64 ||
        capacity < kChunk || capacity % kChunk != 0 || capacity > (int64_t(1) << 31))
        return fail(BFP_ESHAPE, "head_dim 64/128/256, kv_heads 1..64, capacity a positive multiple of 64");
    *code_bytes = (size_t)kv_heads * capacity * row_code_bytes(fmt, head_dim);
    *exp_bytes = (size_t)kv_heads * capacity * (head_dim / 16);
    return BFP_OK;
}

int bfp_kv_append(const bfp_kv_cache *cache, const uint16_t *k, const uint16_t *v, int64_t pos, int n_new,
                  bfp_stream_t stream) {
    int rc = check_cache(cache);
    if (rc) return rc;
    if (!k || !v) return fail(BFP_EINVAL, "null k or v");
    if (n_new < 1 || pos < 0 || pos + n_new > cache->capacity) return fail(BFP_ESHAPE, "tokens outside the capacity");
    if (((uintptr_t)k & 15u) || ((uintptr_t)v & 15u)) return fail(BFP_EALIGN, "k and v must be 16-byte aligned");
    KvArgs a{cache->kv_heads, cache->head_dim, cache->k_fmt, cache->v_fmt, cache->v_rotated, cache->capacity,
             static_cast<uint8_t *>(cache->k_codes), static_cast<uint8_t *>(cache->k_exps),
             static_cast<uint8_t *>(cache->v_codes), static_cast<uint8_t *>(cache->v_exps)};
    const int64_t rows = (int64_t)n_new * cache->kv_heads * 2;
    const dim3 grid((unsigned)((rows + 3) / 4));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (cache->head_dim) {
        case 64: e = launch_pdl(kv_append_kernel<2>, grid, dim3(128), 0, st, a, k, v, pos, n_new); break;
        case 128: e = launch_pdl(kv_append_kernel<4>, grid, dim3(128), 0, st, a, k, v, pos, n_new); break;
        default: e = launch_pdl(kv_append_kernel<8>, grid, dim3(128), 0, st, a, k, v, pos, n_new); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "launch kv append");
    return BFP_OK;
}

int bfp_attn_workspace_size(const bfp_kv_cache *cache, int q_heads, int64_t n_ctx, size_t *bytes) {
    if (!bytes) return fail(BFP_EINVAL, "null bytes");
    int rc = check_cache(cache);
    if (rc) return rc;
    if (q_heads < cache->kv_heads || q_heads % cache->kv_heads || q_heads / cache->kv_heads > kMaxGroup)
        return fail(BFP_ESHAPE, "q_heads must be kv_heads times 1..8");
    if (n_ctx < 1 || n_ctx > cache->capacity) return fail(BFP_ESHAPE, "n_ctx must be in 1..capacity");
    int S = 0;
    rc = attn_split(cache, n_ctx, &S);
    if (rc) return rc;
    *bytes = kWsHeader + (size_t)cache->kv_heads * S * (q_heads / cache->kv_heads) * (cache->head_dim + 2) * 4;
    return BFP_OK;
}

int bfp_attn_decode(const bfp_kv_cache *cache, const uint16_t *q, int q_heads, int64_t n_ctx, float scale, float *out,
                    void *ws, size_t ws_bytes, bfp_stream_t stream) {
    size_t need = 0;
    int rc = bfp_attn_workspace_size(cache, q_heads, n_ctx, &need);
    if (rc) return rc;
    if (!q || !out) return fail(BFP_EINVAL, "null q or out");
    if (!ws || ws_bytes < need) return fail(BFP_EWORKSPACE, "workspace smaller than bfp_attn_workspace_size");
    if (!aligned16(q) || !aligned16(out) || !aligned16(ws)) return fail(BFP_EALIGN, "pointers must be 16-byte aligned");
    int S = 0;
    rc = attn_split(cache, n_ctx, &S);
    if (rc) return rc;
    AttnArgs a;
    a.kvh = cache->kv_heads;
    a.G = q_heads / cache->kv_heads;
    a.S = S;
    a.nchunk = (int)((n_ctx + kChunk - 1) / kChunk);
    a.cap = cache->capacity;
    a.n_ctx = n_ctx;
    a.scale = scale;
    a.kc = static_cast<const uint8_t *>(cache->k_codes);
    a.ke = static_cast<const uint8_t *>(cache->k_exps);
    a.vc = static_cast<const uint8_t *>(cache->v_codes);
    a.ve = static_cast<const uint8_t *>(cache->v_exps);
    a.q = q;
    a.status = static_cast<uint32_t *>(ws);
    a.part = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kWsHeader);
    a.wait = wait_cfg();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (cache->head_dim) {
        case 64: rc = launch_partial_d<2>(a, cache->k_fmt, cache->v_fmt, st); break;
        case 128: rc = launch_partial_d<4>(a, cache->k_fmt, cache->v_fmt, st); break;
        default: rc = launch_partial_d<8>(a, cache->k_fmt, cache->v_fmt, st); break;
    }
    if (rc) return rc;
    cudaError_t e;
    const float *part = a.part;
    switch (cache->head_dim) {
        case 64: e = launch_pdl(attn_merge_kernel<64>, dim3(q_heads), dim3(64), 0, st, part, a.kvh, a.G, S, cache->v_rotated, out); break;
        case 128: e = launch_pdl(attn_merge_kernel<128>, dim3(q_heads), dim3(128), 0, st, part, a.kvh, a.G, S, cache->v_rotated, out); break;
        default: e = launch_pdl(attn_merge_kernel<256>, dim3(q_heads), dim3(256), 0, st, part, a.kvh, a.G, S, cache->v_rotated, out); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "launch attention merge");
    return BFP_OK;
}

}  // extern "C"
