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
// The codes are stored in tiles of 16 tokens x 16 values laid out in the
// operand order of mma.sync m16n8k16, so that each lane's fragment is one 32-
// or 64-bit shared-memory load and each appended token writes only its own
// words, halves or bytes (layout in include/bfpmoe.h).
//
// Attention: the context is split into chunks of kChunk tokens; CTA (s, h)
// takes KV head h and a contiguous range of chunks, streams each chunk's K and
// V tiles and exponents into shared memory with bulk copies (two stages), and
// keeps a running softmax (max, sum, weighted V sum) for the G query heads of
// the group, with both contractions on the tensor cores. A second launch
// merges the CTAs' partial results per query head and, for rotated V, applies
// H_d / d.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <vector>

#include "bfp_launch.h"
#include "bfp_pack.h"

namespace bfp {

using namespace dev;

namespace {

constexpr int kChunk = 64;         // tokens per shared-memory stage
constexpr int kAttnThreads = 256;  // 8 warps
constexpr int kMaxGroup = 8;       // query heads per KV head

__host__ __device__ constexpr int code_bytes_per_token(int fmt, int d) { return fmt == BFP_FMT_BFP8 ? d : d / 2; }

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

// fp16 bit pattern whose value is code's magnitude times 2^-24 with its sign (a subnormal: exact).
__device__ __forceinline__ uint32_t code_pattern(uint32_t code, int mb) {
    return (code & ((1u << mb) - 1u)) | (((code >> mb) & 1u) << 15);
}

// Byte offset, inside a 16-token x 16-column tile, of token row r's codes (see include/bfpmoe.h).
__device__ __forceinline__ int k8_word_off(int r, int j) { return (4 * (r & 7) + j) * 8 + (r >> 3) * 4; }
__device__ __forceinline__ int k4_half_off(int r, int j) { return (4 * (r & 7) + j) * 4 + (r >> 3) * 2; }
__device__ __forceinline__ int v8_byte_off(int r, int c) { return (4 * (c & 7) + (r >> 2)) * 8 + (c >> 3) * 4 + (r & 3); }
__device__ __forceinline__ int v4_byte_off(int r, int c) { return (4 * (c & 7) + (r >> 2)) * 4 + (r & 3); }

// One warp per (token, KV head, K or V) row: load d bf16 values (VPL per lane, contiguous), rotate V
// if asked (fp32 fast Walsh-Hadamard transform, stages h = 1, 2, 4, ...), encode 16-value blocks and
// store them in the tile order of the cache.
template <int VPL>
__global__ void __launch_bounds__(128) kv_append_kernel(const KvArgs a, const uint16_t *k, const uint16_t *v,
                                                        int64_t pos, int n_new) {
    grid_dep_launch_dependents();
    grid_dep_wait();
    constexpr int D = VPL * kWarp, NB = D / 16;
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
    uint32_t c[VPL];
#pragma unroll
    for (int t = 0; t < VPL; ++t) c[t] = bfp_code(u[t], E, mb);
    const int64_t slot = pos + tok;            // token slot
    const int r = (int)(slot & 15);            // row in its 16-token tile group
    const int b = lane / L;                    // block of this lane's columns
    const int cb0 = (lane % L) * VPL;          // first column within the block
    const int tb = fmt == BFP_FMT_BFP8 ? 256 : 128;
    uint8_t *tile = (which ? a.vc : a.kc) + (((int64_t)h * (a.cap / 16) + (slot >> 4)) * NB + b) * tb;
    uint8_t *exps = (which ? a.ve : a.ke) + ((int64_t)h * a.cap + slot) * NB;
    if ((lane % L) == 0) exps[b] = (uint8_t)E;
    if (!which) {
        // K: a row's codes of columns 4j..4j+3 are one 32-bit word (BFP8) or one 16-bit half (BFP4)
        if (fmt == BFP_FMT_BFP8) {
            uint32_t cc[VPL < 4 ? 4 : VPL];
#pragma unroll
            for (int t = 0; t < VPL; ++t) cc[t] = c[t];
            if (VPL == 2) {  // two lanes hold the four codes of a word
                cc[2] = __shfl_down_sync(0xffffffffu, c[0], 1);
                cc[3] = __shfl_down_sync(0xffffffffu, c[VPL - 1], 1);
            }
            if (VPL >= 4 || (lane & 1) == 0) {
#pragma unroll
                for (int j = 0; j < (VPL < 4 ? 1 : VPL / 4); ++j) {
                    const uint32_t p01 = code_pattern(cc[4 * j], 7) | (code_pattern(cc[4 * j + 1], 7) << 16);
                    const uint32_t p23 = code_pattern(cc[4 * j + 2], 7) | (code_pattern(cc[4 * j + 3], 7) << 16);
                    *reinterpret_cast<uint32_t *>(tile + k8_word_off(r, (cb0 >> 2) + j)) = p01 | __funnelshift_l(p23, p23, 8);
                }
            }
        } else {
            if (VPL >= 4) {
#pragma unroll
                for (int j = 0; j < VPL / 4; ++j)
                    *reinterpret_cast<uint16_t *>(tile + k4_half_off(r, (cb0 >> 2) + j)) =
                        (uint16_t)(c[4 * j] | (c[4 * j + 1] << 4) | (c[4 * j + 2] << 8) | (c[4 * j + 3] << 12));
            } else {  // two codes: one byte of the half
                tile[k4_half_off(r, cb0 >> 2) + ((cb0 & 3) >> 1)] = (uint8_t)(c[0] | (c[VPL - 1] << 4));
            }
        }
    } else {
        // V: a token's code of column c sits in its own byte (BFP8), or shares a byte with column c + 8 (BFP4)
        if (fmt == BFP_FMT_BFP8) {
#pragma unroll
            for (int t = 0; t < VPL; ++t) tile[v8_byte_off(r, cb0 + t)] = (uint8_t)c[t];
        } else {
            uint32_t hi[VPL];
#pragma unroll
            for (int t = 0; t < VPL; ++t) hi[t] = __shfl_xor_sync(0xffffffffu, c[t], L / 2);
            if (cb0 < 8)
#pragma unroll
                for (int t = 0; t < VPL; ++t) tile[v4_byte_off(r, cb0 + t)] = (uint8_t)(c[t] | (hi[t] << 4));
        }
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

// Two 4-bit codes (low byte of x: first code in the low nibble) -> fp16x2 subnormal patterns.
__device__ __forceinline__ uint32_t nib2_pattern(uint32_t x) {
    const uint32_t s = (x & 0xFu) | ((x & 0xF0u) << 12);
    return (s & 0x00070007u) | ((s & 0x00080008u) << 12);
}
// Two 8-bit codes (bytes 0 and 2 of s, other bytes zero) -> fp16x2 subnormal patterns.
__device__ __forceinline__ uint32_t byte2_pattern(uint32_t s) { return (s & 0x007F007Fu) | ((s & 0x00800080u) << 8); }

// Decode attention, first launch. Per 64-token chunk, with NB = D / 16 blocks per row:
//   scores: S^T (tokens x heads) = K_tile (16 tokens x 16 dims, BFP codes as fp16 subnormals) x q (16 dims
//     x 8 heads, fp16 scaled by 2^sq) on mma.sync m16n8k16, zero C, folded into fp32 with each token
//     row's block scale; warp w takes token slice w / 2 and half the blocks;
//   softmax: warp g keeps head g's running max m, sum l, and writes the chunk's weights p;
//   values: O (heads x dims) += P' (8 heads x 16 tokens) x V_tile (16 tokens x 8 dims), where P' carries
//     each token's block scale relative to the slice's largest (p 2^(E_t - E_ref) <= 1, as fp16 hi + lo),
//     folded with 2^E_ref; warp w takes blocks w, w + 8, ...
// The contraction index is permuted the same way in both operands: fragment slots (2t, 2t+1, 2t+8,
// 2t+9) of lane (g, t) carry dims (tokens) 4t .. 4t+3, which is how the tiles are stored.
template <int VPL, int KF, int VF>
__global__ void __launch_bounds__(kAttnThreads) attn_partial_kernel(const AttnArgs a) {
    constexpr int D = VPL * kWarp, NB = D / 16;
    constexpr int KMB = KF == BFP_FMT_BFP8 ? 7 : 3, VMB = VF == BFP_FMT_BFP8 ? 7 : 3;
    constexpr int TBK = KF == BFP_FMT_BFP8 ? 256 : 128, TBV = VF == BFP_FMT_BFP8 ? 256 : 128;
    constexpr int SK = kChunk / 16 * NB * TBK, SKE = kChunk * NB, SV = kChunk / 16 * NB * TBV;
    constexpr int STAGE = SK + 2 * SKE + SV;
    constexpr int NBA = NB / 2;            // blocks per warp in the scores pass
    constexpr int NBC = (NB + 7) / 8;      // blocks per warp in the values pass
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float pw[kChunk][kMaxGroup];        // the chunk's softmax weights, [token][head]
    __shared__ float spart[2][kChunk][kMaxGroup];  // scores, one part per half of the blocks
    __shared__ float alpha_s[kMaxGroup], m_s[kMaxGroup], l_s[kMaxGroup], qmax_s[kAttnThreads / kWarp];
    __shared__ uint64_t full[2];
    __shared__ int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g4 = lane >> 2, t4 = lane & 3;
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
    const uint8_t *kc = a.kc + (int64_t)h * a.cap * (NB * TBK / 16), *ke = a.ke + (int64_t)h * a.cap * NB;
    const uint8_t *vc = a.vc + (int64_t)h * a.cap * (NB * TBV / 16), *ve = a.ve + (int64_t)h * a.cap * NB;
    auto issue = [&](int ci) {  // thread 0: chunk ci into stage (ci - c0) & 1
        const int st = (ci - c0) & 1;
        uint8_t *dst = smem + st * STAGE;
        const int64_t t0 = (int64_t)ci * kChunk;
        mbar_arrive_expect_tx(&full[st], STAGE);
        bulk_g2s(dst, kc + t0 * (NB * TBK / 16), SK, &full[st]);
        bulk_g2s(dst + SK, ke + t0 * NB, SKE, &full[st]);
        bulk_g2s(dst + SK + SKE, vc + t0 * (NB * TBV / 16), SV, &full[st]);
        bulk_g2s(dst + SK + SKE + SV, ve + t0 * NB, SKE, &full[st]);
    };
    if (tid == 0) {
        if (c0 < c1) issue(c0);
        if (c0 + 1 < c1) issue(c0 + 1);
    }
    // q of the group in fp16, scaled by 2^sq so that max |q| lies in [2^14, 2^15)
    const uint16_t *qg = a.q + (int64_t)h * G * D;
    float qm = 0.f;
    for (int i = tid; i < G * D; i += kAttnThreads) qm = fmaxf(qm, fabsf(__uint_as_float((uint32_t)qg[i] << 16)));
    qm = warp_max(qm);
    if (lane == 0) qmax_s[warp] = qm;
    __syncthreads();
    for (int w = 0; w < kAttnThreads / kWarp; ++w) qm = fmaxf(qm, qmax_s[w]);
    const int sq = frag_shift(qm);
    const float sfac = mul_pow2(a.scale, 24 - sq);  // scores = folded MMA sums * 2^24 * 2^-sq * scale
    const int sl_a = warp >> 1, half = warp & 1;
    uint32_t bq[NBA][2];
#pragma unroll
    for (int bi = 0; bi < NBA; ++bi) {
        const int d0 = (half * NBA + bi) * 16 + 4 * t4;
        float qv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            qv[j] = g4 < G ? mul_pow2(__uint_as_float((uint32_t)qg[g4 * D + d0 + j] << 16), sq) : 0.f;
        bq[bi][0] = pack_half2(qv[0], qv[1]);
        bq[bi][1] = pack_half2(qv[2], qv[3]);
    }
    float acc[NBC][2][2];
#pragma unroll
    for (int bi = 0; bi < NBC; ++bi)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) acc[bi][hh][0] = acc[bi][hh][1] = 0.f;

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
        const int nv = (int)min64((int64_t)kChunk, a.n_ctx - (int64_t)ci * kChunk);
        // ---- scores
        {
            float cs[4] = {0.f, 0.f, 0.f, 0.f};
            const int ra = 16 * sl_a + g4;  // token rows ra and ra + 8 of the chunk
#pragma unroll
            for (int bi = 0; bi < NBA; ++bi) {
                const int b = half * NBA + bi;
                uint32_t A[4];
                if (KF == BFP_FMT_BFP8) {
                    const uint2 w = *reinterpret_cast<const uint2 *>(sk + (sl_a * NB + b) * TBK + lane * 8);
                    A[0] = w.x & kMaskBfp8;
                    A[2] = rotr(w.x, 8) & kMaskBfp8;
                    A[1] = w.y & kMaskBfp8;
                    A[3] = rotr(w.y, 8) & kMaskBfp8;
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(sk + (sl_a * NB + b) * TBK + lane * 4);
                    A[0] = nib2_pattern(w & 0xFFu);
                    A[2] = nib2_pattern((w >> 8) & 0xFFu);
                    A[1] = nib2_pattern((w >> 16) & 0xFFu);
                    A[3] = nib2_pattern(w >> 24);
                }
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(c, A, bq[bi][0], bq[bi][1]);
                const float e0 = exact_pow2((int)ske[ra * NB + b] - 127 - (KMB - 1));
                const float e1 = exact_pow2((int)ske[(ra + 8) * NB + b] - 127 - (KMB - 1));
                cs[0] = fmaf(c[0], e0, cs[0]);
                cs[1] = fmaf(c[1], e0, cs[1]);
                cs[2] = fmaf(c[2], e1, cs[2]);
                cs[3] = fmaf(c[3], e1, cs[3]);
            }
            spart[half][ra][2 * t4] = cs[0];
            spart[half][ra][2 * t4 + 1] = cs[1];
            spart[half][ra + 8][2 * t4] = cs[2];
            spart[half][ra + 8][2 * t4 + 1] = cs[3];
        }
        __syncthreads();
        // ---- running softmax: warp g updates head g over the chunk's scores
        if (warp < G) {
            const int g = warp;
            float sc[kChunk / kWarp];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < kChunk / kWarp; ++j) {
                const int i = lane + j * kWarp;
                sc[j] = i < nv ? (spart[0][i][g] + spart[1][i][g]) * sfac : -INFINITY;
                mx = fmaxf(mx, sc[j]);
            }
            mx = warp_max(mx);
            const float m_old = m_s[g], m_new = fmaxf(m_old, mx);
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < kChunk / kWarp; ++j) {
                const int i = lane + j * kWarp;
                const float p = i < nv ? __expf(sc[j] - m_new) : 0.f;
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
        // ---- weighted V sum
        if (warp < NB) {
            const float al = g4 < G ? alpha_s[g4] : 0.f;
#pragma unroll
            for (int bi = 0; bi < NBC; ++bi)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    acc[bi][hh][0] *= al;
                    acc[bi][hh][1] *= al;
                }
#pragma unroll
            for (int bi = 0; bi < NBC; ++bi) {
                const int b = warp + 8 * bi;
                if (b >= NB) break;
#pragma unroll
                for (int sl = 0; sl < kChunk / 16; ++sl) {
                    if (16 * sl >= nv) break;  // the rest of the chunk is past the context
                    const int tk = 16 * sl + 4 * t4;
                    int Ek[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) Ek[j] = tk + j < nv ? (int)sve[(tk + j) * NB + b] : 0;  // slots past the context hold anything
                    int Er = max(max(Ek[0], Ek[1]), max(Ek[2], Ek[3]));
                    Er = max(Er, __shfl_xor_sync(0xffffffffu, Er, 1));
                    Er = max(Er, __shfl_xor_sync(0xffffffffu, Er, 2));
                    float p[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        p[j] = g4 < G ? pw[tk + j][g4] * exact_pow2(max(Ek[j] - Er, -149)) : 0.f;
                    const __half2 h01 = __floats2half2_rn(p[0], p[1]), h23 = __floats2half2_rn(p[2], p[3]);
                    const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                    const __half2 l01 = __floats2half2_rn(p[0] - f01.x, p[1] - f01.y);
                    const __half2 l23 = __floats2half2_rn(p[2] - f23.x, p[3] - f23.y);
                    const uint32_t Ahi[4] = {*reinterpret_cast<const uint32_t *>(&h01), 0u,
                                             *reinterpret_cast<const uint32_t *>(&h23), 0u};
                    const uint32_t Alo[4] = {*reinterpret_cast<const uint32_t *>(&l01), 0u,
                                             *reinterpret_cast<const uint32_t *>(&l23), 0u};
                    uint32_t Bv[2][2];
                    if (VF == BFP_FMT_BFP8) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(sv + (sl * NB + b) * TBV + lane * 8);
                        Bv[0][0] = byte2_pattern(__byte_perm(w.x, 0u, 0x4140));
                        Bv[0][1] = byte2_pattern(__byte_perm(w.x, 0u, 0x4342));
                        Bv[1][0] = byte2_pattern(__byte_perm(w.y, 0u, 0x4140));
                        Bv[1][1] = byte2_pattern(__byte_perm(w.y, 0u, 0x4342));
                    } else {
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(sv + (sl * NB + b) * TBV + lane * 4);
                        const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
                        Bv[0][0] = nib2_pattern((lo & 0xFu) | ((lo >> 4) & 0xF0u));
                        Bv[0][1] = nib2_pattern(((lo >> 16) & 0xFu) | ((lo >> 20) & 0xF0u));
                        Bv[1][0] = nib2_pattern((hi & 0xFu) | ((hi >> 4) & 0xF0u));
                        Bv[1][1] = nib2_pattern(((hi >> 16) & 0xFu) | ((hi >> 20) & 0xF0u));
                    }
                    const float f = exact_pow2(Er - 127 - (VMB - 1));
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float c[4] = {0.f, 0.f, 0.f, 0.f};
                        mma16816(c, Ahi, Bv[hh][0], Bv[hh][1]);
                        mma16816(c, Alo, Bv[hh][0], Bv[hh][1]);
                        acc[bi][hh][0] = fmaf(c[0], f, acc[bi][hh][0]);
                        acc[bi][hh][1] = fmaf(c[1], f, acc[bi][hh][1]);
                    }
                }
            }
        }
        __syncthreads();  // the stage is free again
        if (tid == 0 && ci + 2 < c1) {
            fence_proxy_async_shared();
            issue(ci + 2);
        }
    }
    // ---- partial results: o = acc * 2^24 (the codes entered as multiples of 2^-24), then m and l
    float *base = a.part + (((int64_t)h * a.S + s) * G) * (D + 2);
    if (warp < NB && g4 < G) {
#pragma unroll
        for (int bi = 0; bi < NBC; ++bi) {
            const int b = warp + 8 * bi;
            if (b >= NB) break;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int col = 16 * b + 8 * hh + 2 * t4;
                base[(int64_t)g4 * (D + 2) + col] = acc[bi][hh][0] * 16777216.f;
                base[(int64_t)g4 * (D + 2) + col + 1] = acc[bi][hh][1] * 16777216.f;
            }
        }
    }
    if (tid < G) {
        base[(int64_t)tid * (D + 2) + D] = m_s[tid];
        base[(int64_t)tid * (D + 2) + D + 1] = l_s[tid];
    }
}

constexpr int kMergeThreads = 1024;
constexpr int kMaxSplits = 1024;

// Deterministic block reductions over kMergeThreads threads (warp butterflies, then warp 0 in order).
__device__ __forceinline__ float block_max(float v, float *red) {
    v = warp_max(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        const float r = warp_max(red[threadIdx.x]);
        if (threadIdx.x == 0) red[32] = r;
    }
    __syncthreads();
    const float r = red[32];
    __syncthreads();
    return r;
}
__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        const float r = warp_sum(red[threadIdx.x]);
        if (threadIdx.x == 0) red[32] = r;
    }
    __syncthreads();
    const float r = red[32];
    __syncthreads();
    return r;
}

// One CTA per query head: merge the S partial results (max, weights and normaliser over all threads;
// the weighted sum with the splits dealt to kMergeThreads / D groups of D threads); then rotate back
// (H_d / d) when V is stored rotated.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const float *part, int kvh, int G, int S, int rot,
                                                                   float *out) {
    constexpr int NSG = kMergeThreads / D;
    __shared__ float w_s[kMaxSplits];
    __shared__ float red[33];
    __shared__ float osum[NSG][D];
    __shared__ float x[D];
    grid_dep_wait();
    const int j = blockIdx.x, h = j / G, g = j % G, tid = threadIdx.x;
    const int64_t sstride = (int64_t)G * (D + 2);
    const float *pj = part + ((int64_t)h * S * G + g) * (D + 2);  // split s at pj + s * sstride
    float m = -INFINITY;
    for (int s = tid; s < S; s += kMergeThreads) m = fmaxf(m, pj[s * sstride + D]);
    const float M = block_max(m, red);
    float l = 0.f;
    for (int s = tid; s < S; s += kMergeThreads) {
        const float ms = pj[s * sstride + D];
        const float w = ms == -INFINITY ? 0.f : __expf(ms - M);  // a split with no tokens has m = -inf
        w_s[s] = w;
        l = fmaf(pj[s * sstride + D + 1], w, l);
    }
    const float L = block_sum(l, red);  // its barriers also publish w_s
    const int col = tid % D, sg = tid / D;
    float o = 0.f;
    for (int s = sg; s < S; s += NSG) o = fmaf(pj[s * sstride + col], w_s[s], o);
    osum[sg][col] = o;
    __syncthreads();
    float y = 0.f;
    if (sg == 0) {
        for (int k = 0; k < NSG; ++k) y += osum[k][col];
        y /= L;
        x[col] = y;
    }
    if (rot) {
        __syncthreads();
        for (int hh = 1; hh < D; hh <<= 1) {
            float a = 0.f, b = 0.f;
            if (sg == 0) {
                a = x[col & ~hh];
                b = x[col | hh];
            }
            __syncthreads();
            if (sg == 0) x[col] = (col & hh) ? a - b : a + b;
            __syncthreads();
        }
        if (sg == 0) y = x[col] * (1.0f / D);
    }
    if (sg == 0) out[(int64_t)j * D + col] = y;
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
    *S = (int)std::min<int64_t>(s, kMaxSplits);
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
    constexpr int STAGE = kChunk * (code_bytes_per_token(KF, D) + code_bytes_per_token(VF, D) + 2 * (D / 16));
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
    *code_bytes = (size_t)kv_heads * capacity * code_bytes_per_token(fmt, head_dim);
    *exp_bytes = (size_t)kv_heads * capacity * (head_dim / 16);
    return BFP_OK;
}

int bfp_kv_encode_host(const bfp_kv_cache *cache, const uint16_t *k, const uint16_t *v, int64_t pos, int n_new,
                       int nthreads) {
    int rc = check_cache(cache);
    if (rc) return rc;
    if (!k || !v) return fail(BFP_EINVAL, "null k or v");
    if (n_new < 1 || pos < 0 || pos + n_new > cache->capacity) return fail(BFP_ESHAPE, "tokens outside the capacity");
    const int d = cache->head_dim, nb = d / 16, kvh = cache->kv_heads;
    const int64_t rows = (int64_t)n_new * kvh * 2;
    const bool good = parallel_groups(rows, nthreads, [&](int64_t row) {
        const int which = (int)(row & 1);
        const int64_t rest = row >> 1, tok = rest / kvh;
        const int h = (int)(rest % kvh);
        const uint16_t *src = (which ? v : k) + (tok * kvh + h) * d;
        std::vector<float> x((size_t)d);
        for (int i = 0; i < d; ++i) {
            const uint32_t u = (uint32_t)src[i] << 16;
            std::memcpy(&x[(size_t)i], &u, 4);
        }
        if (which && cache->v_rotated)  // fast Walsh-Hadamard transform in fp32, stages 1, 2, 4, ...
            for (int hh = 1; hh < d; hh <<= 1)
                for (int i = 0; i < d; ++i)
                    if (!(i & hh)) {
                        const float a = x[(size_t)i], b = x[(size_t)(i + hh)];
                        x[(size_t)i] = a + b;
                        x[(size_t)(i + hh)] = a - b;
                    }
        const int fmt = which ? cache->v_fmt : cache->k_fmt, mb = fmt == BFP_FMT_BFP8 ? 7 : 3;
        const int tb = fmt == BFP_FMT_BFP8 ? 256 : 128;
        const int64_t slot = pos + tok, r = slot & 15;
        uint8_t *cc = static_cast<uint8_t *>(which ? cache->v_codes : cache->k_codes);
        uint8_t *ce = static_cast<uint8_t *>(which ? cache->v_exps : cache->k_exps);
        for (int b = 0; b < nb; ++b) {
            uint8_t E, c[16];
            if (!encode_block(&x[(size_t)16 * b], mb, &E, c)) return false;
            ce[((int64_t)h * cache->capacity + slot) * nb + b] = E;
            uint8_t *tile = cc + (((int64_t)h * (cache->capacity / 16) + (slot >> 4)) * nb + b) * tb;
            for (int j = 0; j < 4; ++j) {  // K: a row's 4 codes of columns 4j..4j+3 in its word or half
                if (which) break;
                if (fmt == BFP_FMT_BFP8) {
                    auto pat = [](uint32_t code) { return (code & 0x7Fu) | (((code >> 7) & 1u) << 15); };
                    const uint32_t p01 = pat(c[4 * j]) | (pat(c[4 * j + 1]) << 16);
                    const uint32_t p23 = pat(c[4 * j + 2]) | (pat(c[4 * j + 3]) << 16);
                    const uint32_t w = p01 | ((p23 << 8) | (p23 >> 24));
                    std::memcpy(tile + (4 * (r & 7) + j) * 8 + (r >> 3) * 4, &w, 4);
                } else {
                    const uint16_t hw = (uint16_t)(c[4 * j] | (c[4 * j + 1] << 4) | (c[4 * j + 2] << 8) |
                                                   (c[4 * j + 3] << 12));
                    std::memcpy(tile + (4 * (r & 7) + j) * 4 + (r >> 3) * 2, &hw, 2);
                }
            }
            if (which) {  // V: one byte per (token, column), or per (token, column pair c, c + 8)
                if (fmt == BFP_FMT_BFP8)
                    for (int col = 0; col < 16; ++col) tile[(4 * (col & 7) + (r >> 2)) * 8 + (col >> 3) * 4 + (r & 3)] = c[col];
                else
                    for (int col = 0; col < 8; ++col)
                        tile[(4 * col + (r >> 2)) * 4 + (r & 3)] = (uint8_t)(c[col] | (c[col + 8] << 4));
            }
        }
        return true;
    });
    if (!good) return fail(BFP_ENONFINITE, "k or v holds NaN or Inf");
    return BFP_OK;
}

int bfp_kv_read_fields(const bfp_kv_cache *cache, int which, int64_t t0, int64_t n, uint8_t *exps, uint8_t *codes) {
    if (!cache) return fail(BFP_EINVAL, "null cache");
    if (which != 0 && which != 1) return fail(BFP_EINVAL, "which must be 0 (K) or 1 (V)");
    int rc = check_cache(cache);
    if (rc) return rc;
    if (!exps || !codes) return fail(BFP_EINVAL, "null output");
    if (t0 < 0 || n < 1 || t0 + n > cache->capacity) return fail(BFP_ESHAPE, "tokens outside the capacity");
    const int d = cache->head_dim, nb = d / 16, fmt = which ? cache->v_fmt : cache->k_fmt;
    const int tb = fmt == BFP_FMT_BFP8 ? 256 : 128;
    const uint8_t *cc = static_cast<const uint8_t *>(which ? cache->v_codes : cache->k_codes);
    const uint8_t *ce = static_cast<const uint8_t *>(which ? cache->v_exps : cache->k_exps);
    for (int h = 0; h < cache->kv_heads; ++h)
        for (int64_t i = 0; i < n; ++i) {
            const int64_t t = t0 + i, r = t & 15;
            for (int b = 0; b < nb; ++b) {
                exps[((int64_t)h * n + i) * nb + b] = ce[((int64_t)h * cache->capacity + t) * nb + b];
                const uint8_t *tile = cc + (((int64_t)h * (cache->capacity / 16) + (t >> 4)) * nb + b) * tb;
                uint8_t *out = codes + ((int64_t)h * n + i) * d + 16 * b;
                for (int c = 0; c < 16; ++c) {
                    uint32_t code;
                    if (!which && fmt == BFP_FMT_BFP8) {  // pattern word: P(c0, c1) | rotl(P(c2, c3), 8)
                        uint32_t w;
                        std::memcpy(&w, tile + (4 * (r & 7) + c / 4) * 8 + (r >> 3) * 4, 4);
                        const uint32_t p = (c & 2) ? ((w >> 8) | (w << 24)) : w;  // rotate right by 8 for c2, c3
                        const uint32_t half = (c & 1) ? (p >> 16) : (p & 0xFFFFu);
                        code = (half & 0x7Fu) | (((half >> 15) & 1u) << 7);
                    } else if (!which) {
                        const uint8_t byte = tile[(4 * (r & 7) + c / 4) * 4 + (r >> 3) * 2 + (c & 3) / 2];
                        code = (c & 1) ? (byte >> 4) : (byte & 15u);
                    } else if (fmt == BFP_FMT_BFP8) {
                        code = tile[(4 * (c & 7) + (r >> 2)) * 8 + (c >> 3) * 4 + (r & 3)];
                    } else {
                        const uint8_t byte = tile[(4 * (c & 7) + (r >> 2)) * 4 + (r & 3)];
                        code = (c >> 3) ? (byte >> 4) : (byte & 15u);
                    }
                    out[c] = (uint8_t)code;
                }
            }
        }
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
        case 64: e = launch_pdl(attn_merge_kernel<64>, dim3(q_heads), dim3(kMergeThreads), 0, st, part, a.kvh, a.G, S, cache->v_rotated, out); break;
        case 128: e = launch_pdl(attn_merge_kernel<128>, dim3(q_heads), dim3(kMergeThreads), 0, st, part, a.kvh, a.G, S, cache->v_rotated, out); break;
        default: e = launch_pdl(attn_merge_kernel<256>, dim3(q_heads), dim3(kMergeThreads), 0, st, part, a.kvh, a.G, S, cache->v_rotated, out); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "launch attention merge");
    return BFP_OK;
}

}  // extern "C"
