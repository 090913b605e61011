// Tensor-core inner loops over tile records (include/bfpmoe.h layout).
//
// One record = 16 weight rows x CB blocks of 16 along k. A warp reads the
// record's 512 code bytes as one 16-byte vector per lane, unpacks each block
// into an A fragment (fp16 subnormal lanes +-m * 2^-24, exact), multiplies it
// by the activation fragment of the same block with mma.sync m16n8k16 into a
// zeroed fp32 tile, and folds that tile into the running sum scaled by the
// block's 2^(E-127): one BFP block is exactly one k16 MMA step, so the
// per-16-value exponent is applied where it belongs and nothing is rounded
// before the fp32 sum. The constant 2^(24 - (mb-1)) and the activation's own
// power-of-two scale are applied once, in the epilogue.
#pragma once

#include "bfp_device.cuh"

namespace bfp {
namespace dev {

// acc[r][grp][i] += sum over the record's blocks of 2^(E-127) * (A_r . B_grp)
//   recs[r]:  record r in shared memory (NREC records share the activation fragments)
//   frag:     activation fragments, [grp][block][lane] uint2; frag_lo (HILO) a second,
//             low-order part added into the same tile before scaling
//   kb0:      index of the record's first block in the fragment arrays
//   grp_mask: bit g set = compute activation group g (8 rows each)
template <int FMT, int NGRP, int NREC, bool HILO>
__device__ __forceinline__ void mma_records(const uint8_t *const recs[NREC], const uint2 *frag, const uint2 *frag_lo,
                                            int kbp, int kb0, int lane, uint32_t grp_mask,
                                            float acc[NREC][NGRP][4]) {
    const int g = lane >> 2;
    uint4 wq[NREC];
    uint32_t e0[NREC], e1[NREC];
#pragma unroll
    for (int r = 0; r < NREC; ++r) {
        wq[r] = *reinterpret_cast<const uint4 *>(recs[r] + 16 * lane);
        if constexpr (FMT == 4) {
            const uint2 eq = *reinterpret_cast<const uint2 *>(recs[r] + 512 + 8 * g);
            e0[r] = eq.x;
            e1[r] = eq.y;
        } else {
            e0[r] = *reinterpret_cast<const uint32_t *>(recs[r] + 512 + 4 * g);
            e1[r] = 0;
        }
    }
    constexpr int CB = FMT == 4 ? 4 : 2;
#pragma unroll
    for (int b = 0; b < CB; ++b) {
        uint2 bx[NGRP], bl[NGRP];
#pragma unroll
        for (int grp = 0; grp < NGRP; ++grp) {
            if (grp_mask & (1u << grp)) {
                bx[grp] = frag[(grp * kbp + kb0 + b) * kWarp + lane];
                if constexpr (HILO) bl[grp] = frag_lo[(grp * kbp + kb0 + b) * kWarp + lane];
            }
        }
#pragma unroll
        for (int r = 0; r < NREC; ++r) {
            uint32_t a[4];
            float s0, s1;
            if constexpr (FMT == 4) {
                const uint32_t wsel = b == 0 ? wq[r].x : b == 1 ? wq[r].y : b == 2 ? wq[r].z : wq[r].w;
                unpack_bfp4(wsel, a);
                const uint32_t ew = b < 2 ? e0[r] : e1[r];
                s0 = exp_scale(ew, 2 * (b & 1));
                s1 = exp_scale(ew, 2 * (b & 1) + 1);
            } else {
                if (b == 0)
                    unpack_bfp8(wq[r].x, wq[r].y, a);
                else
                    unpack_bfp8(wq[r].z, wq[r].w, a);
                s0 = exp_scale(e0[r], 2 * b);
                s1 = exp_scale(e0[r], 2 * b + 1);
            }
#pragma unroll
            for (int grp = 0; grp < NGRP; ++grp) {
                if (grp_mask & (1u << grp)) {
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(c, a, bx[grp].x, bx[grp].y);
                    if constexpr (HILO) mma16816(c, a, bl[grp].x, bl[grp].y);
                    acc[r][grp][0] = fmaf(s0, c[0], acc[r][grp][0]);
                    acc[r][grp][1] = fmaf(s0, c[1], acc[r][grp][1]);
                    acc[r][grp][2] = fmaf(s1, c[2], acc[r][grp][2]);
                    acc[r][grp][3] = fmaf(s1, c[3], acc[r][grp][3]);
                }
            }
        }
    }
}

// Position of accumulator element (grp, i) of a lane in the 16 x (8*NGRP) output tile:
//   weight row (within the 16-row group) and activation row.
__device__ __forceinline__ int acc_wrow(int lane, int i) { return (lane >> 2) + 8 * (i >> 1); }
__device__ __forceinline__ int acc_xrow(int lane, int grp, int i) { return 8 * grp + 2 * (lane & 3) + (i & 1); }

// Activation fragments for rows r < m of bf16 x (row stride ldx, k columns):
// optional RMS normalisation t = bf16(x / sqrt(mean(x^2) + eps)) (fp32), then
// each row scaled by the power of two shift[r] that puts its max |value| in
// [2^14, 2^15) and rounded to fp16 (exact for every bf16 value above
// 2^-14 of the row maximum). Rows >= m and blocks >= k/16 are zero.
// Called by the NC consumer threads only (named barrier 1).
template <int NC>
__device__ __noinline__ void build_act_frags(const uint16_t *x, int64_t ldx, int m, int k, int kbp, int ngrp, bool norm, float eps,
                                uint32_t *frag, int *shift, float *inv_out, int tid, int warp, int lane) {
    const int nvec = ngrp * kbp * kWarp * 2 / 4;
    for (int i = tid; i < nvec; i += NC) reinterpret_cast<uint4 *>(frag)[i] = make_uint4(0, 0, 0, 0);
    for (int r = warp; r < m; r += NC / kWarp) {
        const uint16_t *xr = x + (int64_t)r * ldx;
        float inv = 1.f;
        if (norm) {
            float ss = 0.f;
            for (int j = lane; j < k; j += kWarp) {
                float v = bf16_bits_to_f32(xr[j]);
                ss = fmaf(v, v, ss);
            }
            ss = warp_sum(ss);
            inv = 1.0f / sqrtf(ss / (float)k + eps);
        }
        float mx = 0.f;
        for (int j = lane; j < k; j += kWarp) {
            float v = bf16_bits_to_f32(xr[j]);
            if (norm) v = __bfloat162float(__float2bfloat16_rn(v * inv));
            mx = fmaxf(mx, fabsf(v));
        }
        mx = warp_max(mx);
        if (lane == 0) {
            shift[r] = frag_shift(mx);
            if (inv_out) inv_out[r] = inv;
        }
    }
    bar_sync(1, NC);
    const int kb = k / 16;
    const int total = m * kb * 8;
    for (int idx = tid; idx < total; idx += NC) {
        const int r = idx / (kb * 8);
        const int rem = idx - r * kb * 8;
        const int b = rem >> 3, j = rem & 7;
        const uint32_t two = *reinterpret_cast<const uint32_t *>(x + (int64_t)r * ldx + 16 * b + 2 * j);
        float v0 = bf16_bits_to_f32(two & 0xFFFFu), v1 = bf16_bits_to_f32(two >> 16);
        if (norm) {
            const float inv = inv_out[r];
            v0 = __bfloat162float(__float2bfloat16_rn(v0 * inv));
            v1 = __bfloat162float(__float2bfloat16_rn(v1 * inv));
        }
        const int sh = shift[r];
        frag[frag_word(r, b, j, kbp)] = pack_half2(scalbnf(v0, sh), scalbnf(v1, sh));
    }
    bar_sync(1, NC);
}


}  // namespace dev
}  // namespace bfp
