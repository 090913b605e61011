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
#include "bfp_trace.h"

namespace bfp {
namespace dev {

// Exponent bytes of one record (16 rows x CB blocks), and how many of a call's bytes each lane converts.
template <int FMT>
__host__ __device__ constexpr int rec_exp_bytes() { return FMT == 4 ? 64 : 32; }
// Scratch floats one warp needs for mma_records<FMT, *, NREC, *>.
template <int FMT, int NREC>
__host__ __device__ constexpr int rec_scale_floats() { return NREC * rec_exp_bytes<FMT>(); }

// acc[r][grp][i] += sum over the record's blocks of 2^(E-127) * (A_r . B_grp), grp < NG
//   recs[r]:  record r in shared memory (NREC records share the activation fragments)
//   frag:     activation fragments of the first group computed: [grp][block][lane] uint2, groups
//             kbp blocks apart; frag_lo (HILO) a second, low-order part added into the same
//             tile before scaling, same layout
//   kb0:      index of the record's first block in the fragment arrays (a multiple of the
//             record's block count)
//   esc:      this warp's scratch of rec_scale_floats<FMT, NREC>() floats (16-byte aligned)
// Branch-free: the group count is a template parameter, so the compiler can interleave the
// independent tiles of a record. The four lanes of a row pair (lane >> 2 equal) need the same
// block scales, so the warp first turns the records' exponent bytes into fp32 scales once, each
// lane its share, through esc: the integer work per scale is done once instead of four times.
template <int FMT, int NG, int NREC, bool HILO>
__device__ __forceinline__ void mma_records(const uint8_t *const recs[NREC], const uint2 *frag, const uint2 *frag_lo,
                                            int kbp, int kb0, int lane, float *esc, float acc[NREC][NG][4]) {
    constexpr int EB = rec_exp_bytes<FMT>();
    constexpr int CB = FMT == 4 ? 4 : 2;
    constexpr int BPL = NREC * EB / kWarp;  // exponent bytes converted per lane
    static_assert(BPL == 1 || BPL == 2 || BPL == 4, "unsupported record count");
    const int g = lane >> 2;
    uint4 wq[NREC];
#pragma unroll
    for (int r = 0; r < NREC; ++r) wq[r] = *reinterpret_cast<const uint4 *>(recs[r] + 16 * lane);
    {
        const int byte0 = lane * BPL;  // byte of the call's exponents, records in order
        const uint8_t *rp = recs[0];
#pragma unroll
        for (int r = 1; r < NREC; ++r)
            if (byte0 >= r * EB) rp = recs[r];
        const uint8_t *src = rp + kRecCodes + byte0 % EB;
        __syncwarp();  // every lane is done reading the previous call's scales
        if constexpr (BPL == 4) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(src);
            *reinterpret_cast<float4 *>(esc + byte0) =
                make_float4(exp_scale(w, 0), exp_scale(w, 1), exp_scale(w, 2), exp_scale(w, 3));
        } else if constexpr (BPL == 2) {
            const uint32_t w = *reinterpret_cast<const uint16_t *>(src);
            *reinterpret_cast<float2 *>(esc + byte0) = make_float2(exp_scale(w, 0), exp_scale(w, 1));
        } else {
            esc[byte0] = exp_scale(*src, 0);
        }
        __syncwarp();
    }
    // this lane's scales: record r, block b -> sc[r][2b] (row g), sc[r][2b + 1] (row g + 8)
    float sc[NREC][2 * CB];
#pragma unroll
    for (int r = 0; r < NREC; ++r) {
#pragma unroll
        for (int q = 0; q < CB / 2; ++q) {
            const float4 f = *reinterpret_cast<const float4 *>(esc + r * EB + 2 * CB * g + 4 * q);
            sc[r][4 * q] = f.x;
            sc[r][4 * q + 1] = f.y;
            sc[r][4 * q + 2] = f.z;
            sc[r][4 * q + 3] = f.w;
        }
    }
    // fragment of block kb0 + b for this lane: lane ^ frag_swz(kb0 + b), and since kb0 is a
    // multiple of CB, (kb0 + b) & 7 = (kb0 & 7) | b
    const int l0 = lane ^ ((kb0 & 7) << 2);
    const uint2 *fh = frag + (int64_t)kb0 * kWarp;
    const uint2 *fl = HILO ? frag_lo + (int64_t)kb0 * kWarp : nullptr;
#pragma unroll
    for (int b = 0; b < CB; ++b) {
        const int li = b * kWarp + (l0 ^ (b << 2));
        uint2 bx[NG], bl[NG];
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) {
            bx[grp] = fh[(int64_t)grp * kbp * kWarp + li];
            if constexpr (HILO) bl[grp] = fl[(int64_t)grp * kbp * kWarp + li];
        }
#pragma unroll
        for (int r = 0; r < NREC; ++r) {
            uint32_t a[4];
            if constexpr (FMT == 4) {
                const uint32_t wsel = b == 0 ? wq[r].x : b == 1 ? wq[r].y : b == 2 ? wq[r].z : wq[r].w;
                unpack_bfp4(wsel, a);
            } else {
                if (b == 0)
                    unpack_bfp8(wq[r].x, wq[r].y, a);
                else
                    unpack_bfp8(wq[r].z, wq[r].w, a);
            }
            const float s0 = sc[r][2 * b], s1 = sc[r][2 * b + 1];
#pragma unroll
            for (int grp = 0; grp < NG; ++grp) {
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

// acc[grp][i] += sum over NREC consecutive records of one row group (record r covers the CB blocks
// from kb0 + r * CB) of 2^(E-127) * (A . B_grp): mma_records for records that follow each other
// along k and share one accumulator (the down projection's row groups). One exponent pass and one
// set of loads for all NREC records, so the per-record overhead is paid once per call.
template <int FMT, int NG, int NREC, bool HILO>
__device__ __forceinline__ void mma_records_k(const uint8_t *recs, int rec_bytes, const uint2 *frag,
                                              const uint2 *frag_lo, int kbp, int kb0, int lane, float *esc,
                                              float acc[NG][4]) {
    constexpr int EB = rec_exp_bytes<FMT>();
    constexpr int CB = FMT == 4 ? 4 : 2;
    constexpr int BPL = NREC * EB / kWarp;  // exponent bytes converted per lane
    static_assert(BPL == 1 || BPL == 2 || BPL == 4, "unsupported record count");
    const int g = lane >> 2;
    uint4 wq[NREC];
#pragma unroll
    for (int r = 0; r < NREC; ++r) wq[r] = *reinterpret_cast<const uint4 *>(recs + (size_t)r * rec_bytes + 16 * lane);
    {
        const int byte0 = lane * BPL;  // byte of the call's exponents, records in order
        const uint8_t *src = recs + (size_t)(byte0 / EB) * rec_bytes + kRecCodes + byte0 % EB;
        __syncwarp();  // every lane is done reading the previous call's scales
        if constexpr (BPL == 4) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(src);
            *reinterpret_cast<float4 *>(esc + byte0) =
                make_float4(exp_scale(w, 0), exp_scale(w, 1), exp_scale(w, 2), exp_scale(w, 3));
        } else if constexpr (BPL == 2) {
            const uint32_t w = *reinterpret_cast<const uint16_t *>(src);
            *reinterpret_cast<float2 *>(esc + byte0) = make_float2(exp_scale(w, 0), exp_scale(w, 1));
        } else {
            esc[byte0] = exp_scale(*src, 0);
        }
        __syncwarp();
    }
    float sc[NREC][2 * CB];
#pragma unroll
    for (int r = 0; r < NREC; ++r) {
#pragma unroll
        for (int q = 0; q < CB / 2; ++q) {
            const float4 f = *reinterpret_cast<const float4 *>(esc + r * EB + 2 * CB * g + 4 * q);
            sc[r][4 * q] = f.x;
            sc[r][4 * q + 1] = f.y;
            sc[r][4 * q + 2] = f.z;
            sc[r][4 * q + 3] = f.w;
        }
    }
#pragma unroll
    for (int r = 0; r < NREC; ++r) {
        const int kr = kb0 + r * CB;  // a multiple of CB: (kr + b) & 7 = (kr & 7) | b
        const int l0 = lane ^ ((kr & 7) << 2);
        const uint2 *fh = frag + (int64_t)kr * kWarp;
        const uint2 *fl = HILO ? frag_lo + (int64_t)kr * kWarp : nullptr;
#pragma unroll
        for (int b = 0; b < CB; ++b) {
            const int li = b * kWarp + (l0 ^ (b << 2));
            uint2 bx[NG], bl[NG];
#pragma unroll
            for (int grp = 0; grp < NG; ++grp) {
                bx[grp] = fh[(int64_t)grp * kbp * kWarp + li];
                if constexpr (HILO) bl[grp] = fl[(int64_t)grp * kbp * kWarp + li];
            }
            uint32_t a[4];
            if constexpr (FMT == 4) {
                const uint32_t wsel = b == 0 ? wq[r].x : b == 1 ? wq[r].y : b == 2 ? wq[r].z : wq[r].w;
                unpack_bfp4(wsel, a);
            } else {
                if (b == 0)
                    unpack_bfp8(wq[r].x, wq[r].y, a);
                else
                    unpack_bfp8(wq[r].z, wq[r].w, a);
            }
            const float s0 = sc[r][2 * b], s1 = sc[r][2 * b + 1];
#pragma unroll
            for (int grp = 0; grp < NG; ++grp) {
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(c, a, bx[grp].x, bx[grp].y);
                if constexpr (HILO) mma16816(c, a, bl[grp].x, bl[grp].y);
                acc[grp][0] = fmaf(s0, c[0], acc[grp][0]);
                acc[grp][1] = fmaf(s0, c[1], acc[grp][1]);
                acc[grp][2] = fmaf(s1, c[2], acc[grp][2]);
                acc[grp][3] = fmaf(s1, c[3], acc[grp][3]);
            }
        }
    }
}

// Position of accumulator element (grp, i) of a lane in the 16 x (8*NGRP) output tile:
//   weight row (within the 16-row group) and activation row.
__device__ __forceinline__ int acc_wrow(int lane, int i) { return (lane >> 2) + 8 * (i >> 1); }
__device__ __forceinline__ int acc_xrow(int lane, int grp, int i) { return 8 * grp + 2 * (lane & 3) + (i & 1); }

// Segments per activation row: with few rows, each row is split along k over up to 16 warps (whole
// 16-value blocks) so that every warp of the CTA has a share of the row statistics and fragments.
template <int NC>
__device__ __forceinline__ int act_segments(int m, int k) {
    constexpr int NW = NC / kWarp;
    const int kb = k / 16;
    int S = 1;
    while (m * S * 2 <= NW && S * 2 <= 16 && kb % (S * 2) == 0) S *= 2;
    return S;
}

// Statistics of the bf16 activation rows r < m staged in shared memory (row stride ldx elements,
// k columns, k % 16 == 0): shift[r] = the power of two that puts the row's max |value| in
// [2^14, 2^15) for its fp16 fragments, and with norm the RMS normalisation
// t = bf16(x / sqrt(mean(x^2) + eps)) (fp32), applied to the rows in place (inv[r] = the factor).
// The max |t| is bf16(max|x| * inv): rounding is monotonic. red: NC/32 float2 of scratch.
// Called by the NC threads (warps 0 .. NC/32 - 1 of the call; warp = the caller's warp index among
// them) that meet at named barrier `bar`; ends with that barrier.
template <int NC>
__device__ __forceinline__ void act_rows_prepare_body(uint16_t *x, int64_t ldx, int m, int k, bool norm, float eps,
                                              int *shift, float *inv_out, float2 *red, int bar, int warp, int lane) {
    constexpr int NW = NC / kWarp;
    const int S = act_segments<NC>(m, k);
    const int nvs = k / 8 / S;  // 16-byte vectors per segment
    for (int it = warp; it < m * S; it += NW) {
        const int r = it / S, sg = it - r * S;
        uint4 *xr = reinterpret_cast<uint4 *>(x + (int64_t)r * ldx) + sg * nvs;
        float ss = 0.f;
        uint32_t mx2 = 0u;  // max |x| of the low and high bf16 halves, as bit patterns
        for (int i = lane; i < nvs; i += kWarp) {
            const uint4 v = xr[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                mx2 = __vmaxu2(mx2, w[h] & 0x7FFF7FFFu);
                if (norm) {
                    const float lo = bf16_bits_to_f32(w[h] & 0xFFFFu), hi = bf16_bits_to_f32(w[h] >> 16);
                    ss = fmaf(lo, lo, ss);
                    ss = fmaf(hi, hi, ss);
                }
            }
        }
        float mx = bf16_bits_to_f32(max(mx2 & 0xFFFFu, mx2 >> 16));
        mx = warp_max(mx);
        if (norm) ss = warp_sum(ss);
        if (S > 1) {
            if (lane == 0) red[it] = make_float2(ss, mx);  // it < NW when S > 1
        } else {
            float inv = 1.f;
            if (norm) {
                inv = 1.0f / sqrtf(ss / (float)k + eps);
                for (int i = lane; i < nvs; i += kWarp) {
                    uint4 v = xr[i];
                    uint32_t *w = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        w[h] = (uint32_t)f32_to_bf16_bits(bf16_bits_to_f32(w[h] & 0xFFFFu) * inv) |
                               ((uint32_t)f32_to_bf16_bits(bf16_bits_to_f32(w[h] >> 16) * inv) << 16);
                    xr[i] = v;
                }
                mx = bf16_bits_to_f32(f32_to_bf16_bits(mx * inv));
            }
            if (lane == 0) {
                shift[r] = frag_shift(mx);
                if (inv_out) inv_out[r] = inv;
            }
        }
    }
    if (S > 1) {
        bar_sync(bar, NC);
        for (int it = warp; it < m * S; it += NW) {
            const int r = it / S, sg = it - r * S;
            float ss = 0.f, mx = 0.f;
            for (int q = 0; q < S; ++q) {  // segments in order: the same sum in every warp
                const float2 v = red[r * S + q];
                ss += v.x;
                mx = fmaxf(mx, v.y);
            }
            float inv = 1.f;
            if (norm) {
                inv = 1.0f / sqrtf(ss / (float)k + eps);
                uint4 *xr = reinterpret_cast<uint4 *>(x + (int64_t)r * ldx) + sg * nvs;
                for (int i = lane; i < nvs; i += kWarp) {
                    uint4 v = xr[i];
                    uint32_t *w = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        w[h] = (uint32_t)f32_to_bf16_bits(bf16_bits_to_f32(w[h] & 0xFFFFu) * inv) |
                               ((uint32_t)f32_to_bf16_bits(bf16_bits_to_f32(w[h] >> 16) * inv) << 16);
                    xr[i] = v;
                }
                mx = bf16_bits_to_f32(f32_to_bf16_bits(mx * inv));
            }
            if (sg == 0 && lane == 0) {
                shift[r] = frag_shift(mx);
                if (inv_out) inv_out[r] = inv;
            }
        }
    }
    bar_sync(bar, NC);
}
// The same, as a call: one copy of the code for kernels that reach it from more than one place.
template <int NC>
__device__ __noinline__ void act_rows_prepare(uint16_t *x, int64_t ldx, int m, int k, bool norm, float eps,
                                              int *shift, float *inv_out, float2 *red, int bar, int warp, int lane) {
    act_rows_prepare_body<NC>(x, ldx, m, k, norm, eps, shift, inv_out, red, bar, warp, lane);
}

// fp16 activation fragments of the prepared rows (act_rows_prepare): row r scaled by 2^shift[r] and
// rounded to fp16 (exact for every bf16 value above 2^-14 of the row maximum); rows m .. 8 ngrp - 1
// and blocks k/16 .. kbp - 1 are zero. Item (row of the 8 ngrp, segment of the kbp blocks) per warp,
// padding rows and blocks included, so every fragment word is written once and no clearing pass is
// needed; lane (bb, t) = (lane >> 2, lane & 3) assembles whole fragments (cols 2t|2t+1 and
// 2t+8|2t+9 of the segment's blocks b with b & 7 = bb) and stores each with one 8-byte store; the
// XOR swizzle spreads a warp's stores over the banks. Called like act_rows_prepare (tid unused).
template <int NC>
__device__ __forceinline__ void act_rows_frags_body(const uint16_t *x, int64_t ldx, int m, int k, int kbp, int ngrp,
                                            const int *shift, uint32_t *frag, int bar, int tid, int warp, int lane) {
    constexpr int NW = NC / kWarp;
    const int kb = k / 16, mp = 8 * ngrp;
    uint2 *f2 = reinterpret_cast<uint2 *>(frag);
    int S = 1;  // segments per row: spread the rows over every warp
    while (mp * S * 2 <= NW && (kbp / 8) % (S * 2) == 0) S *= 2;
    const int bs = kbp / S;  // blocks per segment (a multiple of 8 when S > 1)
    const int bb = lane >> 2, t = lane & 3;
    for (int it = warp; it < mp * S; it += NW) {
        const int r = it / S, sg = it - r * S;
        const bool real = r < m;
        const uint16_t *xrow = x + (int64_t)(real ? r : 0) * ldx;
        const float sc = real ? pow2f(shift[r]) : 0.f;
        const int grp = r >> 3, g = r & 7;
        uint2 *fr = f2 + (int64_t)grp * kbp * kWarp + ((4 * g + t) ^ (bb << 2));  // (b & 7) == bb
        const int b0 = sg * bs, b1 = b0 + bs;
        for (int b = b0 + ((bb - b0) & 7); b < b1; b += 8) {
            uint2 v = make_uint2(0u, 0u);
            if (real && b < kb) {
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(xrow + 16 * b + 2 * t);
                const uint32_t w1 = *reinterpret_cast<const uint32_t *>(xrow + 16 * b + 2 * t + 8);
                v = make_uint2(pack_half2(bf16_bits_to_f32(w0 & 0xFFFFu) * sc, bf16_bits_to_f32(w0 >> 16) * sc),
                               pack_half2(bf16_bits_to_f32(w1 & 0xFFFFu) * sc, bf16_bits_to_f32(w1 >> 16) * sc));
            }
            fr[(int64_t)b * kWarp] = v;
        }
    }
    bar_sync(bar, NC);
}
// The same, as a call: one copy of the code for kernels that reach it from more than one place.
template <int NC>
__device__ __noinline__ void act_rows_frags(const uint16_t *x, int64_t ldx, int m, int k, int kbp, int ngrp,
                                            const int *shift, uint32_t *frag, int bar, int tid, int warp, int lane) {
    act_rows_frags_body<NC>(x, ldx, m, k, kbp, ngrp, shift, frag, bar, tid, warp, lane);
}

// act_rows_prepare and act_rows_frags in one pass, for rows staged apart from the fragment area (up to
// 16 rows): the warp that converts a segment of row r first takes row r's statistics itself, over the
// whole row (every warp with a segment of the row computes the same values in the same order), so no
// CTA barrier separates the statistics from the fragments and no partial sums cross warps. The same
// fragment values and layout as act_rows_prepare followed by act_rows_frags (with norm, t =
// bf16(x * inv) is formed on the fly and the staged rows are left as they are); shift[r] is written by
// the warp of row r's first segment. Ends with barrier `bar`.
template <int NC>
__device__ __forceinline__ void act_rows_stats_frags_body(const uint16_t *x, int64_t ldx, int m, int k, int kbp,
                                                          int ngrp, bool norm, float eps, int *shift, uint32_t *frag,
                                                          int bar, int warp, int lane) {
    constexpr int NW = NC / kWarp;
    const int kb = k / 16, mp = 8 * ngrp, nv = k / 8;
    uint2 *f2 = reinterpret_cast<uint2 *>(frag);
    int S = 1;  // segments per row: spread the rows over every warp
    while (mp * S * 2 <= NW && (kbp / 8) % (S * 2) == 0) S *= 2;
    const int bs = kbp / S;  // blocks per segment (a multiple of 8 when S > 1)
    const int bb = lane >> 2, t = lane & 3;
    for (int it = warp; it < mp * S; it += NW) {
        const int r = it / S, sg = it - r * S;
        const bool real = r < m;
        const uint16_t *xrow = x + (int64_t)(real ? r : 0) * ldx;
        float sc = 0.f, inv = 1.f;
        if (real) {
            const uint4 *xr = reinterpret_cast<const uint4 *>(xrow);
            float ss = 0.f;
            uint32_t mx2 = 0u;  // max |x| of the low and high bf16 halves, as bit patterns
            for (int i = lane; i < nv; i += kWarp) {
                const uint4 v = xr[i];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    mx2 = __vmaxu2(mx2, w[h] & 0x7FFF7FFFu);
                    if (norm) {
                        const float lo = bf16_bits_to_f32(w[h] & 0xFFFFu), hi = bf16_bits_to_f32(w[h] >> 16);
                        ss = fmaf(lo, lo, ss);
                        ss = fmaf(hi, hi, ss);
                    }
                }
            }
            // bit patterns of non-negative bf16 values order as the values do
            float mx = bf16_bits_to_f32(__reduce_max_sync(0xffffffffu, max(mx2 & 0xFFFFu, mx2 >> 16)));
            if (norm) {
                inv = 1.0f / sqrtf(warp_sum(ss) / (float)k + eps);
                mx = bf16_bits_to_f32(f32_to_bf16_bits(mx * inv));
            }
            const int sh = frag_shift(mx);
            sc = pow2f(sh);
            if (sg == 0 && lane == 0) shift[r] = sh;
        }
        const int grp = r >> 3, g = r & 7;
        uint2 *fr = f2 + (int64_t)grp * kbp * kWarp + ((4 * g + t) ^ (bb << 2));  // (b & 7) == bb
        const int b0 = sg * bs, b1 = b0 + bs;
        for (int b = b0 + ((bb - b0) & 7); b < b1; b += 8) {
            uint2 v = make_uint2(0u, 0u);
            if (real && b < kb) {
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(xrow + 16 * b + 2 * t);
                const uint32_t w1 = *reinterpret_cast<const uint32_t *>(xrow + 16 * b + 2 * t + 8);
                float f[4] = {bf16_bits_to_f32(w0 & 0xFFFFu), bf16_bits_to_f32(w0 >> 16),
                              bf16_bits_to_f32(w1 & 0xFFFFu), bf16_bits_to_f32(w1 >> 16)};
                if (norm) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) f[q] = bf16_bits_to_f32(f32_to_bf16_bits(f[q] * inv));
                }
                v = make_uint2(pack_half2(f[0] * sc, f[1] * sc), pack_half2(f[2] * sc, f[3] * sc));
            }
            fr[(int64_t)b * kWarp] = v;
        }
    }
    bar_sync(bar, NC);
}

// act_rows_frags for four activation groups (32 rows) with the rows staged in the fragment area itself
// (row r at x + r * ldx, bf16). Group g's fragments (kbp blocks) take bytes [g F, (g + 1) F),
// F = kbp * 256, and its staged rows [g R, (g + 1) R), R = 16 ldx bytes; with ldx >= 16 kbp (R >= F),
// going from the first group up, a group's fragments never cover the staged rows of a group still to
// come. Per group, every thread reads its share (at most 8 fragment pairs: kbp <= 128) into registers,
// the threads meet at barrier `bar`, and the pairs are written in place. A warp reads one block of the
// group's 8 rows at once: with ldx = 8 mod 64 (rows 4 banks apart) those reads are free of bank
// conflicts. Same values and layout as act_rows_frags with ngrp = 4. Ends with barrier `bar`.
template <int NC>
__device__ __forceinline__ void act_rows_frags_inplace_body(const uint16_t *x, int64_t ldx, int m, int k, int kbp,
                                                    const int *shift, uint32_t *frag, int bar, int tid) {
    constexpr int KR = 8;
    const int kb = k / 16, per_group = kbp * kWarp;
    uint2 *f2 = reinterpret_cast<uint2 *>(frag);
    for (int grp = 0; grp < 4; ++grp) {
        uint2 v[KR];
#pragma unroll
        for (int j = 0; j < KR; ++j) {
            const int e = tid + j * NC;  // pair e of the group: block e / 32, position e % 32
            v[j] = make_uint2(0u, 0u);
            const int b = e / kWarp, l = (e - b * kWarp) ^ frag_swz(b);  // the lane whose pair sits there
            const int r = 8 * grp + (l >> 2), t = l & 3;
            if (e < per_group && r < m && b < kb) {
                const uint16_t *xr = x + (int64_t)r * ldx + 16 * b + 2 * t;
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(xr);
                const uint32_t w1 = *reinterpret_cast<const uint32_t *>(xr + 8);
                const float sc = pow2f(shift[r]);
                v[j] = make_uint2(pack_half2(bf16_bits_to_f32(w0 & 0xFFFFu) * sc, bf16_bits_to_f32(w0 >> 16) * sc),
                                  pack_half2(bf16_bits_to_f32(w1 & 0xFFFFu) * sc, bf16_bits_to_f32(w1 >> 16) * sc));
            }
        }
        bar_sync(bar, NC);
#pragma unroll
        for (int j = 0; j < KR; ++j) {
            const int e = tid + j * NC;
            if (e < per_group) f2[(int64_t)grp * per_group + e] = v[j];
        }
    }
    bar_sync(bar, NC);
}
// The same, as a call: one copy of the code for kernels that reach it from more than one place.
template <int NC>
__device__ __noinline__ void act_rows_frags_inplace(const uint16_t *x, int64_t ldx, int m, int k, int kbp,
                                                    const int *shift, uint32_t *frag, int bar, int tid) {
    act_rows_frags_inplace_body<NC>(x, ldx, m, k, kbp, shift, frag, bar, tid);
}

}  // namespace dev
}  // namespace bfp
