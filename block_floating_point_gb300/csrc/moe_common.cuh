// Pieces shared by the two MoE layer kernels (moe_layer.cu: any number of rows
// up to 16; moe_row.cu: the one-row latency path): limits, the split of the
// router rows over CTAs, the logits' row stride, and the top-k key order.
#pragma once

#include <stdint.h>

#include "bfp_device.cuh"
#include "bfp_internal.h"

namespace bfp {

constexpr int kMaxRows = 16;
constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 256;

// First router row of CTA c when `rows` rows (the experts, then the shared-gate row) are split over ncta CTAs.
__host__ __device__ inline int router_row_start(int c, int rows, int ncta) { return (int)((int64_t)c * rows / ncta); }
// Row stride (floats) of the logits in the workspace: the E expert logits then the shared-gate logit,
// padded to whole 16-byte vectors.
__host__ __device__ inline int logit_stride(int E) { return (E + 1 + 3) & ~3; }

namespace dev {

// Ordered 32-bit key of a float: larger float <=> larger unsigned key.
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// Inverse of order_key.
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// Compare-exchange on (key, index) pairs: larger key first, lower index first among equal keys.
__device__ __forceinline__ void cmp_xchg(uint32_t &ka, int &qa, uint32_t &kb, int &qb) {
    const bool sw = kb > ka || (kb == ka && qb < qa);
    const uint32_t k0 = sw ? kb : ka, k1 = sw ? ka : kb;
    const int q0 = sw ? qb : qa, q1 = sw ? qa : qb;
    ka = k0;
    kb = k1;
    qa = q0;
    qb = q1;
}
// Sorts 8 (key, index) pairs in registers (Batcher's odd-even merge network, 19 comparators).
__device__ __forceinline__ void sort8_desc(uint32_t k[8], int q[8]) {
    constexpr int net[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6}, {5, 7}, {1, 2}, {5, 6},
                                {0, 4}, {1, 5}, {2, 6}, {3, 7}, {2, 4}, {3, 5}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
    for (int i = 0; i < 19; ++i) cmp_xchg(k[net[i][0]], q[net[i][0]], k[net[i][1]], q[net[i][1]]);
}

}  // namespace dev

// One-row layer path (moe_row.cu). Returns BFP_OK when it launched, a BFP_E* code on error, or
// kRowNotApplicable when the layer's shape does not fit the path (the caller then launches the
// general kernel). row_ws: the workspace's area for this path (row_ws_bytes bytes, 256-byte aligned,
// zero after bfp_workspace_init): an epoch word; one mailbox of router logits per CTA (every CTA
// writes its logits into every mailbox, so each CTA polls lines of its own); h of every slot; the residual
// row between layers of one launch. Values travel as (epoch, value) 64-bit words.
constexpr int kRowNotApplicable = 1;
constexpr int kRowMaxCta = 256;  // CTAs of the one-row kernel at most (mailboxes in the area)
__host__ __device__ inline int row_boxes(int sms) { return sms < kRowMaxCta ? sms : kRowMaxCta; }
__host__ __device__ inline size_t row_ws_logits_off() { return 256; }
__host__ __device__ inline size_t row_ws_h_off(int E, int boxes) {
    return 256 + (((size_t)boxes * logit_stride(E) * 8 + 255) / 256) * 256;
}
__host__ __device__ inline size_t row_ws_x_off(int E, int K, int Fmax, int boxes) {
    return row_ws_h_off(E, boxes) + (size_t)(K + 1) * Fmax * 8;
}
__host__ __device__ inline size_t row_ws_bytes(int E, int K, int Fmax, int H, int boxes) {
    return row_ws_x_off(E, K, Fmax, boxes) + (size_t)(H / 2) * 8;
}
// One launch for nl (1 .. 48) layers of one shape applied in order to one row: layer l + 1 takes layer l's
// residual row (norm: the stack's bf16(x + y) then RMSNorm); x the first layer's input, y / h_out the last
// layer's output, topk_idx / topk_w K entries per layer. kRowNotApplicable when the shapes differ or the
// path does not fit them.
int row_layers_launch(const bfp_moe_layer *layers, int nl, const uint16_t *x, int norm, float *y, uint16_t *h_out,
                      int32_t *topk_idx, float *topk_w, uint32_t *status, uint8_t *row_ws, int fmax,
                      cudaStream_t stream);

}  // namespace bfp
