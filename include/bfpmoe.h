/*
 * bfpmoe.h — C-ABI of the GB300 block-floating-point MoE decode library.
 *
 * Operation sources on the block_floating_point pages ("P1" Qwen3.6-35B-A3B
 * TT-Mixed-BFP4-BFP8-P150 card, "P3" qwen3.6-a3b-blackhole tt-kernel bundle,
 * "P4" Qwen3.8-27B s27v6 card, "P5" Qwen3.8-27B gptq-ctx2 card):
 *   BFP4 experts, BFP8 dense projections and LM head, bf16 router and norms
 *     (P1, "Precision as served");
 *   16-value blocks (P5, "What changed in this release");
 *   round-to-nearest conversion (P1, "Verification", checkpoint bullet);
 *   MoE decode through device top-k routing and batched expert streams, one
 *     gate/up + down expert program for several rows (P1, "Fused decode kernels");
 *   256 experts, top-8 plus a shared expert (P3, opening paragraph);
 *   several users as the rows of one pass that streams every weight once
 *     (P4, "Multi-user decode");
 *   the greedy argmax over the LM head's logits (P1, "Fused decode kernels");
 *   error-compensated (GPTQ-style) BFP4 weights (P5, "What changed in this
 *     release");
 *   the KV cache in BFP8, or K BFP8 with Hadamard-rotated BFP4 V (P3,
 *     QWEN36_KV_DTYPE row; P4, "Changes in s27").
 *
 * Entry points: packing (bfp_packed_size, bfp_encode, bfp_encode_gate_up,
 * bfp_gptq_factor, bfp_encode_gptq, bfp_encode_gate_up_gptq, bfp_read_fields,
 * bfp_decode_host, bfp_unpack_device); the dense projection (bfp_linear,
 * bfp_linear_greedy); the MoE layer and the decode stack (moe_decode_layer,
 * moe_decode_layer_static, moe_stack_decode, moe_stack_decode_greedy); the
 * greedy token (bfp_greedy_tokens); the KV cache and
 * decode attention (bfp_kv_cache_size, bfp_kv_append, bfp_attn_decode; on
 * host copies bfp_kv_encode_host and bfp_kv_read_fields); workspace sizes,
 * status and launch settings.
 *
 * Conventions for every function:
 *   - returns an int status: BFP_OK (0) or a negative BFP_E* code; never
 *     throws, never exits; bfp_last_error() gives a message (thread-local);
 *   - the caller owns and allocates every buffer (host or device); the
 *     library allocates no device memory while it runs (its one built-in
 *     array, see moe_decode_layer_static, comes with the loaded module);
 *   - device work is enqueued on the caller's stream and is asynchronous;
 *     only bfp_workspace_status() synchronises (the stream it is given);
 *   - device pointers must be 16-byte aligned (BFP_EALIGN otherwise);
 *   - invalid shapes give BFP_ESHAPE, null/inconsistent arguments BFP_EINVAL,
 *     CUDA launch errors BFP_ECUDA (with the CUDA message in bfp_last_error).
 *
 * BFP value of a code (sign bit s above an mb-bit magnitude m, mb = 3 for
 * BFP4 and 7 for BFP8) under its block's exponent byte E:
 *     v = (-1)^s * m * 2^(E - 127 - (mb - 1)).
 * E is the largest fp32 exponent field in the block (0 for an all-zero
 * block); m is round-to-nearest-even, saturating at 2^mb - 1; zero, -0 and
 * fp32 subnormals encode as +0; NaN/Inf are rejected (BFP_ENONFINITE).
 *
 * Packed layout of a matrix W [n x k] (k % 16 == 0), "tile-record" layout:
 *   16 rows form a row group (NG = ceil(n/16)); along k, CB blocks of 16
 *   values form a chunk (CB = 4 for BFP4, 2 for BFP8; KC = ceil(k/16/CB)).
 *   The buffer is NG*KC records, record (rg, c) at byte (rg*KC + c)*REC,
 *   REC = 576 (BFP4) or 544 (BFP8). A record is
 *     bytes [0, 512):   codes, 16 bytes per lane l = 4*g + t (g = 0..7, t = 0..3)
 *     bytes [512, REC): exponents, byte 512 + (g*CB + b)*2 + h = E of row
 *                       16*rg + g + 8*h, block CB*c + b.
 *   Lane l's 16 bytes are 4 little-endian 32-bit words holding the codes of
 *   rows g and g+8 at the columns {2t, 2t+1, 2t+8, 2t+9} of each block:
 *     BFP4: word b covers block CB*c + b; "pair" p = 0..3 is
 *           (row g, cols 2t|2t+1), (row g+8, 2t|2t+1), (row g, 2t+8|2t+9),
 *           (row g+8, 2t+8|2t+9). The first value of pair p keeps its
 *           magnitude in bits 4p..4p+2 and its sign in bit (15+4p) mod 32;
 *           the second value its magnitude in bits (16+4p..18+4p) mod 32 and
 *           its sign in bit (31+4p) mod 32.
 *     BFP8: words 2b and 2b+1 cover block CB*c + b; word 2b holds pairs
 *           (row g, 2t|2t+1) and (row g+8, 2t|2t+1), word 2b+1 holds
 *           (row g, 2t+8|2t+9) and (row g+8, 2t+8|2t+9); pair q = 0, 1 of a
 *           word keeps its first magnitude in bits 8q..8q+6, sign in bit
 *           (15+8q) mod 32, second magnitude in bits (16+8q..22+8q) mod 32,
 *           sign in bit (31+8q) mod 32.
 *   Rows >= n and blocks >= k/16 are zero (code 0, exponent 0). Every byte
 *   carries information: 0.5625 (BFP4) / 1.0625 (BFP8) bytes per value when
 *   n % 16 == 0 and k % (16*CB) == 0. A warp streams 512 contiguous code
 *   bytes per record, and a rotation plus one mask of a word yields two
 *   fp16 lanes (sign << 15 | magnitude), ready for a tensor-core fragment.
 */
#ifndef BFPMOE_H
#define BFPMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers; NULL is the legacy default stream. */
typedef struct CUstream_st *bfp_stream_t;

enum {
    BFP_OK = 0,
    BFP_EINVAL = -1,     /* null pointer, bad enum, inconsistent sizes */
    BFP_ESHAPE = -2,     /* shape outside the supported range */
    BFP_EALIGN = -3,     /* pointer or stride not 16-byte aligned */
    BFP_ENONFINITE = -4, /* NaN or Inf given to the encoder */
    BFP_EWORKSPACE = -5, /* workspace too small or null */
    BFP_ECUDA = -6,      /* CUDA error (launch, attribute, device query) */
    BFP_ETIMEOUT = -7    /* a device-side wait ran out; reported by bfp_workspace_status */
};

enum { BFP_FMT_BFP4 = 4, BFP_FMT_BFP8 = 8 };

/* A packed BFP matrix (host or device memory, as each function states). */
typedef struct {
    int32_t fmt;      /* BFP_FMT_BFP4 or BFP_FMT_BFP8 */
    int32_t reserved; /* must be 0 */
    int64_t n, k;     /* logical rows and columns; k % 16 == 0 */
    const void *data; /* packed tile-record layout (above), 16-byte aligned */
    int64_t bytes;    /* size of data; must equal bfp_packed_size(fmt, n, k) */
} bfp_matrix;

/* Packed size in bytes of an [n x k] matrix (layout above). n >= 1, k >= 16, k % 16 == 0. */
int bfp_packed_size(int fmt, int64_t n, int64_t k, int64_t *bytes);

/*
 * Host packer. Encodes a row-major fp32 matrix w [n x k] (host memory) into
 * out (host memory, out_bytes >= bfp_packed_size). Round to nearest, ties to
 * even, 16-value blocks along k (P1 "Verification": CPU round-to-nearest
 * conversion; P5: 16-value blocks). nthreads <= 0 picks the host core count.
 * Returns BFP_ENONFINITE (and writes nothing useful) if w holds NaN/Inf.
 */
int bfp_encode(int fmt, const float *w, int64_t n, int64_t k, void *out, int64_t out_bytes, int nthreads);

/*
 * Host packer for one expert's gate and up projections, both [ffn x hidden]
 * row-major fp32 (host). Produces the packed [2*ffn x hidden] matrix whose
 * row group 2i holds gate rows 16i..16i+15 and row group 2i+1 holds up rows
 * 16i..16i+15, so that one contiguous span carries both halves of an
 * f-tile (P1 "Fused decode kernels": one gate/up + down expert program).
 * ffn % 16 == 0.
 */
int bfp_encode_gate_up(int fmt, const float *gate, const float *up, int64_t ffn, int64_t hidden, void *out,
                       int64_t out_bytes, int nthreads);

/*
 * Error-compensated (GPTQ-style) encoding, host only (P5 "What changed in this
 * release": BFP4 weights from a GPTQ variant for block floating point, error
 * compensated inside the 16-value blocks, every value exactly representable so
 * that plain conversion reproduces it; GPTQ: Frantar et al. 2022).
 *
 * bfp_gptq_factor: from calibration inputs x [t x k] (host fp32, row-major: t
 * samples of the k inputs a matrix multiplies) forms
 *     H = x^T x / t + damp * mean(diag(x^T x / t)) * I      (fp64)
 * and writes u [k x k] (host fp64, row-major, zero below the diagonal), the
 * upper-triangular factor with H^-1 = u^T u. damp > 0 (0.01 is usual).
 * BFP_EINVAL if x is all zero or H is not positive definite, BFP_ENONFINITE
 * for NaN/Inf in x. k <= 65536.
 *
 * bfp_encode_gptq: like bfp_encode (same packed output, same shapes), but each
 * row's columns are quantised left to right and each rounding error e_j =
 * (v_j - q_j) / u[j][j] is taken off the later columns, v_l -= e_j * u[j][l],
 * in fp64. A block's exponent comes from its compensated values when its first
 * column is reached; values round to nearest (ties to even) on that grid and
 * saturate; a block whose magnitudes all fit one bit less is then stored with
 * its exponent lowered, so bfp_encode of the decoded matrix gives the same
 * bytes. With a diagonal H the result is bfp_encode's. u: a factor for this
 * k (from bfp_gptq_factor). BFP_ENONFINITE for NaN/Inf in w or a compensated
 * value beyond the fp32 range.
 *
 * bfp_encode_gate_up_gptq: bfp_encode_gate_up's interleaved layout, each half
 * encoded as bfp_encode_gptq with the same u (gate and up see the same input).
 */
int bfp_gptq_factor(const float *x, int64_t t, int64_t k, double damp, double *u, int nthreads);
int bfp_encode_gptq(int fmt, const float *w, int64_t n, int64_t k, const double *u, void *out, int64_t out_bytes,
                    int nthreads);
int bfp_encode_gate_up_gptq(int fmt, const float *gate, const float *up, int64_t ffn, int64_t hidden, const double *u,
                            void *out, int64_t out_bytes, int nthreads);

/*
 * Host reader of a packed matrix (w->data in host memory): the logical
 * fields, exps [n x k/16] and codes [n x k] (one code per byte, sign << mb |
 * magnitude). Test aid for bit-exact comparisons.
 */
int bfp_read_fields(const bfp_matrix *w, uint8_t *exps, uint8_t *codes);

/* Host decode of a packed matrix (host memory) to row-major fp32 [n x k]; exact. */
int bfp_decode_host(const bfp_matrix *w, float *out);

/*
 * Device decode of a packed matrix (device memory) to row-major fp32
 * [n x k] (device memory), through the same fragment unpack and tensor-core
 * instruction the kernels use (each block multiplied by unit columns).
 * Test aid for the bit-exact unpack check.
 */
int bfp_unpack_device(const bfp_matrix *w, float *out, bfp_stream_t stream);

/*
 * Workspace for bfp_linear with m rows: *bytes of device memory that must be
 * zeroed once (bfp_workspace_init) before first use; every successful call
 * leaves it zeroed again. One workspace may serve calls in stream order only.
 */
int bfp_linear_workspace_size(const bfp_matrix *w, int m, size_t *bytes);

/*
 * Dense BFP decode projection (P1 "Precision as served": dense projections and
 * LM head in BFP8; P4 "Multi-user decode": all rows in one weight pass; P4
 * "What changed in this release (s27v6)": up to 32 rows in one tile row):
 *     y[r][o] = sum_j x[r][j] * W[o][j],   r < m, o < n,
 * x bf16 [m x k] (device, row stride ldx elements, ldx % 8 == 0), fp32
 * accumulation. y (nullable) receives fp32 [m x n], y_bf16 (nullable) the
 * round-to-nearest-even bf16 of the same fp32 values; both row stride ldy
 * elements. At least one output must be given. 1 <= m <= 32 (every weight
 * is read from HBM once for all m rows); m > 16 needs k <= 2048
 * (BFP_ESHAPE otherwise). W in device memory. ws: bfp_linear_workspace_size
 * bytes (device).
 */
int bfp_linear(const bfp_matrix *w, const uint16_t *x, int m, int64_t ldx, float *y, uint16_t *y_bf16, int64_t ldy,
               void *ws, size_t ws_bytes, bfp_stream_t stream);

/*
 * bfp_linear with the greedy next token folded into its epilogue (P1 "Fused
 * decode kernels": the greedy arg max taken on the LM head's tiles, without
 * writing out and re-reading the vocabulary-wide logits): tokens[r] (int32,
 * device, 4-byte aligned) = the index o of the largest y[r][o], ties to the
 * lower index, -0 equal to +0, NaN never chosen (a row with nothing else gives
 * 0): the same rule as bfp_greedy_tokens, on the kernel's own fp32 outputs.
 * y (nullable) receives those fp32 outputs as bfp_linear does; with y null
 * no output row is written at all. One launch: every CTA reduces its outputs
 * to one key per row and the last CTA to finish reduces the CTAs' keys (a
 * counter in ws, left at zero by every successful call). m, x, ws as for
 * bfp_linear.
 */
int bfp_linear_greedy(const bfp_matrix *w, const uint16_t *x, int m, int64_t ldx, float *y, int64_t ldy,
                      int32_t *tokens, void *ws, size_t ws_bytes, bfp_stream_t stream);

/*
 * One MoE decode layer's weights (all device memory).
 * Shapes: hidden % 16 == 0, ffn % 16 == 0, shared_ffn % 16 == 0,
 * 1 <= top_k <= 8, top_k <= n_experts <= 256.
 */
typedef struct {
    int32_t hidden, n_experts, ffn, top_k, shared_ffn;
    int32_t expert_fmt;            /* BFP_FMT_BFP4 (as served) or BFP_FMT_BFP8 */
    const uint16_t *router;        /* [n_experts x hidden] bf16, row-major */
    const float *router_bias;      /* nullable [n_experts] fp32, added to the logits before softmax and top-k */
    const uint16_t *shared_gate;   /* [hidden] bf16: the shared expert is scaled by sigmoid(shared_gate . x) */
    const void *experts_gate_up;   /* n_experts packed [2*ffn x hidden] matrices (bfp_encode_gate_up) */
    const void *experts_down;      /* n_experts packed [hidden x ffn] matrices (bfp_encode) */
    int64_t gate_up_stride;        /* bytes between consecutive experts' gate/up; >= packed size, % 16 == 0 */
    int64_t down_stride;           /* bytes between consecutive experts' down; >= packed size, % 16 == 0 */
    const void *shared_gate_up;    /* packed [2*shared_ffn x hidden] */
    const void *shared_down;       /* packed [hidden x shared_ffn] */
} bfp_moe_layer;

/*
 * Device workspace for moe_decode_layer / moe_stack_decode with m rows: zeroed
 * once (bfp_workspace_init) before first use; a successful call leaves it
 * ready for the next call with any m up to the size it was made for. After a
 * device-side error (BFP_ETIMEOUT) it must be initialised again. Calls that
 * share a workspace run in stream order.
 */
int moe_workspace_size(const bfp_moe_layer *layer, int m, size_t *bytes);

/* Zeroes a workspace (any of this library's) on the stream; also clears its status word. */
int bfp_workspace_init(void *ws, size_t ws_bytes, bfp_stream_t stream);

/*
 * One MoE decode layer for m rows (1..16) of bf16 input x [m x hidden]
 * (device, row-major, contiguous). Per row r:
 *     l = router . x_r (+ router_bias)   fp32 logits
 *     p = softmax(l); S = the top_k largest l (ties: lower index), in
 *     descending order; w_s = p_s / sum_S p
 *     y_r = sum_s w_s * D_s(silu(G_s x_r) * (U_s x_r)) + sigmoid(g . x_r) * shared(x_r)
 * with silu(a) = a * sigmoid(a), fp32 accumulation, fp32 intermediates.
 * The union of the experts the rows select is streamed from HBM once
 * (P1 "Fused decode kernels": device top-k routing and batched expert
 * streams). Outputs (device): y fp32 [m x hidden]; topk_idx int32 [m x top_k]
 * and topk_w fp32 [m x top_k] (both nullable) in slot order.
 * One persistent launch (a programmatic dependent launch unless
 * bfp_set_launch_mode asks for a cooperative one); its cross-block waits are
 * bounded and report BFP_ETIMEOUT through bfp_workspace_status.
 */
int moe_decode_layer(const bfp_moe_layer *layer, const uint16_t *x, int m, float *y, int32_t *topk_idx,
                     float *topk_w, void *ws, size_t ws_bytes, bfp_stream_t stream);

/*
 * moe_decode_layer without a workspace argument, for callers that cannot
 * allocate device memory: for example code embedded in a host runtime whose
 * device memory is all owned by that runtime's own allocator, or a
 * latency-critical path that must not call cudaMalloc because it can
 * synchronise the device. The block_floating_point pages have no counterpart;
 * this is a convenience of this library.
 *   - Computes what moe_decode_layer computes (same selection; outputs may
 *     differ in the last fp32 bits: with the smaller scratch the gate/up
 *     phase deals whole units to warps, which changes the order of some
 *     sums); x, y, topk_idx, topk_w as there (caller-owned device memory).
 *   - Scratch: one built-in device array of 2 MiB (2,097,152 bytes). It is
 *     reserved on a device when the library's MoE module first loads there
 *     (with CUDA's lazy module loading: the first MoE call on that device)
 *     and held until the process exits. A layer whose core state needs more
 *     (the workspace without its optional phase-1 hand-off area) is rejected
 *     with BFP_EWORKSPACE; the full-size layer (hidden 2048, 256 experts,
 *     ffn 512, top-8) needs 1,853,952 bytes on a 152-SM GPU (the one-row
 *     kernel's exchange area grows with the SM count).
 *   - The first call on a device looks up the array's device address and
 *     zeroes it, synchronously: make that first call before any stream
 *     capture. Each call then clears the array's counters (and, with one
 *     row, the one-row kernel's exchange area) on its stream.
 *   - Each device has its own copy of the array, and every call on that
 *     device shares it; it keeps the last call's contents. Calls on one
 *     device that can overlap on the GPU (on streams with no ordering
 *     between them) race on it and give wrong results: keep them in one
 *     stream order.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - A device-side wait that times out cannot be reported (there is no
 *     caller-visible workspace status word); use moe_decode_layer when the
 *     status matters.
 */
int moe_decode_layer_static(const bfp_moe_layer *layer, const uint16_t *x, int m, float *y, int32_t *topk_idx,
                            float *topk_w, bfp_stream_t stream);

/*
 * Decode stack: for each of n_layers layers,
 *     h <- bf16( h + MoE_l( bf16(RMSNorm(h)) ) ),  RMSNorm(h) = h / sqrt(mean(h^2) + 1e-6)
 * (unit weight, fp32), then logits = LMhead( bf16(RMSNorm(h)) ) in fp32
 * [m x lm_head->n] (P1 "Fused decode kernels": one-launch RMSNorm, packed LM
 * head). h: bf16 [m x hidden] device, updated in place. lm_head: BFP matrix
 * [vocab x hidden] in device memory. topk_idx (nullable, device int32): every
 * layer's selection in slot order, layer after layer, m * layers[l].top_k
 * entries for layer l (row-major [m x top_k]). ws: moe_stack_workspace_size
 * bytes. Launches: with m = 1 (and the one-row kernel, bfp_set_row_path) the
 * layers run up to 48 per launch when consecutive layers share a shape (P1
 * "Fused decode kernels": fewer, larger device programs): every CTA takes
 * the same share of each layer and the residual row passes from layer to
 * layer inside the launch; otherwise one launch per layer. Then one launch
 * for the LM head.
 */
int moe_stack_workspace_size(const bfp_moe_layer *layers, int n_layers, const bfp_matrix *lm_head, int m,
                             size_t *bytes);
int moe_stack_decode(const bfp_moe_layer *layers, int n_layers, const bfp_matrix *lm_head, uint16_t *h, int m,
                     float *logits, int32_t *topk_idx, void *ws, size_t ws_bytes, bfp_stream_t stream);

/*
 * moe_stack_decode whose LM head also gives the greedy next token of every row
 * (bfp_linear_greedy's rule, folded into the LM head's epilogue: P1 "Fused
 * decode kernels"): tokens int32 [m] (device). logits is nullable here: with
 * null logits the vocabulary-wide logits are never written. Same workspace.
 */
int moe_stack_decode_greedy(const bfp_moe_layer *layers, int n_layers, const bfp_matrix *lm_head, uint16_t *h, int m,
                            float *logits, int32_t *tokens, int32_t *topk_idx, void *ws, size_t ws_bytes,
                            bfp_stream_t stream);

/*
 * Greedy next token for m rows (1..16) of fp32 logits [m x n] (device, row
 * stride ldl >= n elements), the step after the LM head in greedy decoding
 * (P1 "Fused decode kernels": the greedy argmax over the logits, up to 16
 * rows): tokens[r] (int32, device) = the index of the largest logit of row r,
 * ties to the lower index, -0 equal to +0; NaN is never chosen, and a row
 * with no other value gives 0. 1 <= n <= 2^31 - 1. The result is exact (no
 * arithmetic, only comparisons). Two launches on the stream, dependent on
 * the previous kernel; ws: bfp_greedy_workspace_size bytes of device memory,
 * no initialisation needed. logits, tokens and ws 16-byte aligned.
 */
int bfp_greedy_workspace_size(int m, int64_t n, size_t *bytes);
int bfp_greedy_tokens(const float *logits, int m, int64_t n, int64_t ldl, int32_t *tokens, void *ws, size_t ws_bytes,
                      bfp_stream_t stream);

/*
 * BFP KV cache and decode attention (P3 QWEN36_KV_DTYPE row: the attention KV
 * cache as BFP8, re-read in full by every decode step; P4 "Changes in s27",
 * bfp8_v4r: K as BFP8, V Hadamard-rotated and stored as BFP4).
 * Codes follow the BFP rules of bfp_encode (16-value blocks along the head
 * dimension, one exponent byte each; code = sign << mb | magnitude). With
 * v_rotated = 1 a V row is stored as H v, H the Sylvester Hadamard matrix of
 * order head_dim (entries +-1), computed in fp32 by the fast transform
 * (stages 1, 2, 4, ...). Layout (device memory), NB = head_dim / 16:
 *   exponents: k_exps[(h * capacity + t) * NB + b] for KV head h, token slot t,
 *     block b (v_exps likewise);
 *   codes: tiles of 16 token slots x 16 values, tile (h, t / 16, b) at byte
 *     ((h * capacity / 16 + t / 16) * NB + b) * TB, TB = 256 (BFP8) or 128
 *     (BFP4). In a tile, token row r = t % 16 and column c (0..15):
 *     K, BFP8: the codes of columns 4j .. 4j+3 of row r form the 32-bit word
 *       at (4 (r % 8) + j) * 8 + (r / 8) * 4, holding P(c0, c1) | rotl(P(c2, c3), 8)
 *       with P(x, y) = p(x) | p(y) << 16 and p(code) = magnitude | sign << 15;
 *     K, BFP4: the same four codes form the 16-bit half at
 *       (4 (r % 8) + j) * 4 + (r / 8) * 2, column 4j + i in nibble i;
 *     V, BFP8: byte (4 (c % 8) + r / 4) * 8 + (c / 8) * 4 + r % 4;
 *     V, BFP4: byte (4 (c % 8) + r / 4) * 4 + r % 4, column c (< 8) in the low
 *       nibble and column c + 8 in the high one.
 *   This is the operand order of the tensor-core instruction the attention
 *   uses; every append writes whole words, halves or bytes of its own token.
 */
typedef struct {
    int32_t kv_heads, head_dim;        /* kv_heads 1..64; head_dim 64, 128 or 256 */
    int32_t k_fmt, v_fmt;              /* BFP_FMT_BFP8 or BFP_FMT_BFP4 each */
    int32_t v_rotated;                 /* 0 or 1 */
    int32_t reserved;                  /* must be 0 */
    int64_t capacity;                  /* token slots: a positive multiple of 64, at most 2^31 */
    void *k_codes, *k_exps, *v_codes, *v_exps; /* 16-byte aligned; sizes from bfp_kv_cache_size */
} bfp_kv_cache;

/* Bytes of one codes array and of one exponents array for a format and shape. */
int bfp_kv_cache_size(int fmt, int kv_heads, int head_dim, int64_t capacity, size_t *code_bytes, size_t *exp_bytes);

/*
 * Host encoder, the counterpart of bfp_kv_append for a cache whose four
 * arrays are in HOST memory (to pack K/V rows without a GPU, for example a
 * restored session, then copy the arrays to the device): k, v bf16
 * [n_new x kv_heads x head_dim] (host); the same codes, bytes and rotation
 * (fp32, same stage order) as bfp_kv_append. nthreads <= 0: the host's cores.
 * BFP_ENONFINITE for NaN/Inf.
 */
int bfp_kv_encode_host(const bfp_kv_cache *cache, const uint16_t *k, const uint16_t *v, int64_t pos, int n_new,
                       int nthreads);

/*
 * Host reader of a cache (test and inspection aid): with the cache's four
 * arrays in HOST memory (copies of the device arrays), writes the logical
 * fields of tokens t0 .. t0 + n - 1 of K (which = 0) or V (which = 1):
 * exps [kv_heads x n x head_dim/16] and codes [kv_heads x n x head_dim], one
 * code per byte (sign << mb | magnitude), in the stored (rotated) basis.
 */
int bfp_kv_read_fields(const bfp_kv_cache *cache, int which, int64_t t0, int64_t n, uint8_t *exps, uint8_t *codes);

/*
 * Encodes n_new tokens into slots pos .. pos + n_new - 1: k and v are bf16
 * [n_new x kv_heads x head_dim] (device, contiguous, 16-byte aligned). V is
 * rotated first when the cache says so. One launch on the stream; finite
 * inputs assumed (NaN/Inf give unspecified codes).
 */
int bfp_kv_append(const bfp_kv_cache *cache, const uint16_t *k, const uint16_t *v, int64_t pos, int n_new,
                  bfp_stream_t stream);

/*
 * Decode attention of one query token over the first n_ctx cached tokens
 * (1 <= n_ctx <= capacity): for query head j (kv head j / (q_heads / kv_heads),
 * q_heads / kv_heads in 1..8)
 *     s_t = scale * q_j . k_t,  p = softmax(s),  out_j = sum_t p_t v_t
 * (for a rotated cache out_j = H (sum_t p_t v'_t) / head_dim), fp32
 * arithmetic. q: bf16 [q_heads x head_dim]; out: fp32 [q_heads x head_dim]
 * (device). Two launches on the stream; ws: bfp_attn_workspace_size bytes of
 * device memory whose status word (first 4 bytes) must be zero
 * (bfp_workspace_init); a bounded wait that runs out sets BFP_ETIMEOUT there.
 */
int bfp_attn_workspace_size(const bfp_kv_cache *cache, int q_heads, int64_t n_ctx, size_t *bytes);
int bfp_attn_decode(const bfp_kv_cache *cache, const uint16_t *q, int q_heads, int64_t n_ctx, float scale, float *out,
                    void *ws, size_t ws_bytes, bfp_stream_t stream);

/*
 * Synchronises the stream and reads the workspace's status word: *status =
 * BFP_OK or the first device-side error (BFP_ETIMEOUT). The word stays set
 * until bfp_workspace_init.
 */
int bfp_workspace_status(const void *ws, int *status, bfp_stream_t stream);

/*
 * Test hook for the bounded waits: sets the iteration limit of every
 * cross-block wait in later launches from this thread (0 = the default
 * limit, about a second). A limit of 1 makes waits that are not already
 * satisfied give up at once and report BFP_ETIMEOUT.
 */
int bfp_set_wait_limit(int64_t iterations);

/*
 * How the MoE layer kernel (one CTA on every SM, whose CTAs wait on each
 * other) is launched, process-wide:
 *   BFP_LAUNCH_DEPENDENT (default): a programmatic dependent launch on the
 *     stream; the kernel's CTAs take the SMs as the previous kernel's CTAs
 *     leave and wait for that kernel to finish before touching memory, so
 *     back-to-back launches overlap their start-up. The waits between CTAs
 *     assume the layer has the GPU to itself (nothing else holding SMs); if
 *     not, they run out and report BFP_ETIMEOUT rather than hang.
 *   BFP_LAUNCH_COOPERATIVE: a cooperative launch, which the driver starts
 *     only when every CTA fits; for GPUs shared with other work.
 * The dense projection (no waits between CTAs) is always a dependent launch.
 */
enum { BFP_LAUNCH_DEPENDENT = 0, BFP_LAUNCH_COOPERATIVE = 1 };
int bfp_set_launch_mode(int mode);

/*
 * Which kernel runs a one-row MoE layer (moe_decode_layer, moe_decode_layer_static
 * and each layer of moe_stack_decode with m = 1), process-wide: 1 (default) the
 * one-row kernel, built for the shortest dependent chain of single-sequence
 * decode (every CTA's share fixed at launch, all of it requested at once, each
 * CTA summing whole output row groups itself); 0 the general kernel used for
 * m > 1. Both compute the same layer; layers whose shape does not fit the
 * one-row kernel's shared-memory plan use the general kernel either way. A
 * measurement and test hook. BFP_EINVAL for other values.
 */
int bfp_set_row_path(int enabled);

/*
 * Which kernel runs bfp_linear (not the greedy variant, which keeps the
 * mma.sync kernel), process-wide: 0 (default) and 1 the mma.sync kernel; 2
 * the tcgen05 kernel wherever it fits (k a multiple of 128, m <= 32, half of
 * each activation row in shared memory as fp16: k <= 2048 at 32 rows), the
 * mma.sync kernel otherwise. The tcgen05 kernel (P4, "What changed in this
 * release": up to 32 rows in one tile row) folds each block's exponent into
 * its fp16 operand relative to the largest exponent of the row's 128 inputs of
 * a chunk (exact for blocks within 2^15 of it; within 2^-16 of that chunk's
 * largest value otherwise) and accumulates in tensor memory; on GB300 it is
 * slower than the mma.sync kernel at every row count measured (1 to 32), so
 * it is not the default. A measurement and test hook. BFP_EINVAL for other
 * values.
 */
int bfp_set_linear_path(int mode);

/* Message for the last non-OK status returned on this thread. */
const char *bfp_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* BFPMOE_H */
