// Host half of the library: geometry, the BFP packer (round to nearest, ties
// to even, 16-value blocks), the field reader and host decode, error state.
//
// Format sources: 16-value blocks (Qwen3.8-27B gptq-ctx2 card, "What changed
// in this release"); CPU round-to-nearest conversion of the stored BFP
// tensors (Qwen3.6-35B-A3B card, "Verification"); one exponent byte per 16
// values (qwen3.6-a3b-blackhole page, QWEN36_KV_DTYPE row; Qwen3.8-27B s27v6
// card, "Changes in s27"). Bit rules as stated in include/bfpmoe.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "bfp_internal.h"
#include "bfp_pack.h"

namespace bfp {

namespace {
thread_local std::string g_last_error = "ok";
thread_local int64_t g_wait_limit = 0;
std::atomic<int> g_launch_mode{BFP_LAUNCH_DEPENDENT};
std::atomic<int> g_row_path{1};

inline uint32_t f32_to_u32(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
}

inline uint32_t rotl32(uint32_t v, int s) { s &= 31; return s ? (v << s) | (v >> (32 - s)) : v; }
inline uint32_t rotr32(uint32_t v, int s) { s &= 31; return s ? (v >> s) | (v << (32 - s)) : v; }

}  // namespace

// One 16-value block -> exponent byte + 16 codes. Returns false on NaN/Inf.
// E is the largest exponent field; a value with field e keeps its 24-bit
// significand shifted right by (24 - mb) + (E - e), rounded to nearest with
// ties to even, saturated to 2^mb - 1. Fields of 0 (zero, subnormal) give 0.
bool encode_block(const float *v, int mb, uint8_t *E_out, uint8_t codes[16]) {
    uint32_t u[16];
    int E = 0;
    for (int i = 0; i < 16; ++i) {
        u[i] = f32_to_u32(v[i]);
        int e = (int)((u[i] >> 23) & 0xFFu);
        if (e == 0xFF) return false;
        E = std::max(E, e);
    }
    *E_out = (uint8_t)E;
    const uint32_t top = (1u << mb) - 1u;
    for (int i = 0; i < 16; ++i) {
        int e = (int)((u[i] >> 23) & 0xFFu);
        uint32_t mag = 0;
        if (e != 0) {
            uint64_t sig = (uint64_t)((u[i] & 0x7FFFFFu) | 0x800000u);
            int sh = (24 - mb) + (E - e);
            if (sh < 40) {
                // round half to even: add (2^(sh-1) - 1) plus the kept lsb, then truncate
                uint64_t keep_lsb = (sig >> sh) & 1u;
                uint64_t bias = ((uint64_t)1 << (sh - 1)) - 1u + keep_lsb;
                mag = (uint32_t)((sig + bias) >> sh);
            }
            if (mag > top) mag = top;
        }
        uint32_t s = mag ? (u[i] >> 31) : 0u;
        codes[i] = (uint8_t)((s << mb) | mag);
    }
    return true;
}

namespace {

// fp16-lane pattern of one pair of codes: first value in bits 0-15, second in 16-31,
// each as (sign << 15 | magnitude).
inline uint32_t pair_pattern(uint8_t c0, uint8_t c1, int mb) {
    uint32_t m0 = c0 & ((1u << mb) - 1u), s0 = (c0 >> mb) & 1u;
    uint32_t m1 = c1 & ((1u << mb) - 1u), s1 = (c1 >> mb) & 1u;
    return (m0 | (s0 << 15)) | ((m1 | (s1 << 15)) << 16);
}

inline void pattern_codes(uint32_t p, int mb, uint8_t *c0, uint8_t *c1) {
    uint32_t mmask = (1u << mb) - 1u;
    *c0 = (uint8_t)(((p >> 15) & 1u) << mb | (p & mmask));
    *c1 = (uint8_t)(((p >> 31) & 1u) << mb | ((p >> 16) & mmask));
}

}  // namespace

// Write record (rg, c) from a row group's logical fields.
void write_record(const Geometry &g, const GroupFields &f, int64_t c, uint8_t *rec) {
    std::memset(rec, 0, (size_t)g.rec);
    const int64_t kbp = g.kc * g.cb;  // padded blocks per row
    uint32_t *words = reinterpret_cast<uint32_t *>(rec);
    for (int lane = 0; lane < 32; ++lane) {
        int gi = lane >> 2, t = lane & 3;
        for (int b = 0; b < g.cb; ++b) {
            int64_t blk = c * g.cb + b;
            auto code = [&](int row, int col) -> uint8_t { return f.codes[(size_t)row * kbp * 16 + blk * 16 + col]; };
            int r0 = gi, r1 = gi + 8;
            if (g.fmt == BFP_FMT_BFP4) {
                uint32_t w = 0;
                w |= rotl32(pair_pattern(code(r0, 2 * t), code(r0, 2 * t + 1), 3), 0);
                w |= rotl32(pair_pattern(code(r1, 2 * t), code(r1, 2 * t + 1), 3), 4);
                w |= rotl32(pair_pattern(code(r0, 2 * t + 8), code(r0, 2 * t + 9), 3), 8);
                w |= rotl32(pair_pattern(code(r1, 2 * t + 8), code(r1, 2 * t + 9), 3), 12);
                words[lane * 4 + b] = w;
            } else {
                uint32_t w0 = pair_pattern(code(r0, 2 * t), code(r0, 2 * t + 1), 7) |
                              rotl32(pair_pattern(code(r1, 2 * t), code(r1, 2 * t + 1), 7), 8);
                uint32_t w1 = pair_pattern(code(r0, 2 * t + 8), code(r0, 2 * t + 9), 7) |
                              rotl32(pair_pattern(code(r1, 2 * t + 8), code(r1, 2 * t + 9), 7), 8);
                words[lane * 4 + 2 * b] = w0;
                words[lane * 4 + 2 * b + 1] = w1;
            }
        }
    }
    for (int gi = 0; gi < 8; ++gi)
        for (int b = 0; b < g.cb; ++b)
            for (int h = 0; h < 2; ++h)
                rec[kRecCodeBytes + (gi * g.cb + b) * 2 + h] = f.exps[(size_t)(gi + 8 * h) * kbp + c * g.cb + b];
}

namespace {

// Read record (rg, c) back into a row group's logical fields.
void read_record(const Geometry &g, const uint8_t *rec, int64_t c, GroupFields *f) {
    const int64_t kbp = g.kc * g.cb;
    const uint32_t *words = reinterpret_cast<const uint32_t *>(rec);
    for (int lane = 0; lane < 32; ++lane) {
        int gi = lane >> 2, t = lane & 3;
        for (int b = 0; b < g.cb; ++b) {
            int64_t blk = c * g.cb + b;
            auto put = [&](int row, int col, uint8_t v) { f->codes[(size_t)row * kbp * 16 + blk * 16 + col] = v; };
            int r0 = gi, r1 = gi + 8;
            uint8_t a, bb;
            if (g.fmt == BFP_FMT_BFP4) {
                uint32_t w = words[lane * 4 + b];
                const uint32_t mask = 0x80078007u;
                pattern_codes(rotr32(w, 0) & mask, 3, &a, &bb); put(r0, 2 * t, a); put(r0, 2 * t + 1, bb);
                pattern_codes(rotr32(w, 4) & mask, 3, &a, &bb); put(r1, 2 * t, a); put(r1, 2 * t + 1, bb);
                pattern_codes(rotr32(w, 8) & mask, 3, &a, &bb); put(r0, 2 * t + 8, a); put(r0, 2 * t + 9, bb);
                pattern_codes(rotr32(w, 12) & mask, 3, &a, &bb); put(r1, 2 * t + 8, a); put(r1, 2 * t + 9, bb);
            } else {
                const uint32_t mask = 0x807F807Fu;
                uint32_t w0 = words[lane * 4 + 2 * b], w1 = words[lane * 4 + 2 * b + 1];
                pattern_codes(w0 & mask, 7, &a, &bb); put(r0, 2 * t, a); put(r0, 2 * t + 1, bb);
                pattern_codes(rotr32(w0, 8) & mask, 7, &a, &bb); put(r1, 2 * t, a); put(r1, 2 * t + 1, bb);
                pattern_codes(w1 & mask, 7, &a, &bb); put(r0, 2 * t + 8, a); put(r0, 2 * t + 9, bb);
                pattern_codes(rotr32(w1, 8) & mask, 7, &a, &bb); put(r1, 2 * t + 8, a); put(r1, 2 * t + 9, bb);
            }
        }
    }
    for (int gi = 0; gi < 8; ++gi)
        for (int b = 0; b < g.cb; ++b)
            for (int h = 0; h < 2; ++h)
                f->exps[(size_t)(gi + 8 * h) * kbp + c * g.cb + b] = rec[kRecCodeBytes + (gi * g.cb + b) * 2 + h];
}

// Encode rows [16*rg, 16*rg+16) of a row-major fp32 source into group fields.
bool encode_group(const Geometry &g, const float *w, int64_t rg, GroupFields *f) {
    const int64_t kbp = g.kc * g.cb;
    f->codes.assign((size_t)16 * kbp * 16, 0);
    f->exps.assign((size_t)16 * kbp, 0);
    for (int r = 0; r < 16; ++r) {
        int64_t row = rg * 16 + r;
        if (row >= g.n) break;
        for (int64_t b = 0; b < g.kb; ++b) {
            uint8_t E;
            if (!encode_block(w + row * g.k + b * 16, g.mb, &E, &f->codes[(size_t)r * kbp * 16 + b * 16])) return false;
            f->exps[(size_t)r * kbp + b] = E;
        }
    }
    return true;
}

}  // namespace

int resolve_threads(int nthreads, int64_t work) {
    if (nthreads <= 0) nthreads = (int)std::max(1u, std::thread::hardware_concurrency());
    nthreads = (int)std::min<int64_t>(nthreads, std::max<int64_t>(1, work));
    return std::min(nthreads, 256);
}

int fail(int code, const std::string &msg) {
    g_last_error = msg;
    return code;
}
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
int64_t wait_limit() { return g_wait_limit; }
int launch_mode() { return g_launch_mode.load(std::memory_order_relaxed); }
bool row_path() { return g_row_path.load(std::memory_order_relaxed) != 0; }

int make_geometry(int fmt, int64_t n, int64_t k, Geometry *g) {
    if (fmt != BFP_FMT_BFP4 && fmt != BFP_FMT_BFP8) return fail(BFP_EINVAL, "fmt must be BFP_FMT_BFP4 or BFP_FMT_BFP8");
    if (n < 1 || k < 16 || (k % 16) != 0) return fail(BFP_ESHAPE, "need n >= 1, k >= 16, k % 16 == 0");
    if (n > ((int64_t)1 << 40) || k > ((int64_t)1 << 30)) return fail(BFP_ESHAPE, "matrix too large");
    g->fmt = fmt;
    g->mb = fmt == BFP_FMT_BFP4 ? 3 : 7;
    g->n = n;
    g->k = k;
    g->ng = (n + 15) / 16;
    g->kb = k / 16;
    g->cb = fmt == BFP_FMT_BFP4 ? 4 : 2;
    g->kc = (g->kb + g->cb - 1) / g->cb;
    g->rec = kRecCodeBytes + 16 * g->cb;
    return BFP_OK;
}

int check_matrix(const bfp_matrix *w, Geometry *g, bool device_ptr) {
    if (!w) return fail(BFP_EINVAL, "null bfp_matrix");
    if (w->reserved != 0) return fail(BFP_EINVAL, "bfp_matrix.reserved must be 0");
    int rc = make_geometry(w->fmt, w->n, w->k, g);
    if (rc) return rc;
    if (!w->data) return fail(BFP_EINVAL, "bfp_matrix.data is null");
    if (w->bytes != g->bytes()) return fail(BFP_EINVAL, "bfp_matrix.bytes != bfp_packed_size(fmt, n, k)");
    if (device_ptr && !aligned16(w->data)) return fail(BFP_EALIGN, "bfp_matrix.data not 16-byte aligned");
    return BFP_OK;
}

}  // namespace bfp

using namespace bfp;

extern "C" {

int bfp_packed_size(int fmt, int64_t n, int64_t k, int64_t *bytes) {
    if (!bytes) return fail(BFP_EINVAL, "bytes is null");
    Geometry g;
    int rc = make_geometry(fmt, n, k, &g);
    if (rc) return rc;
    *bytes = g.bytes();
    return BFP_OK;
}

int bfp_encode(int fmt, const float *w, int64_t n, int64_t k, void *out, int64_t out_bytes, int nthreads) {
    Geometry g;
    int rc = make_geometry(fmt, n, k, &g);
    if (rc) return rc;
    if (!w || !out) return fail(BFP_EINVAL, "null pointer");
    if (out_bytes < g.bytes()) return fail(BFP_EINVAL, "out_bytes smaller than bfp_packed_size");
    uint8_t *dst = static_cast<uint8_t *>(out);
    bool good = parallel_groups(g.ng, nthreads, [&](int64_t rg) {
        GroupFields f;
        if (!encode_group(g, w, rg, &f)) return false;
        for (int64_t c = 0; c < g.kc; ++c) write_record(g, f, c, dst + (rg * g.kc + c) * g.rec);
        return true;
    });
    if (!good) return fail(BFP_ENONFINITE, "input holds NaN or Inf");
    return BFP_OK;
}

int bfp_encode_gate_up(int fmt, const float *gate, const float *up, int64_t ffn, int64_t hidden, void *out,
                       int64_t out_bytes, int nthreads) {
    if (ffn < 16 || ffn % 16 != 0) return fail(BFP_ESHAPE, "ffn must be a positive multiple of 16");
    Geometry g;
    int rc = make_geometry(fmt, 2 * ffn, hidden, &g);
    if (rc) return rc;
    if (!gate || !up || !out) return fail(BFP_EINVAL, "null pointer");
    if (out_bytes < g.bytes()) return fail(BFP_EINVAL, "out_bytes smaller than bfp_packed_size");
    Geometry half;
    make_geometry(fmt, ffn, hidden, &half);
    uint8_t *dst = static_cast<uint8_t *>(out);
    bool good = parallel_groups(g.ng, nthreads, [&](int64_t rg) {
        GroupFields f;
        const float *src = (rg & 1) ? up : gate;
        if (!encode_group(half, src, rg >> 1, &f)) return false;
        for (int64_t c = 0; c < g.kc; ++c) write_record(g, f, c, dst + (rg * g.kc + c) * g.rec);
        return true;
    });
    if (!good) return fail(BFP_ENONFINITE, "input holds NaN or Inf");
    return BFP_OK;
}

int bfp_read_fields(const bfp_matrix *w, uint8_t *exps, uint8_t *codes) {
    Geometry g;
    int rc = check_matrix(w, &g, false);
    if (rc) return rc;
    if (!exps || !codes) return fail(BFP_EINVAL, "null output");
    const uint8_t *src = static_cast<const uint8_t *>(w->data);
    const int64_t kbp = g.kc * g.cb;
    GroupFields f;
    f.codes.assign((size_t)16 * kbp * 16, 0);
    f.exps.assign((size_t)16 * kbp, 0);
    for (int64_t rg = 0; rg < g.ng; ++rg) {
        for (int64_t c = 0; c < g.kc; ++c) read_record(g, src + (rg * g.kc + c) * g.rec, c, &f);
        for (int r = 0; r < 16; ++r) {
            int64_t row = rg * 16 + r;
            if (row >= g.n) break;
            std::memcpy(codes + row * g.k, &f.codes[(size_t)r * kbp * 16], (size_t)g.k);
            std::memcpy(exps + row * g.kb, &f.exps[(size_t)r * kbp], (size_t)g.kb);
        }
    }
    return BFP_OK;
}

int bfp_decode_host(const bfp_matrix *w, float *out) {
    Geometry g;
    int rc = check_matrix(w, &g, false);
    if (rc) return rc;
    if (!out) return fail(BFP_EINVAL, "null output");
    std::vector<uint8_t> exps((size_t)(g.n * g.kb)), codes((size_t)(g.n * g.k));
    rc = bfp_read_fields(w, exps.data(), codes.data());
    if (rc) return rc;
    const uint32_t mmask = (1u << g.mb) - 1u;
    for (int64_t r = 0; r < g.n; ++r)
        for (int64_t j = 0; j < g.k; ++j) {
            uint8_t c = codes[(size_t)(r * g.k + j)];
            int E = exps[(size_t)(r * g.kb + j / 16)];
            double v = std::ldexp((double)(c & mmask), E - 127 - (g.mb - 1));
            out[r * g.k + j] = (float)((c >> g.mb) & 1u ? -v : v);
        }
    return BFP_OK;
}

int bfp_set_wait_limit(int64_t iterations) {
    if (iterations < 0) return fail(BFP_EINVAL, "negative wait limit");
    g_wait_limit = iterations;
    return BFP_OK;
}

int bfp_set_launch_mode(int mode) {
    if (mode != BFP_LAUNCH_DEPENDENT && mode != BFP_LAUNCH_COOPERATIVE) return fail(BFP_EINVAL, "unknown launch mode");
    g_launch_mode.store(mode, std::memory_order_relaxed);
    return BFP_OK;
}

int bfp_set_row_path(int enabled) {
    if (enabled != 0 && enabled != 1) return fail(BFP_EINVAL, "enabled must be 0 or 1");
    g_row_path.store(enabled, std::memory_order_relaxed);
    return BFP_OK;
}

const char *bfp_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
