// Error-compensated (GPTQ-style) BFP encoding on the host.
//
// The Qwen3.8-27B gptq-ctx2 card ("What changed in this release") stores its
// BFP4 matrices as computed by a GPTQ variant for block floating point: error
// compensation inside the 16-value blocks, every value exactly representable so
// that the plain conversion reproduces it bit for bit. GPTQ is the published
// method of Frantar et al. (2022): with H the Hessian X^T X of the layer's
// calibration inputs X, the columns of W are quantised one at a time and each
// rounding error is moved onto the columns not yet quantised, through the
// upper Cholesky factor U of H^-1 (H^-1 = U^T U).
//
// Readings (the card gives no more): H = X^T X / t + damp * mean(diag) * I;
// columns in their natural order; a block's exponent comes from its current,
// already compensated values when its first column is reached (the largest
// fp32-style exponent field, values below 2^-126 counting as zero); values are
// rounded on that grid to nearest, ties to even, saturating; after its 16
// columns the block is put in canonical form (exponent lowered while every
// magnitude fits one bit less), which is what plain conversion gives for the
// same values. All arithmetic is fp64, each product and sum rounded on its own
// (this file is compiled without floating-point contraction).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "bfp_internal.h"
#include "bfp_pack.h"

namespace bfp {

namespace {

// fp32-style biased exponent field of an fp64 value: floor(log2|v|) + 127, 0 below 2^-126.
inline int exp_field(double v) {
    const double a = std::fabs(v);
    if (!(a >= 0x1p-126)) return 0;
    int p;
    std::frexp(a, &p);
    return p + 126;
}

// GPTQ over one row: v (the row's k values, overwritten) -> exps[k/16], codes[k].
// Returns false if a compensated value leaves the fp32 exponent range.
bool gptq_row(double *v, int64_t k, const double *u, int mb, uint8_t *exps, uint8_t *codes) {
    const int top = (1 << mb) - 1;
    int mag[16];
    for (int64_t b = 0; b < k / 16; ++b) {
        const int64_t j0 = 16 * b;
        int E = 0;
        for (int i = 0; i < 16; ++i) E = std::max(E, exp_field(v[j0 + i]));
        if (E >= 255) return false;
        const int s = E - 127 - (mb - 1);
        for (int i = 0; i < 16; ++i) {
            const int64_t j = j0 + i;
            const double x = v[j];
            int m = 0;
            double q = 0.0;
            if (E != 0 && exp_field(x) != 0) {
                m = (int)std::min<double>(std::nearbyint(std::ldexp(std::fabs(x), -s)), (double)top);
                if (m > 0) q = std::copysign(std::ldexp((double)m, s), x);
            }
            mag[i] = m;
            codes[j] = (uint8_t)(((m > 0 && x < 0) ? (1 << mb) : 0) | m);
            const double *ur = u + j * k;
            const double err = (x - q) / ur[j];
            for (int64_t l = j + 1; l < k; ++l) {
                const double d = err * ur[l];
                v[l] = v[l] - d;
            }
        }
        int mx = 0;
        for (int i = 0; i < 16; ++i) mx = std::max(mx, mag[i]);
        if (mx == 0) {
            E = 0;
        } else {
            int sh = 0;
            while (E - sh > 1 && (mx << sh) < (1 << (mb - 1))) ++sh;
            if (sh) {
                E -= sh;
                for (int i = 0; i < 16; ++i) codes[j0 + i] = (uint8_t)((codes[j0 + i] & (1 << mb)) | (mag[i] << sh));
            }
        }
        exps[b] = (uint8_t)E;
    }
    return true;
}

// Rows [16*rg, 16*rg+16) of a row-major fp32 source through gptq_row into group fields.
bool gptq_group(const Geometry &g, const float *w, int64_t rg, const double *u, GroupFields *f) {
    const int64_t kbp = g.kc * g.cb;
    f->codes.assign((size_t)16 * kbp * 16, 0);
    f->exps.assign((size_t)16 * kbp, 0);
    std::vector<double> v((size_t)g.k);
    for (int r = 0; r < 16; ++r) {
        const int64_t row = rg * 16 + r;
        if (row >= g.n) break;
        for (int64_t j = 0; j < g.k; ++j) {
            const float x = w[row * g.k + j];
            if (!std::isfinite(x)) return false;
            v[(size_t)j] = x;
        }
        if (!gptq_row(v.data(), g.k, u, g.mb, &f->exps[(size_t)r * kbp], &f->codes[(size_t)r * kbp * 16]))
            return false;
    }
    return true;
}

bool factor_ok(const double *u, int64_t k) {
    for (int64_t j = 0; j < k; ++j)
        if (!(u[j * k + j] > 0.0) || !std::isfinite(u[j * k + j])) return false;
    return true;
}

}  // namespace

}  // namespace bfp

using namespace bfp;

extern "C" {

int bfp_gptq_factor(const float *x, int64_t t, int64_t k, double damp, double *u, int nthreads) {
    if (!x || !u) return fail(BFP_EINVAL, "null pointer");
    if (t < 1 || k < 1 || k > (int64_t(1) << 16)) return fail(BFP_ESHAPE, "need t >= 1 and 1 <= k <= 65536");
    if (!(damp > 0.0) || !std::isfinite(damp)) return fail(BFP_EINVAL, "damp must be positive");
    const size_t kk = (size_t)k;
    const int64_t k4 = (k + 3) / 4 * 4;
    // X^T (k rows of t samples, zero rows up to a multiple of 4) in fp64, so that every entry of H is
    // one contiguous dot product
    std::vector<double> xt((size_t)k4 * (size_t)t, 0.0);
    for (int64_t s = 0; s < t; ++s)
        for (int64_t a = 0; a < k; ++a) {
            const float v = x[s * k + a];
            if (!std::isfinite(v)) return fail(BFP_ENONFINITE, "calibration inputs hold NaN or Inf");
            xt[(size_t)a * t + s] = v;
        }
    // H = X^T X / t: 4 x 4 tiles of the upper triangle, each entry summed over the samples in order
    std::vector<double> h(kk * kk);
    parallel_groups(k4 / 4, nthreads, [&](int64_t ta) {
        const int64_t a0 = 4 * ta;
        for (int64_t b0 = a0; b0 < k4; b0 += 4) {
            double acc[4][4] = {};
            const double *xa[4], *xb[4];
            for (int i = 0; i < 4; ++i) {
                xa[i] = &xt[(size_t)(a0 + i) * t];
                xb[i] = &xt[(size_t)(b0 + i) * t];
            }
            for (int64_t s = 0; s < t; ++s) {
                const double va[4] = {xa[0][s], xa[1][s], xa[2][s], xa[3][s]};
                const double vb[4] = {xb[0][s], xb[1][s], xb[2][s], xb[3][s]};
                for (int i = 0; i < 4; ++i)
                    for (int j = 0; j < 4; ++j) acc[i][j] = acc[i][j] + va[i] * vb[j];
            }
            for (int i = 0; i < 4; ++i)
                for (int j = 0; j < 4; ++j) {
                    const int64_t a = a0 + i, b = b0 + j;
                    if (a < k && b < k && b >= a) h[(size_t)a * kk + b] = acc[i][j] / (double)t;
                }
        }
        return true;
    });
    for (int64_t a = 0; a < k; ++a)
        for (int64_t b = 0; b < a; ++b) h[(size_t)a * kk + b] = h[(size_t)b * kk + a];
    double mean = 0.0;
    for (int64_t a = 0; a < k; ++a) mean += h[(size_t)a * kk + a];
    mean /= (double)k;
    if (!(mean > 0.0)) return fail(BFP_EINVAL, "calibration inputs are all zero");
    const double lam = damp * mean;
    for (int64_t a = 0; a < k; ++a) h[(size_t)a * kk + a] += lam;
    // With J the order reversal, P = J H J = L L^T (lower Cholesky factor L), so H = R R^T with
    // R = J L J upper triangular, H^-1 = R^-T R^-1, and U = R^-1 = J L^-1 J is the upper factor with
    // H^-1 = U^T U. L: blocked right-looking factorisation of P in place (lower triangle).
    std::vector<double> pm(kk * kk);
    for (int64_t i = 0; i < k; ++i)
        for (int64_t j = 0; j <= i; ++j) pm[(size_t)i * kk + j] = h[(size_t)(k - 1 - i) * kk + (k - 1 - j)];
    auto P = [&](int64_t i, int64_t j) -> double & { return pm[(size_t)i * kk + j]; };
    constexpr int64_t kNb = 64;
    for (int64_t kb = 0; kb < k; kb += kNb) {
        const int64_t e = std::min(kb + kNb, k);
        for (int64_t j = kb; j < e; ++j) {  // the diagonal block
            double d = P(j, j);
            for (int64_t l = kb; l < j; ++l) d -= P(j, l) * P(j, l);
            if (!(d > 0.0)) return fail(BFP_EINVAL, "Hessian not positive definite (raise damp)");
            const double piv = std::sqrt(d);
            P(j, j) = piv;
            for (int64_t i = j + 1; i < e; ++i) {
                double acc = P(i, j);
                for (int64_t l = kb; l < j; ++l) acc -= P(i, l) * P(j, l);
                P(i, j) = acc / piv;
            }
        }
        if (e == k) break;
        // the panel below it, one row at a time
        parallel_groups(k - e, nthreads, [&](int64_t ii) {
            const int64_t i = e + ii;
            for (int64_t j = kb; j < e; ++j) {
                double acc = P(i, j);
                for (int64_t l = kb; l < j; ++l) acc -= P(i, l) * P(j, l);
                P(i, j) = acc / P(j, j);
            }
            return true;
        });
        // the trailing matrix, one row at a time
        parallel_groups(k - e, nthreads, [&](int64_t ii) {
            const int64_t i = e + ii;
            const double *pi = &pm[(size_t)i * kk + kb];
            for (int64_t j = e; j <= i; ++j) {
                const double *pj = &pm[(size_t)j * kk + kb];
                double acc = 0.0;
                for (int64_t l = 0; l < e - kb; ++l) acc = acc + pi[l] * pj[l];
                P(i, j) -= acc;
            }
            return true;
        });
    }
    // L^-1 column by column (forward substitution), written reversed into U
    std::memset(u, 0, kk * kk * sizeof(double));
    parallel_groups(k, nthreads, [&](int64_t c) {
        std::vector<double> col((size_t)(k - c));
        col[0] = 1.0 / P(c, c);
        for (int64_t i = c + 1; i < k; ++i) {
            const double *pi = &pm[(size_t)i * kk];
            double acc = 0.0;
            for (int64_t l = c; l < i; ++l) acc += pi[l] * col[(size_t)(l - c)];
            col[(size_t)(i - c)] = -acc / pi[i];
        }
        for (int64_t i = c; i < k; ++i) u[(size_t)(k - 1 - i) * kk + (k - 1 - c)] = col[(size_t)(i - c)];
        return true;
    });
    return BFP_OK;
}

int bfp_encode_gptq(int fmt, const float *w, int64_t n, int64_t k, const double *u, void *out, int64_t out_bytes,
                    int nthreads) {
    Geometry g;
    int rc = make_geometry(fmt, n, k, &g);
    if (rc) return rc;
    if (!w || !u || !out) return fail(BFP_EINVAL, "null pointer");
    if (out_bytes < g.bytes()) return fail(BFP_EINVAL, "out_bytes smaller than bfp_packed_size");
    if (!factor_ok(u, k)) return fail(BFP_EINVAL, "u must have a positive finite diagonal");
    uint8_t *dst = static_cast<uint8_t *>(out);
    bool good = parallel_groups(g.ng, nthreads, [&](int64_t rg) {
        GroupFields f;
        if (!gptq_group(g, w, rg, u, &f)) return false;
        for (int64_t c = 0; c < g.kc; ++c) write_record(g, f, c, dst + (rg * g.kc + c) * g.rec);
        return true;
    });
    if (!good) return fail(BFP_ENONFINITE, "input holds NaN or Inf, or a compensated value left the fp32 range");
    return BFP_OK;
}

int bfp_encode_gate_up_gptq(int fmt, const float *gate, const float *up, int64_t ffn, int64_t hidden, const double *u,
                            void *out, int64_t out_bytes, int nthreads) {
    if (ffn < 16 || ffn % 16 != 0) return fail(BFP_ESHAPE, "ffn must be a positive multiple of 16");
    Geometry g;
    int rc = make_geometry(fmt, 2 * ffn, hidden, &g);
    if (rc) return rc;
    if (!gate || !up || !u || !out) return fail(BFP_EINVAL, "null pointer");
    if (out_bytes < g.bytes()) return fail(BFP_EINVAL, "out_bytes smaller than bfp_packed_size");
    if (!factor_ok(u, hidden)) return fail(BFP_EINVAL, "u must have a positive finite diagonal");
    Geometry half;
    make_geometry(fmt, ffn, hidden, &half);
    uint8_t *dst = static_cast<uint8_t *>(out);
    bool good = parallel_groups(g.ng, nthreads, [&](int64_t rg) {
        GroupFields f;
        if (!gptq_group(half, (rg & 1) ? up : gate, rg >> 1, u, &f)) return false;
        for (int64_t c = 0; c < g.kc; ++c) write_record(g, f, c, dst + (rg * g.kc + c) * g.rec);
        return true;
    });
    if (!good) return fail(BFP_ENONFINITE, "input holds NaN or Inf, or a compensated value left the fp32 range");
    return BFP_OK;
}

}  // extern "C"
