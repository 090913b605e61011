// Host packer pieces shared by the plain and the error-compensated encoders.
#pragma once

#include <atomic>
#include <cstdint>
#include <thread>
#include <vector>

#include "bfp_internal.h"

namespace bfp {

// Logical fields of one row group: codes[16][kbp*16] and exps[16][kbp] (zero padded).
struct GroupFields {
    std::vector<uint8_t> codes, exps;
};

// One 16-value block -> exponent byte + 16 codes (round to nearest, ties to even, saturating; the
// rules of bfp_encode). Returns false on NaN/Inf.
bool encode_block(const float *v, int mb, uint8_t *E_out, uint8_t codes[16]);

// Write record (rg, c) of the packed layout from a row group's logical fields.
void write_record(const Geometry &g, const GroupFields &f, int64_t c, uint8_t *rec);

// Threads to use for `work` independent items (nthreads <= 0: the host's core count).
int resolve_threads(int nthreads, int64_t work);

// Run fn(i) for i in [0, n) over threads; fn returns false on failure, which stops the rest.
template <class F>
bool parallel_groups(int64_t n, int nthreads, F fn) {
    nthreads = resolve_threads(nthreads, n);
    std::atomic<int64_t> next{0};
    std::atomic<bool> good{true};
    auto worker = [&]() {
        for (;;) {
            int64_t i = next.fetch_add(1);
            if (i >= n || !good.load()) return;
            if (!fn(i)) good.store(false);
        }
    };
    std::vector<std::thread> pool;
    for (int t = 1; t < nthreads; ++t) pool.emplace_back(worker);
    worker();
    for (auto &t : pool) t.join();
    return good.load();
}

}  // namespace bfp
