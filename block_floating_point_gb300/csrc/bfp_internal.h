// Internal declarations shared by the library's host and device translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include "../../include/bfpmoe.h"

namespace bfp {

// Tile-record geometry of a packed matrix (see include/bfpmoe.h, "Packed layout").
struct Geometry {
    int fmt = 0;
    int mb = 0;          // magnitude bits: 3 (BFP4) or 7 (BFP8)
    int64_t n = 0, k = 0;
    int64_t ng = 0;      // row groups of 16
    int64_t kb = 0;      // blocks of 16 along k
    int cb = 0;          // blocks per chunk: 4 (BFP4) or 2 (BFP8)
    int64_t kc = 0;      // chunks per row group
    int rec = 0;         // bytes per record: 576 (BFP4) or 544 (BFP8)
    int64_t bytes() const { return ng * kc * (int64_t)rec; }
    int64_t group_bytes() const { return kc * (int64_t)rec; }
};

constexpr int kRecCodeBytes = 512;

// Fills g; returns BFP_OK or an error (with message set).
int make_geometry(int fmt, int64_t n, int64_t k, Geometry *g);

// Error reporting (thread-local message).
int fail(int code, const std::string &msg);

// Validation helpers.
bool aligned16(const void *p);
int check_matrix(const bfp_matrix *w, Geometry *g, bool device_ptr);

// Bounded-wait iteration limit for launches issued from this thread (0 = default).
int64_t wait_limit();

// How the MoE layer kernel is launched (bfp_set_launch_mode; process-wide).
int launch_mode();

// Whether one-row MoE layers run on the one-row kernel (bfp_set_row_path; process-wide).
bool row_path();

}  // namespace bfp
