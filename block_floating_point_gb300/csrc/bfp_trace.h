// Optional per-CTA timestamps (%globaltimer, ns) for studying where a kernel's
// time goes. Compiled in only with -DBFP_TRACE; the library as built by
// build.py has none of it, and BFP_TRACE_AT expands to nothing.
#pragma once

#ifdef BFP_TRACE
#define BFP_TRACE_SLOTS 128
// One copy per translation unit, set through that unit's bfp_debug_set_trace
// (trace builds only); one row of slots per CTA.
static __device__ unsigned long long *g_bfp_trace = nullptr;
#define BFP_TRACE_AT(slot)                                                                                  \
    do {                                                                                                    \
        if (g_bfp_trace != nullptr && threadIdx.x == 0)                                                     \
            g_bfp_trace[(size_t)blockIdx.x * BFP_TRACE_SLOTS + (slot)] = bfp::dev::global_ns();              \
    } while (0)
// Thread t stamps a slot of its CTA's row.
#define BFP_TRACE_AT_T(slot, t)                                                                             \
    do {                                                                                                    \
        if (g_bfp_trace != nullptr && threadIdx.x == (t))                                                   \
            g_bfp_trace[(size_t)blockIdx.x * BFP_TRACE_SLOTS + (slot)] = bfp::dev::global_ns();              \
    } while (0)
// Lane 0 of every warp stamps slot (base + warp index) of its CTA's row.
#define BFP_TRACE_WARP(base)                                                                                \
    do {                                                                                                    \
        if (g_bfp_trace != nullptr && (threadIdx.x & 31) == 0)                                              \
            g_bfp_trace[(size_t)blockIdx.x * BFP_TRACE_SLOTS + (base) + (threadIdx.x >> 5)] =               \
                bfp::dev::global_ns();                                                                      \
    } while (0)
// Lane 0 of every warp stores a value into slot (base + warp index) of its CTA's row.
#define BFP_TRACE_WARP_SET(base, v)                                                                         \
    do {                                                                                                    \
        if (g_bfp_trace != nullptr && (threadIdx.x & 31) == 0)                                              \
            g_bfp_trace[(size_t)blockIdx.x * BFP_TRACE_SLOTS + (base) + (threadIdx.x >> 5)] = (v);          \
    } while (0)
// Stores a value (a duration accumulated in registers, a count) into a slot of thread 0's row.
#define BFP_TRACE_SET(slot, v)                                                                              \
    do {                                                                                                    \
        if (g_bfp_trace != nullptr && threadIdx.x == 0)                                                     \
            g_bfp_trace[(size_t)blockIdx.x * BFP_TRACE_SLOTS + (slot)] = (v);                               \
    } while (0)
#define BFP_TRACE_NOW() ((unsigned long long)clock64())  // SM cycles (cheap), for durations
#else
#define BFP_TRACE_SET(slot, v) \
    do {                       \
    } while (0)
#define BFP_TRACE_NOW() 0ull
#define BFP_TRACE_WARP(base) \
    do {                     \
    } while (0)
#define BFP_TRACE_AT_T(slot, t) \
    do {                        \
    } while (0)
#define BFP_TRACE_WARP_SET(base, v) \
    do {                            \
    } while (0)
#define BFP_TRACE_AT(slot) \
    do {                   \
    } while (0)
#endif
