// Greedy next-token choice over the LM head's fp32 logits (bfp_greedy_tokens): for each row, the index
// of the largest logit, ties to the lower index (the decode step after the LM head, P1 "Fused decode
// kernels": LM head then sampling; greedy decoding takes the arg max).
//
// Two dependent launches. The first spreads every row over S CTAs; each CTA reduces its slice to one
// 64-bit key (an order-preserving image of the value in the high word, the complement of the index
// in the low word, so that the unsigned maximum is the largest value and, among equal values, the
// lowest index) and stores it. The second takes the maximum of a row's S keys and writes the index.
// NaN logits are never chosen; a row with no other value gives index 0. The logits are read where
// the LM head left them (normally in L2), once.
#include <cuda_runtime.h>

#include "bfp_launch.h"

namespace bfp {

using namespace dev;

namespace {

constexpr int kGreedyThreads = 512;

__device__ __forceinline__ unsigned long long greedy_key(float v, int64_t i) {
    v += 0.0f;  // -0 and +0 compare equal: one key for both
    const uint32_t u = __float_as_uint(v);
    const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)k << 32) | (0xFFFFFFFFu - (uint32_t)i);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) { return a > b ? a : b; }

__global__ void __launch_bounds__(kGreedyThreads) greedy_partial(const float *logits, int64_t n, int64_t ldl, int S,
                                                                 unsigned long long *part) {
    __shared__ unsigned long long wbest[kGreedyThreads / kWarp];
    grid_dep_launch_dependents();
    grid_dep_wait();  // the logits come from the previous kernel on the stream
    const int r = blockIdx.y, s = blockIdx.x, tid = threadIdx.x;
    const int64_t c0 = n * s / S, c1 = n * (s + 1) / S;
    const float *row = logits + (int64_t)r * ldl;
    unsigned long long best = 0ull;  // below every real key (a NaN-only slice keeps it)
    constexpr int U = 8;  // loads in flight per thread
    int64_t i = c0 + tid;
    for (; i + (U - 1) * kGreedyThreads < c1; i += U * kGreedyThreads) {
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = __ldcg(row + i + u * kGreedyThreads);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v[u] == v[u]) best = umax64(best, greedy_key(v[u], i + u * kGreedyThreads));
    }
    for (; i < c1; i += kGreedyThreads) {
        const float v = __ldcg(row + i);
        if (v == v) best = umax64(best, greedy_key(v, i));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
    if ((tid & 31) == 0) wbest[tid >> 5] = best;
    __syncthreads();
    if (tid < kWarp) {
        best = tid < kGreedyThreads / kWarp ? wbest[tid] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
        if (tid == 0) part[(int64_t)r * S + s] = best;
    }
}

__global__ void __launch_bounds__(kWarp) greedy_final(const unsigned long long *part, int S, int32_t *tokens) {
    grid_dep_wait();  // the partial keys of the previous launch
    const int r = blockIdx.x, lane = threadIdx.x;
    unsigned long long best = 0ull;
    for (int s = lane; s < S; s += kWarp) best = umax64(best, part[(int64_t)r * S + s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (lane == 0) tokens[r] = best == 0ull ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
}

// CTAs per row: about two waves of the SMs over all rows, at least 2048 logits per CTA.
int greedy_split(int m, int64_t n, int *S) {
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    int64_t s = std::max<int64_t>(1, (int64_t)2 * di.sms / m);
    s = std::min<int64_t>(s, std::max<int64_t>(1, n / 2048));
    *S = (int)s;
    return BFP_OK;
}

int check_greedy(int m, int64_t n, int64_t ldl) {
    if (m < 1 || m > 16) return fail(BFP_ESHAPE, "m must be in 1..16");
    if (n < 1 || n > (int64_t(1) << 31) - 1) return fail(BFP_ESHAPE, "n must be in 1..2^31-1");
    if (ldl < n) return fail(BFP_EINVAL, "ldl must be >= n");
    return BFP_OK;
}

template <typename K, typename... Args>
cudaError_t launch_dependent(K kern, dim3 grid, dim3 block, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

}  // namespace bfp

using namespace bfp;

extern "C" int bfp_greedy_workspace_size(int m, int64_t n, size_t *bytes) {
    if (!bytes) return fail(BFP_EINVAL, "null bytes");
    int rc = check_greedy(m, n, n);
    if (rc) return rc;
    int S = 0;
    rc = greedy_split(m, n, &S);
    if (rc) return rc;
    *bytes = (size_t)m * S * sizeof(unsigned long long);
    return BFP_OK;
}

extern "C" int bfp_greedy_tokens(const float *logits, int m, int64_t n, int64_t ldl, int32_t *tokens, void *ws,
                                 size_t ws_bytes, bfp_stream_t stream) {
    int rc = check_greedy(m, n, ldl);
    if (rc) return rc;
    if (!logits || !tokens) return fail(BFP_EINVAL, "null pointer");
    if (!aligned16(logits) || !aligned16(tokens) || !aligned16(ws))
        return fail(BFP_EALIGN, "logits, tokens and ws must be 16-byte aligned");
    int S = 0;
    rc = greedy_split(m, n, &S);
    if (rc) return rc;
    if (!ws || ws_bytes < (size_t)m * S * sizeof(unsigned long long))
        return fail(BFP_EWORKSPACE, "workspace smaller than bfp_greedy_workspace_size");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    auto *part = static_cast<unsigned long long *>(ws);
    cudaError_t e = launch_dependent(greedy_partial, dim3(S, m), dim3(kGreedyThreads), st, logits, n, ldl, S, part);
    if (e != cudaSuccess) return cuda_fail(e, "launch greedy_partial");
    e = launch_dependent(greedy_final, dim3(m), dim3(kWarp), st, (const unsigned long long *)part, S, tokens);
    if (e != cudaSuccess) return cuda_fail(e, "launch greedy_final");
    return BFP_OK;
}
