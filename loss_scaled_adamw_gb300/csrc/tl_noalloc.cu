// tl_noalloc.cu - tl_unscale_norm_noalloc: unscale + overflow check + global
// norm + clip coefficient over a caller's fp32 gradient list, without any
// allocation.
//
// Who needs this.  tl_create allocates device memory (its chunk table, norm
// partials and scalars) with cudaMalloc.  Some callers cannot do that: a
// process whose device memory is entirely handed to another allocator (a
// framework's caching allocator or a fixed serving budget), code that must not
// allocate after initialisation (latency-critical or certified loops), and code
// running where a new allocation would break an ongoing capture or an external
// memory plan.  For them this entry point does the unscale / overflow / norm /
// clip part of the step with scratch memory that the library brings with it: a
// file-scope __device__ array below, which every GPU that loads this code holds
// until the process exits.
//
// When the scratch comes into being.  Under CUDA's lazy module loading (the
// default of recent toolkits) the module holding the array is loaded on a
// device at its first use there: the first call of this entry point on that
// device (its symbol lookup, occupancy query or launch).  That first call
// therefore takes device memory once (the 512 KiB array and the module's code)
// and can fail for want of it; it must come before any stream capture and
// before all device memory has been handed to another allocator.  Every later
// call on that device allocates nothing.  With CUDA_MODULE_LOADING=EAGER in the
// environment the module is loaded with the CUDA context instead.
//
// Limits: at most kNoAllocMaxTensors tensors and kNoAllocMaxChunks chunks of
// kChunk elements (2^16 * 2^14 = 2^30 elements); larger lists are rejected
// with TL_EINVAL.  The scratch is shared by every call on a device and keeps
// the last call's partials; each call writes every partial it later reads, so
// nothing has to start at zero, but calls that overlap on the GPU (two streams
// at once) race on it and must be serialised by the caller.
#include "tl_internal.cuh"

#include <cfloat>
#include <cmath>
#include <mutex>

#include "../../include/tl.h"

namespace tl {
namespace {

constexpr int kNoAllocMaxTensors = 256;
constexpr int kNoAllocNormThreads = 1024;  // one CTA; its last warp reads one per-warp sum per lane
constexpr int64_t kNoAllocMaxChunks = int64_t(1) << 16;
constexpr int kMaxDevices = 64;

// The scratch: one fp64 squared-norm partial per chunk (512 KiB per device).
static __device__ __align__(256) double g_noalloc_partials[kNoAllocMaxChunks];

struct NoAllocList {
    float* acc[kNoAllocMaxTensors];
    int64_t numel[kNoAllocMaxTensors];
    int64_t chunk_begin[kNoAllocMaxTensors + 1];  // first chunk of each tensor; [ntensors] = total
    int32_t ntensors;
};

__device__ __forceinline__ int tensor_of_chunk(const NoAllocList& L, int64_t c) {
    int lo = 0, hi = L.ntensors - 1;  // the last tensor whose first chunk is <= c
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (L.chunk_begin[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// u = acc * (1/S) in place; one partial sum of fp32 squares per chunk (fp32 over
// 8 elements, fp64 per thread, fixed-order block reduction).  A simpler
// summation than the allocating path's float-float one (this entry point has no
// scratch for per-warp partials); its norm meets the same 1e-6 relative bound.
__global__ void __launch_bounds__(kThreads)
k_noalloc_unscale(const __grid_constant__ NoAllocList L, float inv_s, int64_t nchunks) {
    __shared__ double red[kThreads / 32];
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        const int t = tensor_of_chunk(L, c);
        const int64_t start = (c - L.chunk_begin[t]) * kChunk;
        const int64_t rest = L.numel[t] - start;
        const int len = static_cast<int>(rest < kChunk ? rest : kChunk);
        float* __restrict__ a = L.acc[t] + start;
        double tsum = 0.0;
        int done = 0;
        if ((reinterpret_cast<uintptr_t>(a) & 15u) == 0) {
            const int nv = len / 8;
            for (int i = threadIdx.x; i < nv; i += kThreads) {
                float4 x = reinterpret_cast<float4*>(a)[2 * i];
                float4 y = reinterpret_cast<float4*>(a)[2 * i + 1];
                float u[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
                float q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    u[e] = __fmul_rn(u[e], inv_s);
                    q[e] = __fmul_rn(u[e], u[e]);
                }
                reinterpret_cast<float4*>(a)[2 * i] = make_float4(u[0], u[1], u[2], u[3]);
                reinterpret_cast<float4*>(a)[2 * i + 1] = make_float4(u[4], u[5], u[6], u[7]);
                const float s = __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                                          __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
                if (!isinf(s)) {
                    tsum = __dadd_rn(tsum, static_cast<double>(s));
                } else {
                    double d = 0.0;
#pragma unroll
                    for (int e = 0; e < 8; ++e) d = __dadd_rn(d, static_cast<double>(q[e]));
                    tsum = __dadd_rn(tsum, d);
                }
            }
            done = nv * 8;
        }
        for (int j = done + threadIdx.x; j < len; j += kThreads) {
            const float u = __fmul_rn(a[j], inv_s);
            a[j] = u;
            tsum = __dadd_rn(tsum, static_cast<double>(__fmul_rn(u, u)));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tsum = __dadd_rn(tsum, __shfl_xor_sync(0xffffffffu, tsum, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = tsum;
        __syncthreads();
        if (threadIdx.x == 0) {
            double s = 0.0;
#pragma unroll
            for (int k = 0; k < kThreads / 32; ++k) s = __dadd_rn(s, red[k]);
            g_noalloc_partials[c] = s;  // device code names the scratch directly
        }
        __syncthreads();
    }
}

// Fixed-order reduction of the partials, then norm, clip coefficient and the
// overflow decision (a non-finite u makes its square, hence the sum, non-finite).
__global__ void __launch_bounds__(kNoAllocNormThreads)
k_noalloc_norm(const double* __restrict__ partials, int64_t nchunks, float max_norm, tl_norm_result* out) {
    __shared__ double red[kNoAllocNormThreads / 32];
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < nchunks; i += kNoAllocNormThreads) s = __dadd_rn(s, partials[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __dadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x < 32) {
        double v = red[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = __dadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (threadIdx.x == 0) {
            const float norm = __double2float_rn(__dsqrt_rn(v));
            float coef = 1.0f;
            if (max_norm > 0.0f) {
                const float cc = __fdiv_rn(max_norm, __fadd_rn(norm, 1e-6f));
                if (cc < 1.0f) coef = cc;
            }
            out->norm = norm;
            out->coef = coef;
            out->found_inf = isfinite(v) ? 0 : 1;
            out->reserved = 0;
            out->sumsq = v;
        }
    }
}

std::mutex g_setup_mu;
double* g_scratch_addr[kMaxDevices] = {nullptr};
int g_grid[kMaxDevices] = {0};

// A normal power of two: its reciprocal is then exact and finite (a subnormal S
// below 2^-127 would make 1/S overflow to infinity).
bool pow2(float x) {
    if (!(x >= FLT_MIN) || !std::isfinite(x)) return false;
    int e = 0;
    return std::frexp(x, &e) == 0.5f;
}

}  // namespace
}  // namespace tl

extern "C" int tl_unscale_norm_noalloc(int64_t ntensors, const int64_t* numel, float* const* acc, float S,
                                       float max_norm, tl_norm_result* out, tl_stream stream) {
    using namespace tl;
    if (ntensors < 0 || ntensors > kNoAllocMaxTensors) return TL_EINVAL;
    if (ntensors > 0 && (numel == nullptr || acc == nullptr)) return TL_EINVAL;
    if (out == nullptr || (reinterpret_cast<uintptr_t>(out) & 7u) != 0) return TL_EINVAL;
    if (!pow2(S) || std::isnan(max_norm)) return TL_EINVAL;
    NoAllocList L;
    L.ntensors = static_cast<int32_t>(ntensors);
    int64_t nchunks = 0;
    for (int64_t i = 0; i < ntensors; ++i) {
        if (numel[i] < 0) return TL_EINVAL;
        if (numel[i] > 0 && (acc[i] == nullptr || (reinterpret_cast<uintptr_t>(acc[i]) & 3u) != 0)) return TL_EINVAL;
        L.acc[i] = acc[i];
        L.numel[i] = numel[i];
        L.chunk_begin[i] = nchunks;
        nchunks += (numel[i] + kChunk - 1) / kChunk;
        if (nchunks > kNoAllocMaxChunks) return TL_EINVAL;  // beyond the scratch: rejected
    }
    L.chunk_begin[ntensors] = nchunks;
    // distinct tensors must not overlap (each u is written once)
    for (int64_t i = 0; i < ntensors; ++i)
        for (int64_t j = i + 1; j < ntensors; ++j) {
            if (numel[i] == 0 || numel[j] == 0) continue;
            const uintptr_t a0 = reinterpret_cast<uintptr_t>(acc[i]), a1 = a0 + uintptr_t(numel[i]) * 4;
            const uintptr_t b0 = reinterpret_cast<uintptr_t>(acc[j]), b1 = b0 + uintptr_t(numel[j]) * 4;
            if (a0 < b1 && b0 < a1) return TL_EINVAL;
        }

    // Set-up, once per device, with that device current: the scratch array's
    // device address (in host code its name is only a host-side stand-in).
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return TL_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return TL_EINVAL;
    double* partials = nullptr;
    int grid = 0;
    {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (g_scratch_addr[dev] == nullptr) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || p == nullptr) return TL_ECUDA;
            int sms = 0, per_sm = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TL_ECUDA;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_noalloc_unscale, kThreads, 0) != cudaSuccess)
                return TL_ECUDA;
            g_grid[dev] = sms * (per_sm > 0 ? per_sm : 1);
            g_scratch_addr[dev] = static_cast<double*>(p);
        }
        partials = g_scratch_addr[dev];
        grid = g_grid[dev];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (nchunks > 0) {
        const int g = static_cast<int>(nchunks < grid ? nchunks : grid);
        k_noalloc_unscale<<<g, kThreads, 0, s>>>(L, 1.0f / S, nchunks);  // S a normal power of two: exact
        if (cudaGetLastError() != cudaSuccess) return TL_ECUDA;
    }
    k_noalloc_norm<<<1, kNoAllocNormThreads, 0, s>>>(partials, nchunks, max_norm, out);
    if (cudaGetLastError() != cudaSuccess) return TL_ECUDA;
    return TL_OK;
}
