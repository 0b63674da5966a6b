// tl_kernels.cu - sm_103a kernels of the loss-scaled AdamW optimizer step.
//
// The step is bound by HBM bandwidth (well under one flop per byte), so the
// kernels are streaming kernels, not tensor-core kernels: a persistent grid
// walks a device-resident chunk table (multi-tensor apply), each thread moves
// 8 elements per access with 128-bit loads and stores and keeps several such
// vectors in flight, and a chunk whose pointers are not 16-byte aligned, or
// the tail of a tensor, takes a coalesced scalar path.
//
// Floating point.  Every element-wise operation is written as an explicit
// round-to-nearest intrinsic (__fmul_rn, __fadd_rn, __fsub_rn, __fdiv_rn,
// __fsqrt_rn, __fmaf_rn and the fp64 forms), and this file is compiled with
// -fmad=false, so nothing is contracted or reassociated: each output element is
// the correctly rounded result of one declared sequence of operations.
//
// Pages cited (by title):
//   [MP]  "Mixed precision, loss scaling, gradient accumulation, and activation
//         checkpointing" (tinyllm module L11.1)
//   [MEG] "Megatron Internals III: Mixed Precision, Loss Scaling, and Grad Clipping"
//   [ZRO] "Your weights fit on one device but Adam's moments do not - how do you
//         shard the optimizer state?"
//   [RST] "Practical LLM in Rust", ch. 13 "Accumulate gradients and recompute activations"
#include "tl_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace tl {
namespace {

// Minimum resident CTAs per SM requested from the compiler (register budget) for
// the accumulation kernel (the first micro-batch, which reads no partial sum,
// needs fewer registers), the many-list kernels (TL_MINB_FEW: launches of one or two lists, whose chunks
// are worked faster when more of them are in flight), the AdamW kernel and its
// re-materialising form; *_UNROLL: 8-element vectors per thread per trip of the
// AdamW loops.  The defaults are the fastest measured (one vector per thread at
// 2 CTAs/SM equals two at 1 CTA/SM on the 1.24B list, 2-4 % faster on the
// ragged 100k list, whose segments are mostly partial).
#ifndef TL_MINB_ACC
#define TL_MINB_ACC 4
#endif
#ifndef TL_MINB_ACC_FIRST
#define TL_MINB_ACC_FIRST 6
#endif
#ifndef TL_MINB_MANY
#define TL_MINB_MANY 3
#endif
// 8-bit lists: with whole 16-element blocks per lane (TL_E4M3_BLOCKS) the 8-list
// forms run at 3 CTAs per SM, where ptxas keeps part of the loop-invariant state in
// local memory (L1); measured on the 1.24B list: 2.64 ms against 2.83 at 2 CTAs per
// SM without spills (and 2.83 for 8-element vectors at 4 CTAs per SM)
#ifndef TL_MINB_MANY_E4M3
#define TL_MINB_MANY_E4M3 (TL_E4M3_BLOCKS ? 3 : 4)
#endif
// Small-tensor groups (a warp per tensor, a few hundred elements each) are
// latency-bound: more resident CTAs keep more tensors in flight.  The one- and
// two-list forms of the many-list kernel, and AdamW.
#ifndef TL_MINB_GROUP_FEW
#define TL_MINB_GROUP_FEW 5
#endif
#ifndef TL_MINB_ADAM_GROUP
#define TL_MINB_ADAM_GROUP 3
#endif
#ifndef TL_MINB_FEW
#define TL_MINB_FEW 5
#endif
#ifndef TL_REMAT_UNROLL
#define TL_REMAT_UNROLL 1
#endif
#ifndef TL_MINB_REMAT_FEW
#define TL_MINB_REMAT_FEW 3
#endif
#ifndef TL_MINB_REMAT
#define TL_MINB_REMAT 2
#endif
#ifndef TL_ADAM_UNROLL
#define TL_ADAM_UNROLL 1
#endif
#ifndef TL_MINB_ADAM
#define TL_MINB_ADAM 2
#endif

constexpr int kVec = 8;     // elements per vector access (16 B of a 16-bit stream)
constexpr int kUnroll = 4;  // vectors in flight per thread in the accumulate/unscale kernels
constexpr int kScalar = 8;  // elements per thread in flight on the scalar path (streams of unequal phase)
// ... in the many-list kernel's forms for one or two lists, and for more lists
#ifndef TL_SCALAR_FEW
#define TL_SCALAR_FEW 2
#endif
#ifndef TL_SCALAR_MANY
#define TL_SCALAR_MANY 1
#endif
#ifndef TL_SCALAR_FEW_GROUP
#define TL_SCALAR_FEW_GROUP 2
#endif
// 8-bit lists in whole-CTA segments: a lane takes whole 16-element blocks (16 codes
// and their scale per list and load) where every stream is 16-byte aligned
#ifndef TL_E4M3_BLOCKS
#define TL_E4M3_BLOCKS 1
#endif
// AdamW's scalar path (u read from the buffer): the last partial trip of a segment
// batched with clamped indices instead of element by element (TL_ADAM_CLAMP;
// gapped ragged list: 2.15 -> 2.11 ms, the small-tensor groups 9 % faster)
#ifndef TL_ADAM_CLAMP
#define TL_ADAM_CLAMP 1
#endif
// squared-norm partials: two float-float accumulators per lane (SumSqT's P).  Off:
// with them the ragged list's check pass was 1 % faster but the 8-list pass over the
// 1.24B list 7 % slower (register spills), and every partial-writing kernel must take
// the same form for the passes to agree bit for bit.
#ifndef TL_SQ_PAIRS
#define TL_SQ_PAIRS 0
#endif
// many-list pass: products and weighted sums two fp32 lanes per instruction
#ifndef TL_PAIRS
#define TL_PAIRS 1
#endif

// ---------------------------------------------------------------------------
// 8-element vector access
// ---------------------------------------------------------------------------

// fp32 streams: 8 elements = 32 bytes per access.  TL_V8 selects one 256-bit
// access (sm_100+ ld/st.global.v8) instead of two 128-bit ones; TL_LDHINT /
// TL_STHINT select L1 no-allocate or evict-first (streaming) cache hints.  The
// defaults (256-bit, L1 no-allocate) were the fastest of the measured variants
// on every kernel (e.g. clip+AdamW 6.13 -> 6.47 TB/s, first accumulation
// 5.16 -> 6.16 TB/s at 1.24B parameters).
#ifndef TL_V8
#define TL_V8 1
#endif
#ifndef TL_LDHINT
#define TL_LDHINT 1
#endif
#ifndef TL_STHINT
#define TL_STHINT 1
#endif

#if TL_LDHINT == 1
#define TL_LD_Q ".L1::no_allocate"
#elif TL_LDHINT == 2
#define TL_LD_Q ".cs"
#else
#define TL_LD_Q ""
#endif
#if TL_STHINT == 1
#define TL_ST_Q ".L1::no_allocate"
#elif TL_STHINT == 2
#define TL_ST_Q ".cs"
#else
#define TL_ST_Q ""
#endif

// `wide` (all fp32 pointers of the chunk 32-byte aligned, checked per chunk)
// selects the 256-bit form, which needs 32-byte alignment; otherwise two
// 128-bit accesses, which need 16.
__device__ __forceinline__ void ld8_f32(const float* __restrict__ p, float (&x)[8], bool wide) {
#if TL_V8
    if (wide) {
        asm volatile("ld.global" TL_LD_Q ".v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]), "=f"(x[4]), "=f"(x[5]), "=f"(x[6]), "=f"(x[7])
                     : "l"(p));
        return;
    }
#endif
#if TL_LDHINT != 0
    asm volatile("ld.global" TL_LD_Q ".v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]) : "l"(p));
    asm volatile("ld.global" TL_LD_Q ".v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(x[4]), "=f"(x[5]), "=f"(x[6]), "=f"(x[7]) : "l"(p + 4));
#else
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
#endif
}

__device__ __forceinline__ void st8_f32(float* __restrict__ p, const float (&x)[8], bool wide) {
#if TL_V8
    if (wide) {
        asm volatile("st.global" TL_ST_Q ".v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                     :: "l"(p), "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7])
                     : "memory");
        return;
    }
#endif
#if TL_STHINT != 0
    asm volatile("st.global" TL_ST_Q ".v4.f32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]) : "memory");
    asm volatile("st.global" TL_ST_Q ".v4.f32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p + 4), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]) : "memory");
#else
    reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
#endif
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t r, float& lo, float& hi) {
    lo = __uint_as_float(r << 16);          // bf16 -> fp32 is exact: the upper half of the word
    hi = __uint_as_float(r & 0xffff0000u);
}

__device__ __forceinline__ void unpack_f16x2(uint32_t r, float& lo, float& hi) {
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = r;
    const float2 f = __half22float2(h);     // fp16 -> fp32 is exact
    lo = f.x;
    hi = f.y;
}

// Two E4M3 codes (the low byte first) to fp32, exactly: the hardware converts
// E4M3 pairs to fp16 pairs (every E4M3 value, NaN included, is an fp16 value).
__device__ __forceinline__ void unpack_e4m3x2(uint32_t codes2, float& lo, float& hi) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes2 & 0xffffu), __NV_E4M3);
    unpack_f16x2(static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16), lo, hi);
}

// Micro-batch gradient streams: read once per kernel, through the read-only path.
// Element i of a segment's stream `base`; `sc` points at the segment's block
// scales (8-bit gradients only; the other types ignore it).  A segment starts
// on a multiple of 16 elements and 8-bit vectors sit on multiples of 8, so the
// 8 elements of one vector share one scale.
template <int DT> struct Grad;

template <> struct Grad<kBF16> {
    static constexpr int kBytes = 2;
    __device__ static __forceinline__ void ld8(const void* base, int64_t i, float (&x)[8], const float*) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(base) + i));
        unpack_bf16x2(r.x, x[0], x[1]); unpack_bf16x2(r.y, x[2], x[3]);
        unpack_bf16x2(r.z, x[4], x[5]); unpack_bf16x2(r.w, x[6], x[7]);
    }
    __device__ static __forceinline__ float ld1(const void* base, int64_t i, const float*) {
        return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(base) + i)) << 16);
    }
};

template <> struct Grad<kF16> {
    static constexpr int kBytes = 2;
    __device__ static __forceinline__ void ld8(const void* base, int64_t i, float (&x)[8], const float*) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(base) + i));
        unpack_f16x2(r.x, x[0], x[1]); unpack_f16x2(r.y, x[2], x[3]);
        unpack_f16x2(r.z, x[4], x[5]); unpack_f16x2(r.w, x[6], x[7]);
    }
    __device__ static __forceinline__ float ld1(const void* base, int64_t i, const float*) {
        const unsigned short b = __ldg(static_cast<const unsigned short*>(base) + i);
        return __half2float(__ushort_as_half(b));
    }
};

template <> struct Grad<kF32> {
    static constexpr int kBytes = 4;
    __device__ static __forceinline__ void ld8(const void* base, int64_t i, float (&x)[8], const float*) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
        const float4 a = __ldg(p), b = __ldg(p + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    __device__ static __forceinline__ float ld1(const void* base, int64_t i, const float*) {
        return __ldg(static_cast<const float*>(base) + i);
    }
};

// 8-bit gradients: element value = fl32(code value * block scale) ("Training at
// Scale", section 41.5: dequantize before accumulation).
template <> struct Grad<kE4M3> {
    static constexpr int kBytes = 1;
    __device__ static __forceinline__ void ld8(const void* base, int64_t i, float (&x)[8], const float* sc) {
        const uint2 c = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned char*>(base) + i));
        const float s = __ldg(sc + (i >> 4));
        unpack_e4m3x2(c.x, x[0], x[1]); unpack_e4m3x2(c.x >> 16, x[2], x[3]);
        unpack_e4m3x2(c.y, x[4], x[5]); unpack_e4m3x2(c.y >> 16, x[6], x[7]);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(x[e], s);
    }
    __device__ static __forceinline__ float ld1(const void* base, int64_t i, const float* sc) {
        float lo, hi;
        unpack_e4m3x2(__ldg(static_cast<const unsigned char*>(base) + i), lo, hi);
        return __fmul_rn(lo, __ldg(sc + (i >> 4)));
    }
};

// The block scales of a segment's 8-bit gradient stream (nullptr for the other types).
template <int GDT>
__device__ __forceinline__ const float* grad_scales(const void* base, const Chunk& ch) {
    if (GDT != kE4M3) return nullptr;
    return reinterpret_cast<const float*>(static_cast<const char*>(base) + ch.gscale) + (ch.start >> 4);
}

// Raw 16-byte loads of 8 gradient elements and the exact conversion of element e
// (for the many-list kernel, which keeps only the raw words live).
template <int DT> struct GradRaw;

template <> struct GradRaw<kBF16> {
    using T = uint4;
    __device__ static __forceinline__ T ld(const void* base, int64_t i, const float*) {
        return __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(base) + i));
    }
    __device__ static __forceinline__ float at(const T& r, int e) {
        const uint32_t w = e < 2 ? r.x : e < 4 ? r.y : e < 6 ? r.z : r.w;
        return (e & 1) ? __uint_as_float(w & 0xffff0000u) : __uint_as_float(w << 16);
    }
};

template <> struct GradRaw<kF16> {
    using T = uint4;
    __device__ static __forceinline__ T ld(const void* base, int64_t i, const float*) {
        return __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(base) + i));
    }
    __device__ static __forceinline__ float at(const T& r, int e) {
        const uint32_t w = e < 2 ? r.x : e < 4 ? r.y : e < 6 ? r.z : r.w;
        return __half2float(__ushort_as_half(static_cast<unsigned short>((e & 1) ? (w >> 16) : (w & 0xffffu))));
    }
};

template <> struct GradRaw<kF32> {
    struct T { float4 a, b; };
    __device__ static __forceinline__ T ld(const void* base, int64_t i, const float*) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
        return T{__ldg(p), __ldg(p + 1)};
    }
    __device__ static __forceinline__ float at(const T& r, int e) {
        const float4& h = e < 4 ? r.a : r.b;
        const int k = e & 3;
        return k == 0 ? h.x : k == 1 ? h.y : k == 2 ? h.z : h.w;
    }
};

template <> struct GradRaw<kE4M3> {
    struct T { uint2 c; float s; };
    __device__ static __forceinline__ T ld(const void* base, int64_t i, const float* sc) {
        return T{__ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned char*>(base) + i)), __ldg(sc + (i >> 4))};
    }
    __device__ static __forceinline__ float at(const T& r, int e) {
        const uint32_t w = e < 4 ? r.c.x : r.c.y;
        float lo, hi;
        unpack_e4m3x2((e & 2) ? (w >> 16) : w, lo, hi);
        return __fmul_rn((e & 1) ? hi : lo, r.s);
    }
};

// Model-precision parameter stores: round to nearest even ([MP] section 2, rd16).
template <int DT> struct Param;

template <> struct Param<kBF16> {
    __device__ static __forceinline__ uint32_t pack2(float lo, float hi) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&b);
    }
    __device__ static __forceinline__ void st1(void* base, int64_t i, float x) {
        static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(x);
    }
};

template <> struct Param<kF16> {
    __device__ static __forceinline__ uint32_t pack2(float lo, float hi) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ static __forceinline__ void st1(void* base, int64_t i, float x) {
        static_cast<__half*>(base)[i] = __float2half_rn(x);
    }
};

template <int DT>
__device__ __forceinline__ void st8_param(void* base, int64_t i, const float (&x)[8]) {
    uint4 r;
    r.x = Param<DT>::pack2(x[0], x[1]);
    r.y = Param<DT>::pack2(x[2], x[3]);
    r.z = Param<DT>::pack2(x[4], x[5]);
    r.w = Param<DT>::pack2(x[6], x[7]);
    *reinterpret_cast<uint4*>(static_cast<unsigned short*>(base) + i) = r;
}

__device__ __forceinline__ bool aligned16(const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

__device__ __forceinline__ bool aligned32(const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & 31u) == 0;
}

// A chunk is one segment (a piece of one large tensor, worked by the whole CTA:
// NT = kThreads) or a group of up to kGroup small tensors (one per warp: NT =
// 32; warps beyond the group idle).  Each kernel's per-segment body is a
// template on NT, so both forms have compile-time strides.

// ---------------------------------------------------------------------------
// a2: accumulate micro-batch i.  [RST] ch. 13 "Weight each mean by the targets
// it represents"; [MP] section 2 "Gradient accumulation" (no zeroing between
// micro-batches).  acc = w*g (first) or fma(w, g, acc).
// ---------------------------------------------------------------------------
// Vector plan of one segment.  head elements are done one by one first, then
// whole 8-element vectors from element head on, then the tail.  head is 0 when
// every stream is already on a 16-byte boundary; when the streams are not, but
// all sit at the same element phase r modulo 8 (tensors packed back to back in
// every list), head = 8 - r puts each fp32 stream on a 32-byte and each 16-bit
// stream on a 16-byte boundary; otherwise there is no vector part.
struct VecPlan {
    int head;
    bool vec;
    bool wide;  // fp32 streams 32-byte aligned from head on: 256-bit accesses
};

template <int ES>
__device__ __forceinline__ int ephase(const void* p) {
    return static_cast<int>((reinterpret_cast<uintptr_t>(p) / ES) & 7);
}

// In the vector plan the head (< 8 elements) and the tail (< 8) of a segment are
// single elements.  A segment that takes them early gives each to one thread:
// head element t to thread t, tail element done + (t - 8) to thread t >= 8 (a
// warp has 32 threads).  Returns the element of thread t, or -1.
__device__ __forceinline__ int edge_element(int t, int head, int done, int len) {
    if (t < head) return t;
    if (t >= 8 && t - 8 < len - done) return done + (t - 8);
    return -1;
}

// ---------------------------------------------------------------------------
// Rotated vectors: 16-bit streams whose element phase differs from the frame's
// (the read side of the many-list forms of one or two lists, whole-CTA segments).
// The frame is one stream's alignment; lanes 0-30 of a warp work 31 consecutive
// 8-element vectors o = head + 8 i, and lane 31 only helps.  For a stream whose
// phase is d elements past the frame's (1..7), every lane loads the aligned 16-byte
// block that starts d elements before its vector (lane 31: before the vector after
// lane 30's), takes the next block from lane L + 1 with a shuffle, and picks its 8
// values out of the two; so each block is loaded once and no load waits for
// another.  A block that holds any byte of a tensor lies in that byte's memory
// pages, so the loads are always safe, and the bytes outside the vector are never
// used.  (The same on the AdamW pass, with its three rotated fp32 stores, measured
// slower than element-by-element access: the shuffles and selects of four streams
// outweigh the wider accesses.)
// ---------------------------------------------------------------------------
constexpr int kRotLanes = 31;   // vectors per warp and trip on the rotated path

// 8 consecutive 16-bit values (as a raw 16-byte word) at element o of a stream d
// elements (0..7) past the frame's phase, read-only data.  act: this lane works a
// vector; ld: this lane's block is needed (its vector, or the vector before it,
// exists).  Every lane of the warp calls this (shuffles).  The words from word d / 2
// on are taken with a shifter of selects (a switch over d would cost branch
// resolution on every vector), and an odd rotation joins half-words with funnel
// shifts.
__device__ __forceinline__ uint4 ld16_rot(const unsigned short* x, int o, int d, bool act, bool ld) {
    if (d == 0) return act ? __ldg(reinterpret_cast<const uint4*>(x + o)) : make_uint4(0u, 0u, 0u, 0u);
    uint4 b = make_uint4(0u, 0u, 0u, 0u), n;
    if (ld) b = __ldg(reinterpret_cast<const uint4*>(x + o - d));   // 16-byte aligned
    n.x = __shfl_down_sync(0xffffffffu, b.x, 1);
    n.y = __shfl_down_sync(0xffffffffu, b.y, 1);
    n.z = __shfl_down_sync(0xffffffffu, b.z, 1);
    n.w = __shfl_down_sync(0xffffffffu, b.w, 1);
    const uint32_t w[8] = {b.x, b.y, b.z, b.w, n.x, n.y, n.z, n.w};
    const bool s2 = (d & 4) != 0, s1 = (d & 2) != 0;
    uint32_t y[6], r[5];
#pragma unroll
    for (int k = 0; k < 6; ++k) y[k] = s2 ? w[k + 2] : w[k];
#pragma unroll
    for (int k = 0; k < 5; ++k) r[k] = s1 ? y[k + 1] : y[k];
    const uint32_t sh = (d & 1) ? 16u : 0u;
    return make_uint4(__funnelshift_r(r[0], r[1], sh), __funnelshift_r(r[1], r[2], sh), __funnelshift_r(r[2], r[3], sh),
                      __funnelshift_r(r[3], r[4], sh));
}

template <int NT, int GDT, bool FIRST>
__device__ __forceinline__ void accumulate_segment(const Chunk& ch, int t, const void* const* gp, float w) {
    float* __restrict__ acc0 = ch.acc;
    const void* gb = gp[ch.tensor];
    const char* g0 = static_cast<const char*>(gb) + ch.start * Grad<GDT>::kBytes;
    const float* sc = grad_scales<GDT>(gb, ch);
    const int len = ch.len;
    VecPlan pl{0, false, false};
    if (aligned16(acc0) && aligned16(g0)) pl = VecPlan{0, true, aligned32(acc0)};
    else if (ephase<4>(acc0) == ephase<Grad<GDT>::kBytes>(g0)) pl = VecPlan{(8 - ephase<4>(acc0)) & 7, true, true};
    if (GDT == kE4M3 && pl.head != 0) pl.vec = false;  // an 8-bit vector must not straddle two blocks
    int head = 0, done = 0;
    if (pl.vec) {
        head = min(pl.head, len);
        const bool wide = pl.wide;
        float* __restrict__ acc = acc0 + head;
        const void* g = g0 + head * Grad<GDT>::kBytes;
        const int nv = (len - head) / kVec;
        int i = t;
        for (; i + (kUnroll - 1) * NT < nv; i += kUnroll * NT) {
            float gx[kUnroll][8], ax[kUnroll][8];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) Grad<GDT>::ld8(g, int64_t(i + u * NT) * kVec, gx[u], sc);
            if (!FIRST) {
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) ld8_f32(acc + (i + u * NT) * kVec, ax[u], wide);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    ax[u][e] = FIRST ? __fmul_rn(w, gx[u][e]) : __fmaf_rn(w, gx[u][e], ax[u][e]);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) st8_f32(acc + (i + u * NT) * kVec, ax[u], wide);
        }
        for (; i < nv; i += NT) {
            float gx[8], ax[8];
            Grad<GDT>::ld8(g, int64_t(i) * kVec, gx, sc);
            if (!FIRST) ld8_f32(acc + i * kVec, ax, wide);
#pragma unroll
            for (int e = 0; e < 8; ++e) ax[e] = FIRST ? __fmul_rn(w, gx[e]) : __fmaf_rn(w, gx[e], ax[e]);
            st8_f32(acc + i * kVec, ax, wide);
        }
        done = head + nv * kVec;
    }
    auto one = [&](int j) {
        const float gj = Grad<GDT>::ld1(g0, j, sc);
        acc0[j] = FIRST ? __fmul_rn(w, gj) : __fmaf_rn(w, gj, acc0[j]);
    };
    for (int j = t; j < head; j += NT) one(j);          // head
    // tail, or the whole segment without a vector part: kScalar elements per
    // thread loaded before any is stored
    int j = done + t;
    for (; j + (kScalar - 1) * NT < len; j += kScalar * NT) {
        float gx[kScalar], ax[kScalar];
#pragma unroll
        for (int q = 0; q < kScalar; ++q) {
            gx[q] = Grad<GDT>::ld1(g0, j + q * NT, sc);
            if (!FIRST) ax[q] = acc0[j + q * NT];
        }
#pragma unroll
        for (int q = 0; q < kScalar; ++q) acc0[j + q * NT] = FIRST ? __fmul_rn(w, gx[q]) : __fmaf_rn(w, gx[q], ax[q]);
    }
    for (; j < len; j += NT) one(j);
}

// Warp w's tensor of group chunk c.  The groups follow the whole-CTA chunks in the
// table, kGroup segments each (a short group is padded with empty segments), and
// the launch over the groups starts at c0 = the first group, whose first segment
// is segment c0 (the whole-CTA chunks before it hold one segment each).
__device__ __forceinline__ const Chunk& group_segment(const Chunk* __restrict__ chunks, int64_t c0, int64_t c) {
    return chunks[c0 + (c - c0) * kGroup + (threadIdx.x >> 5)];
}

// Chunks [c0, c1) in runs of `run` consecutive chunks of the table, CTA b taking
// runs b, b + gridDim.x, ...: work(c) for every chunk of a run in table order, then
// done(first chunk of the run).  Runs are fixed by the table, not by the grid, so a
// sum kept over a run has the same order on any device.
template <class Work, class Done>
__device__ __forceinline__ void for_runs(int64_t c0, int64_t c1, int run, Work work, Done done) {
    for (int64_t r0 = c0 + int64_t(blockIdx.x) * run; r0 < c1; r0 += int64_t(gridDim.x) * run) {
        const int64_t r1 = r0 + run < c1 ? r0 + run : c1;
        for (int64_t c = r0; c < r1; ++c) work(c);
        done(r0);
    }
}

// Lists of short segments take the split forms (TL_PAIR_SEGS; tl_plan reports the
// forms by the default, on).
#ifndef TL_PAIR_SEGS
#define TL_PAIR_SEGS 1
#endif
constexpr bool kPairSegs = TL_PAIR_SEGS != 0;
// ... and so do the AdamW passes (TL_SPLIT_ADAM)
#ifndef TL_SPLIT_ADAM
#define TL_SPLIT_ADAM 1
#endif
constexpr bool kSplitAdam = TL_SPLIT_ADAM != 0;

// The runs of a partial-writing kernel by its form: NT = kThreads, every chunk by
// the whole CTA; NT = kSplitThreads, the CTA split into kThreads / NT parts that work
// as many chunks of a run at once (part h: chunks r0 + h, r0 + h + kThreads / NT,
// ...), for lists of short segments (runs of several chunks), where a thread's
// share of a segment's setup then comes with several times the vectors; NT = 32,
// small-tensor groups (one warp per tensor).  A thread works chunk c as thread
// threadIdx.x % NT of its segment.  The partials stay per run (finish_warp,
// finish_run), and every partial-writing kernel of a context takes the same form,
// so the passes that reach the same u give their lanes the same elements.
template <int NT, class Work, class Done>
__device__ __forceinline__ void for_runs_nt(int64_t c0, int64_t c1, int run, Work work, Done done) {
    if (NT != kSplitThreads) {
        for_runs(c0, c1, run, work, done);
        return;
    }
    const int h = threadIdx.x / kSplitThreads;
    for (int64_t r0 = c0 + int64_t(blockIdx.x) * run; r0 < c1; r0 += int64_t(gridDim.x) * run) {
        const int64_t r1 = r0 + run < c1 ? r0 + run : c1;
        for (int64_t c = r0 + h; c < r1; c += kThreads / kSplitThreads) work(c);
        done(r0);
    }
}

// The chunks of a split form of a pass without partials (AdamW): the CTA's
// kThreads / NT parts take chunks c0 + P b + h, then every P gridDim.x (P parts,
// CTA b, part h).
template <int NT, class Work>
__device__ __forceinline__ void for_split_chunks(int64_t c0, int64_t c1, Work work) {
    constexpr int P = kThreads / NT;
    const int h = threadIdx.x / NT;
    for (int64_t c = c0 + int64_t(blockIdx.x) * P + h; c < c1; c += int64_t(gridDim.x) * P) work(c);
}

// The whole-CTA chunks of a persistent CTA (c0 + blockIdx.x, then every gridDim.x),
// each descriptor handed to work(c, ch).  With PF the next descriptor is loaded
// into registers before the current chunk is worked, so that its load overlaps the
// work instead of heading the next chunk's chain of dependent loads.  The AdamW
// kernels take it (4 % faster on the 1.24B list); in the accumulation kernels it
// measured no gain and costs registers the two-list forms do not have.
template <bool PF, class Work>
__device__ __forceinline__ void for_chunks(const Chunk* __restrict__ chunks, int64_t c0, int64_t c1, Work work) {
    if (PF) {
        int64_t c = c0 + blockIdx.x;
        if (c >= c1) return;
        Chunk cur = chunks[c];
        for (;;) {
            const int64_t cn = c + gridDim.x;
            Chunk nxt = cur;
            if (cn < c1) nxt = chunks[cn];
            work(c, cur);
            if (cn >= c1) break;
            c = cn;
            cur = nxt;
        }
    } else {
        for (int64_t c = c0 + blockIdx.x; c < c1; c += gridDim.x) work(c, chunks[c]);
    }
}

template <int NT, int GDT, bool FIRST>
__global__ void __launch_bounds__(kThreads, FIRST ? TL_MINB_ACC_FIRST : TL_MINB_ACC)
k_accumulate(const Chunk* __restrict__ chunks, int64_t c0, int64_t c1,
             const __grid_constant__ GradTable inl,
             const void* const* __restrict__ gtab, float w) {
    const void* const* gp = gtab != nullptr ? gtab : inl.p;
    if (NT == kThreads) {
        for_chunks<false>(chunks, c0, c1, [&](int64_t, const Chunk& ch) {
            accumulate_segment<kThreads, GDT, FIRST>(ch, threadIdx.x, gp, w);
        });
        return;
    }
    for (int64_t c = c0 + blockIdx.x; c < c1; c += gridDim.x) {
        accumulate_segment<32, GDT, FIRST>(group_segment(chunks, c0, c), threadIdx.x & 31, gp, w);
    }
}

// ---------------------------------------------------------------------------
// a3: last micro-batch + unscale + overflow check + squared-norm partial.
// [MEG] section 8 (cast, divide by the loss scale, place in the fp32 buffer),
// section 6 (overflow flag), section 9 (sum of squares); [MP] section 2 "Loss
// scaling" (S a power of two: exact).  The fp32 squares are summed per thread
// (SumSq below), then per warp in a fixed butterfly; each warp writes one fp64
// partial per chunk, so there are no atomics and no block barrier.
// ---------------------------------------------------------------------------
template <int MODE>
__device__ __forceinline__ float unscale1(float a, float gj, float w, float inv_s) {
    if (MODE == kAccOnly) return __fmul_rn(a, inv_s);
    if (MODE == kFirstOnly) return __fmul_rn(__fmul_rn(w, gj), inv_s);
    return __fmul_rn(__fmaf_rn(w, gj, a), inv_s);
}

// Sum of the fp32 squares fl32(u*u) of one chunk without fp64 arithmetic in the
// element loop (fp64 throughput is scarce on this part).  Ordinary values
// (|u| < 2^56: every square is below 2^112, so no fp32 sum over a chunk can
// overflow) are added into a float-float accumulator (hi, lo) with the
// error-free TwoSum transformation, so a chunk partial is accurate to about
// 1e-13 relative and the fp32 norm almost always rounds exactly as an fp64 sum
// of the same squares does.  (A plain fp32 tree is not enough: it moves the
// fp32 norm by an ulp, hence the clip coefficient, hence masters close to zero
// by many ulps.)  A vector holding a larger or infinite value is summed in fp64
// instead, so the total is infinite exactly when some fp32 square is; NaN
// propagates through the float-float path, and a NaN accumulator at the end of
// a warp's run raises the overflow flag (so the vector path checks no value one
// by one unless the vector holds a large one).
// d + q in fp64 for the rare large-value case of the squared-norm sum, kept out
// of line: inlined into a per-element loop it may be if-converted, and then every
// element issues the fp64 instructions, which this GPU runs at a small fraction
// of the fp32 rate.
__device__ __noinline__ double dadd_out_of_line(double d, float q) {
    return __dadd_rn(d, static_cast<double>(q));
}

// Two fp32 lanes per instruction (sm_100 and later): each lane rounds as the
// scalar instruction does.
__device__ __forceinline__ void add2_rn(float a0, float a1, float b0, float b1, float& d0, float& d1) {
    asm("{ .reg .b64 a, b, d; mov.b64 a, {%2, %3}; mov.b64 b, {%4, %5}; add.rn.f32x2 d, a, b; mov.b64 {%0, %1}, d; }"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2_rn(float a0, float a1, float b0, float b1, float& d0, float& d1) {
    asm("{ .reg .b64 a, b, d; mov.b64 a, {%2, %3}; mov.b64 b, {%4, %5}; sub.rn.f32x2 d, a, b; mov.b64 {%0, %1}, d; }"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul2_rn(float a0, float a1, float b0, float b1, float& d0, float& d1) {
    asm("{ .reg .b64 a, b, d; mov.b64 a, {%2, %3}; mov.b64 b, {%4, %5}; mul.rn.f32x2 d, a, b; mov.b64 {%0, %1}, d; }"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void fma2_rn(float a0, float a1, float b0, float b1, float c0, float c1, float& d0, float& d1) {
    asm("{ .reg .b64 a, b, c, d; mov.b64 a, {%2, %3}; mov.b64 b, {%4, %5}; mov.b64 c, {%6, %7}; "
        "fma.rn.f32x2 d, a, b, c; mov.b64 {%0, %1}, d; }"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// P = false: one float-float accumulator (hi0, lo0) per lane.  P = true: two,
// (hi0, lo0) for the even and (hi1, lo1) for the odd elements of the lane's
// vectors, updated together by two-lane instructions (about half the
// instructions per element, two more registers; a scalar element goes to the
// first).
template <bool P>
struct SumSqT {
    float hi0 = 0.0f, hi1 = 0.0f;
    float lo0 = 0.0f, lo1 = 0.0f;
    double d = 0.0;   // vectors with large values only
    bool big = false;

    __device__ __forceinline__ void add(float q) {
        const float s = __fadd_rn(hi0, q);
        const float bb = __fsub_rn(s, hi0);
        const float err = __fadd_rn(__fsub_rn(hi0, __fsub_rn(s, bb)), __fsub_rn(q, bb));  // hi + q - s, exactly
        hi0 = s;
        lo0 = __fadd_rn(lo0, err);
    }
    // TwoSum of (q0, q1) into the two accumulators (P), or of q0 then q1 into the one
    __device__ __forceinline__ void add2(float q0, float q1) {
        if constexpr (P) {
            float s0, s1, b0, b1, t0, t1, e0, e1, f0, f1;
            add2_rn(hi0, hi1, q0, q1, s0, s1);
            sub2_rn(s0, s1, hi0, hi1, b0, b1);
            sub2_rn(s0, s1, b0, b1, t0, t1);
            sub2_rn(hi0, hi1, t0, t1, e0, e1);
            sub2_rn(q0, q1, b0, b1, f0, f1);
            add2_rn(e0, e1, f0, f1, e0, e1);
            hi0 = s0;
            hi1 = s1;
            add2_rn(lo0, lo1, e0, e1, lo0, lo1);
        } else {
            add(q0);
            add(q1);
        }
    }
    // Eight values of u.  When every |u| is below 2^56 their squares (below 2^112,
    // so a lane's sum stays finite) go to the float-float accumulators; a NaN among
    // them is not looked for here: it makes the accumulator NaN, which nan() reports
    // when the warp finishes.  Otherwise (a large or infinite value, or a NaN beside
    // one) the squares are summed in fp64 and each value is checked: bad is raised
    // for a value that is not finite.
    __device__ __forceinline__ void vec8(const float (&u)[8], bool& bad) {
        const float um = fmaxf(fmaxf(fmaxf(fabsf(u[0]), fabsf(u[1])), fmaxf(fabsf(u[2]), fabsf(u[3]))),
                               fmaxf(fmaxf(fabsf(u[4]), fabsf(u[5])), fmaxf(fabsf(u[6]), fabsf(u[7]))));
        if (!(um < 72057594037927936.0f)) {  // 2^56 or inf (fmaxf drops NaN unless all are)
            big = true;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                bad |= !isfinite(u[e]);
                d = __dadd_rn(d, static_cast<double>(__fmul_rn(u[e], u[e])));
            }
            return;
        }
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            float q0, q1;
            if constexpr (P) {
                mul2_rn(u[e], u[e + 1], u[e], u[e + 1], q0, q1);
            } else {
                q0 = __fmul_rn(u[e], u[e]);
                q1 = __fmul_rn(u[e + 1], u[e + 1]);
            }
            add2(q0, q1);
        }
    }
    // A NaN reached the float-float accumulators (once NaN, hi stays NaN).
    __device__ __forceinline__ bool nan() const { return isnan(hi0) || (P && isnan(hi1)); }
    __device__ __forceinline__ void one(float u) {
        const float q = __fmul_rn(u, u);
        if (fabsf(u) >= 72057594037927936.0f) {
            big = true;
            d = dadd_out_of_line(d, q);
            return;
        }
        add(q);
    }
};
using SumSq = SumSqT<TL_SQ_PAIRS != 0>;

// Fixed-order reduction of a SumSq within a warp: a float-float butterfly
// (TwoSum gives the same exact error term in both lanes of a pair, so every lane
// ends with the same value), fp64 only in a warp that saw a large value.  Each
// warp writes its own partial (kGroup partials per chunk), so finishing a chunk
// needs no block barrier; the partial of warp w of chunk c is always the same
// elements' sum, whatever the grid.
template <bool P>
__device__ __forceinline__ double warp_sumsq(const SumSqT<P>& acc) {
    float hi = acc.hi0, lo = acc.lo0;
    if (P) {
        const float s = __fadd_rn(acc.hi0, acc.hi1);
        const float bb = __fsub_rn(s, acc.hi0);
        const float err = __fadd_rn(__fsub_rn(acc.hi0, __fsub_rn(s, bb)), __fsub_rn(acc.hi1, bb));
        hi = s;
        lo = __fadd_rn(__fadd_rn(acc.lo0, acc.lo1), err);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, hi, o);
        const float ol = __shfl_xor_sync(0xffffffffu, lo, o);
        const float s = __fadd_rn(hi, oh);
        const float bb = __fsub_rn(s, hi);
        const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(oh, bb));
        hi = s;
        lo = __fadd_rn(__fadd_rn(lo, ol), err);
    }
    double d = 0.0;
    if (__any_sync(0xffffffffu, acc.big)) {
        d = acc.d;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) d = __dadd_rn(d, __shfl_xor_sync(0xffffffffu, d, o));
    }
    return __dadd_rn(__dadd_rn(static_cast<double>(hi), static_cast<double>(lo)), d);
}

// The squared-norm partials of a run (its first chunk c) in the contexts that keep
// one slot per warp: warp w writes slot c * kGroup + w, and raises the overflow flag
// if any lane saw a non-finite value.  No barrier: the warps of a CTA never wait for
// each other at the end of a run.
template <bool P>
__device__ __forceinline__ void finish_warp(const SumSqT<P>& sq, bool bad, int64_t c, DevState* st, double* partials) {
    const double part = warp_sumsq(sq);
    const bool any_bad = __any_sync(0xffffffffu, bad || sq.nan());
    if ((threadIdx.x & 31) == 0) {
        partials[c * kGroup + (threadIdx.x >> 5)] = part;
        if (any_bad) st->found_inf = 1;
    }
}

// The squared-norm partial of a run (slot c, its first chunk) in the contexts with
// one slot per run: each warp's sum
// reduced by the fixed butterfly above, then the CTA's warps added in warp order by
// thread 0 after one block barrier (every thread of the CTA ends each of its runs
// together), one fp64 slot per run.  The warp sums sit in one of two shared buffers
// by run parity, so the next run's writes never meet thread 0's reads and one
// barrier per run suffices (the other warps go on with the next run meanwhile).  A warp that saw a non-finite value raises the overflow flag.
template <bool P>
__device__ __forceinline__ void finish_run(const SumSqT<P>& sq, bool bad, int64_t c, int parity, DevState* st,
                                           double* partials) {
    __shared__ double part_w[2][kThreads / 32];
    const double part = warp_sumsq(sq);
    const bool any_bad = __any_sync(0xffffffffu, bad || sq.nan());
    if ((threadIdx.x & 31) == 0) {
        part_w[parity][threadIdx.x >> 5] = part;
        if (any_bad) st->found_inf = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double x = part_w[parity][0];
#pragma unroll
        for (int k = 1; k < kThreads / 32; ++k) x = __dadd_rn(x, part_w[parity][k]);
        partials[c] = x;
    }
}

// The end of a partial-writing launch that finishes the norm itself (fin > 0 slots):
// every CTA, when its chunks are done, publishes its partials and overflow flags
// (a fence per warp) and takes a ticket; the CTA holding the launch's last ticket
// then reduces every partial slot of the table (those of earlier launches of the
// pass included: they completed before this launch began) in a fixed order: thread
// t sums slots t, t + 256, t + 512, ... (coalesced, 8 loads in flight) into eight
// accumulators, slot j going to accumulator (j / 256) mod 8, then the accumulators
// in order and the fixed block reduction.  The order depends on the number of
// slots only, not on the grid.  Nothing waits: the last CTA only runs once every
// other CTA has published.  The ticket counter is reset by the last CTA.
__device__ __noinline__ void finish_pass(DevState* __restrict__ st, const double* __restrict__ partials,
                                         int64_t nslots) {
    __shared__ double red[kThreads / 32];
    __shared__ int last;
    if ((threadIdx.x & 31) == 0) __threadfence();   // this warp's partials and flag, device-wide
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t ticket = atomicAdd(&st->pass_ticket, 1u);
        last = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    constexpr int kBatch = 8;
    double a8[8] = {0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0};
    int64_t j = threadIdx.x;
    for (; j + (kBatch - 1) * kThreads < nslots; j += kBatch * kThreads) {
        double x[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) x[q] = __ldcg(partials + j + q * kThreads);   // written by other SMs
#pragma unroll
        for (int q = 0; q < kBatch; ++q) a8[q & 7] = __dadd_rn(a8[q & 7], x[q]);
    }
    for (int q = 0; j < nslots; j += kThreads, ++q) a8[q & 7] = __dadd_rn(a8[q & 7], __ldcg(partials + j));
    double s = 0.0;
#pragma unroll
    for (int q = 0; q < 8; ++q) s = __dadd_rn(s, a8[q]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __dadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double v = 0.0;
#pragma unroll
        for (int k = 0; k < kThreads / 32; ++k) v = __dadd_rn(v, red[k]);
        st->pass_ticket = 0;
        st->sumsq = v;
        if (!isfinite(v)) st->found_inf = 1;   // an fp32 square overflowed: treated as an overflow
        st->norm = __double2float_rn(__dsqrt_rn(v));
    }
}

template <int NT, int GDT, int MODE>
__device__ __forceinline__ void unscale_segment(const Chunk& ch, int t, const void* const* gp, float w, float inv_s,
                                                SumSq& sq, bool& bad) {
    constexpr bool kReadG = MODE != kAccOnly;
    constexpr bool kReadAcc = MODE != kFirstOnly;
    float* __restrict__ acc0 = ch.acc;
    const void* gb = kReadG ? gp[ch.tensor] : nullptr;
    const char* g0 = kReadG ? static_cast<const char*>(gb) + ch.start * Grad<GDT>::kBytes : nullptr;
    const float* sc = kReadG ? grad_scales<GDT>(gb, ch) : nullptr;
    const int len = ch.len;
    VecPlan pl{0, false, false};
    if (aligned16(acc0) && (!kReadG || aligned16(g0))) pl = VecPlan{0, true, aligned32(acc0)};
    else if (!kReadG || ephase<4>(acc0) == ephase<Grad<GDT>::kBytes>(g0)) pl = VecPlan{(8 - ephase<4>(acc0)) & 7, true, true};
    if (kReadG && GDT == kE4M3 && pl.head != 0) pl.vec = false;  // an 8-bit vector must not straddle two blocks
    int head = 0, done = 0;
    if constexpr (GDT == kE4M3 && NT == kThreads && TL_E4M3_BLOCKS) {
        // 8-bit lists, every stream 16-byte aligned: whole 16-element blocks, one
        // scale and 16 codes per load (the lanes take the elements as k_accum_many
        // does, so that both give the same partials)
        if (pl.vec && aligned16(acc0) && (!kReadG || aligned16(g0))) {
            const int nb = len / 16;
            for (int i = t; i < nb; i += NT) {
                float ax[2][8];
                uint4 c = make_uint4(0u, 0u, 0u, 0u);
                float sb = 0.0f;
                if (kReadG) {
                    c = __ldg(reinterpret_cast<const uint4*>(g0) + i);
                    sb = __ldg(sc + i);
                }
                if (kReadAcc) {
                    ld8_f32(acc0 + 16 * i, ax[0], pl.wide);
                    ld8_f32(acc0 + 16 * i + 8, ax[1], pl.wide);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const GradRaw<kE4M3>::T r{h == 0 ? make_uint2(c.x, c.y) : make_uint2(c.z, c.w), sb};
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        ax[h][e] = unscale1<MODE>(kReadAcc ? ax[h][e] : 0.0f, kReadG ? GradRaw<kE4M3>::at(r, e) : 0.0f,
                                                  w, inv_s);
                    sq.vec8(ax[h], bad);
                }
                st8_f32(acc0 + 16 * i, ax[0], pl.wide);
                st8_f32(acc0 + 16 * i + 8, ax[1], pl.wide);
            }
            done = nb * 16;
            pl.vec = false;
        }
    }
    if (pl.vec) {
        head = min(pl.head, len);
        const bool wide = pl.wide;
        float* __restrict__ acc = acc0 + head;
        const void* g = kReadG ? g0 + head * Grad<GDT>::kBytes : nullptr;
        const int nv = (len - head) / kVec;
        int i = t;
        for (; i + (kUnroll - 1) * NT < nv; i += kUnroll * NT) {
            float gx[kUnroll][8], ax[kUnroll][8];
            if (kReadG) {
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) Grad<GDT>::ld8(g, int64_t(i + u * NT) * kVec, gx[u], sc);
            }
            if (kReadAcc) {
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) ld8_f32(acc + (i + u * NT) * kVec, ax[u], wide);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    ax[u][e] = unscale1<MODE>(kReadAcc ? ax[u][e] : 0.0f, kReadG ? gx[u][e] : 0.0f, w, inv_s);
                sq.vec8(ax[u], bad);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) st8_f32(acc + (i + u * NT) * kVec, ax[u], wide);
        }
        for (; i < nv; i += NT) {
            float gx[8], ax[8];
            if (kReadG) Grad<GDT>::ld8(g, int64_t(i) * kVec, gx, sc);
            if (kReadAcc) ld8_f32(acc + i * kVec, ax, wide);
#pragma unroll
            for (int e = 0; e < 8; ++e) ax[e] = unscale1<MODE>(kReadAcc ? ax[e] : 0.0f, kReadG ? gx[e] : 0.0f, w, inv_s);
            sq.vec8(ax, bad);
            st8_f32(acc + i * kVec, ax, wide);
        }
        done = head + nv * kVec;
    }
    auto one = [&](int j) {
        const float u = unscale1<MODE>(kReadAcc ? acc0[j] : 0.0f, kReadG ? Grad<GDT>::ld1(g0, j, sc) : 0.0f, w, inv_s);
        acc0[j] = u;
        bad |= !isfinite(u);
        sq.one(u);
    };
    for (int j = t; j < head; j += NT) one(j);          // head
    // tail, or the whole segment without a vector part: kScalar elements per
    // thread loaded first, then finished in element order
    int j = done + t;
    for (; j + (kScalar - 1) * NT < len; j += kScalar * NT) {
        float ax[kScalar], gx[kScalar];
#pragma unroll
        for (int q = 0; q < kScalar; ++q) {
            ax[q] = kReadAcc ? acc0[j + q * NT] : 0.0f;
            gx[q] = kReadG ? Grad<GDT>::ld1(g0, j + q * NT, sc) : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < kScalar; ++q) {
            const float u = unscale1<MODE>(ax[q], gx[q], w, inv_s);
            acc0[j + q * NT] = u;
            bad |= !isfinite(u);
            sq.one(u);
        }
    }
    for (; j < len; j += NT) one(j);
}

template <int NT, int GDT, int MODE>
__global__ void __launch_bounds__(kThreads, NT != 32 && GDT != kF32 ? 3 : 2)
k_unscale(const Chunk* __restrict__ chunks, int64_t c0, int64_t c1, int run,
          const __grid_constant__ GradTable inl,
          const void* const* __restrict__ gtab, float w, DevState* __restrict__ st, double* __restrict__ partials,
          int64_t fin) {
    const void* const* gp = gtab != nullptr ? gtab : inl.p;
    const float inv_s = __fdiv_rn(1.0f, st->S);
    SumSq sq;
    bool bad = false;
    int nrun = 0;   // runs finished by this CTA (the parity of finish_run's buffer)
    const bool run_slots = st->run_slots != 0;
    for_runs_nt<NT>(c0, c1, run, [&](int64_t c) {
        if (NT != 32) unscale_segment<NT, GDT, MODE>(chunks[c], threadIdx.x % NT, gp, w, inv_s, sq, bad);
        else unscale_segment<32, GDT, MODE>(group_segment(chunks, c0, c), threadIdx.x & 31, gp, w, inv_s, sq, bad);
    }, [&](int64_t r0) {
        if (run_slots) finish_run(sq, bad, r0, nrun++ & 1, st, partials);
        else finish_warp(sq, bad, r0, st, partials);
        sq = SumSq();
        bad = false;
    });
    if (fin > 0) finish_pass(st, partials, fin);
}

// ---------------------------------------------------------------------------
// a2 + a3 over resident micro-batches: up to kMaxMany gradient lists read in one
// pass.  Per element the operations are those of the per-micro-batch kernels in
// the same order (acc = w_1 g_1, then acc = fma(w_i, g_i, acc), then u = acc/S),
// so the result is bit-identical; acc is written once (as u when LAST) instead
// of once per micro-batch.  FIRST: no partial sum in acc yet.  LAST: finish
// with the unscale, overflow check and squared-norm partial of a3.
// ---------------------------------------------------------------------------
// acc = w_0 g_0 + w_1 g_1 + ... (per element in list order) over one 8-element vector
// of each of the kk lists, then (LAST) the unscale and the overflow / squared-norm
// bookkeeping of the last micro-batch
template <int GDT, bool FIRST, bool LAST, int KM, class SQ>
__device__ __forceinline__ void mix_lists(const typename GradRaw<GDT>::T (&raw)[KM], const ManyArgs& a, int kk,
                                          float inv_s, SQ& sq, bool& bad, float (&ax)[8]) {
    if constexpr (GDT == kE4M3 && TL_PAIRS) {
        // 8-bit lists (issue-bound): decode two codes at a time and take the scale
        // product and the weighted sum two lanes per instruction
#pragma unroll
        for (int q = 0; q < KM; ++q)
            if (q == 0 || q < kk) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t wd = k < 2 ? raw[q].c.x : raw[q].c.y;
                    float lo, hi;
                    unpack_e4m3x2((k & 1) ? (wd >> 16) : wd, lo, hi);
                    mul2_rn(lo, hi, raw[q].s, raw[q].s, lo, hi);      // code value x block scale
                    if (q == 0 && FIRST) mul2_rn(a.w[0], a.w[0], lo, hi, ax[2 * k], ax[2 * k + 1]);
                    else fma2_rn(a.w[q], a.w[q], lo, hi, ax[2 * k], ax[2 * k + 1], ax[2 * k], ax[2 * k + 1]);
                }
            }
    } else if constexpr (TL_PAIRS) {
        // the weighted sum two lanes per instruction (elements 2k and 2k + 1)
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const float x0 = GradRaw<GDT>::at(raw[0], e), x1 = GradRaw<GDT>::at(raw[0], e + 1);
            if (FIRST) mul2_rn(a.w[0], a.w[0], x0, x1, ax[e], ax[e + 1]);
            else fma2_rn(a.w[0], a.w[0], x0, x1, ax[e], ax[e + 1], ax[e], ax[e + 1]);
        }
#pragma unroll
        for (int q = 1; q < KM; ++q)
            if (q < kk) {
#pragma unroll
                for (int e = 0; e < 8; e += 2)
                    fma2_rn(a.w[q], a.w[q], GradRaw<GDT>::at(raw[q], e), GradRaw<GDT>::at(raw[q], e + 1), ax[e],
                            ax[e + 1], ax[e], ax[e + 1]);
            }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            ax[e] = FIRST ? __fmul_rn(a.w[0], GradRaw<GDT>::at(raw[0], e))
                          : __fmaf_rn(a.w[0], GradRaw<GDT>::at(raw[0], e), ax[e]);
#pragma unroll
        for (int q = 1; q < KM; ++q)
            if (q < kk) {
#pragma unroll
                for (int e = 0; e < 8; ++e) ax[e] = __fmaf_rn(a.w[q], GradRaw<GDT>::at(raw[q], e), ax[e]);
            }
    }
    if (LAST) {
#pragma unroll
        for (int e = 0; e < 8; e += 2) mul2_rn(ax[e], ax[e + 1], inv_s, inv_s, ax[e], ax[e + 1]);
        sq.vec8(ax, bad);
    }
}

template <int NT, int GDT, bool FIRST, bool LAST, int KM, bool STORE, bool ROT, class SQ>
__device__ __forceinline__ void many_segment(const Chunk& ch, int t, const GradTableMany& inl, const ManyArgs& a,
                                             float inv_s, SQ& sq, bool& bad) {
    const int kk = a.k;
    float* __restrict__ acc0 = ch.acc;
    const char* g[KM];
    // 8-bit gradients: the block scales of list q start soff bytes after its codes (the
    // same offset for every list: it depends on the tensor and the segment only)
    const int64_t soff = GDT == kE4M3 ? ch.gscale - ch.start + (ch.start >> 2) : 0;
    auto gs = [&](int q) { return GDT == kE4M3 ? reinterpret_cast<const float*>(g[q] + soff) : nullptr; };
    // without the store of u the accumulation buffer is not touched: the lists
    // alone decide the vector plan
    bool al = !STORE || aligned16(acc0);
    bool same = true;
    int r = STORE ? ephase<4>(acc0) : 0;
#pragma unroll
    for (int q = 0; q < KM; ++q) {
        if (q < kk) {
            const void* base = a.tabs[q] != nullptr ? a.tabs[q][ch.tensor] : inl.p[q * a.ntensors + ch.tensor];
            g[q] = static_cast<const char*>(base) + ch.start * Grad<GDT>::kBytes;
            if (!STORE && q == 0) r = ephase<Grad<GDT>::kBytes>(g[0]);
            al = al && aligned16(g[q]);
            same = same && ephase<Grad<GDT>::kBytes>(g[q]) == r;
        } else {
            g[q] = nullptr;
        }
    }
    const int len = ch.len;
    VecPlan pl{0, false, false};
    if (al) pl = VecPlan{0, true, !STORE || aligned32(acc0)};
    else if (same) pl = VecPlan{(8 - r) & 7, true, true};
    if (GDT == kE4M3 && pl.head != 0) pl.vec = false;  // an 8-bit vector must not straddle two blocks
    int head = 0, done = 0;
    if constexpr (GDT == kE4M3 && NT == kThreads && TL_E4M3_BLOCKS) {
        // 8-bit lists, every stream 16-byte aligned: whole 16-element blocks, one
        // scale and 16 codes per list and load, each half as one 8-element vector (the
        // lanes take the elements as k_unscale does, so that both give the same partials)
        if (pl.vec && al) {
            const int nb = len / 16;
            for (int i = t; i < nb; i += NT) {
                typename GradRaw<GDT>::T lo[KM], hi[KM];
#pragma unroll
                for (int q = 0; q < KM; ++q)
                    if (q < kk) {
                        const uint4 c = __ldg(reinterpret_cast<const uint4*>(g[q]) + i);
                        const float sb = __ldg(gs(q) + i);
                        lo[q] = typename GradRaw<GDT>::T{make_uint2(c.x, c.y), sb};
                        hi[q] = typename GradRaw<GDT>::T{make_uint2(c.z, c.w), sb};
                    }
                float a0[8], a1[8];
                if (!FIRST) {
                    ld8_f32(acc0 + 16 * i, a0, pl.wide);
                    ld8_f32(acc0 + 16 * i + 8, a1, pl.wide);
                }
                mix_lists<GDT, FIRST, LAST>(lo, a, kk, inv_s, sq, bad, a0);
                mix_lists<GDT, FIRST, LAST>(hi, a, kk, inv_s, sq, bad, a1);
                if (STORE) {
                    st8_f32(acc0 + 16 * i, a0, pl.wide);
                    st8_f32(acc0 + 16 * i + 8, a1, pl.wide);
                }
            }
            done = nb * 16;
            pl.vec = false;
        }
    }
    // streams of unequal phase (16-bit lists, whole-CTA segments): rotated vectors in
    // the frame of the accumulation buffer (or of list 0 when it is not written)
    constexpr bool kRotForm = ROT && NT != 32 && KM <= kFewLists && (GDT == kBF16 || GDT == kF16);
    const bool rot = kRotForm && !pl.vec;
    const int fr = STORE ? ephase<4>(acc0) : ephase<2>(g[0]);
    if (rot) pl = VecPlan{(8 - fr) & 7, true, true};
    if constexpr (kRotForm) {
      if (rot) {
        head = min(pl.head, len);
        const int nv = (len - head) / kVec;
        const int lane = t & 31;
        int dq[KM];
#pragma unroll
        for (int q = 0; q < KM; ++q) dq[q] = q < kk ? (ephase<2>(g[q]) - fr) & 7 : 0;
        for (int base = (t >> 5) * kRotLanes; base < nv; base += (NT / 32) * kRotLanes) {   // warp-uniform trips
            const int i = base + lane;
            const bool act = lane < kRotLanes && i < nv;
            const bool ld = i <= nv;
            const int o = head + i * kVec;
            typename GradRaw<GDT>::T raw[KM];
#pragma unroll
            for (int q = 0; q < KM; ++q)
                if (q < kk) raw[q] = ld16_rot(reinterpret_cast<const unsigned short*>(g[q]), o, dq[q], act, ld);
            if (act) {
                float ax[8];
                if (!FIRST) ld8_f32(acc0 + o, ax, true);
                mix_lists<GDT, FIRST, LAST>(raw, a, kk, inv_s, sq, bad, ax);
                if (STORE) st8_f32(acc0 + o, ax, true);
            }
        }
        done = head + nv * kVec;
      }
    }
    if (!rot && pl.vec) {
        head = min(pl.head, len);
        const bool wide = pl.wide;
        float* __restrict__ acc = acc0 + head;
        const int gofs = head * Grad<GDT>::kBytes;
        const int nv = (len - head) / kVec;
        auto mix = [&](const typename GradRaw<GDT>::T (&raw)[KM], float (&ax)[8]) {
            mix_lists<GDT, FIRST, LAST>(raw, a, kk, inv_s, sq, bad, ax);
        };
        for (int i = t; i < nv; i += NT) {
            // all kk loads in flight first; each stream's 8 values are unpacked
            // inside the multiply-add chain (per element still q = 0, 1, ... in order)
            typename GradRaw<GDT>::T raw[KM];
#pragma unroll
            for (int q = 0; q < KM; ++q)
                if (q < kk) raw[q] = GradRaw<GDT>::ld(g[q] + gofs, int64_t(i) * kVec, gs(q));
            float ax[8];
            if (!FIRST) ld8_f32(acc + i * kVec, ax, wide);
            mix(raw, ax);
            if (STORE) st8_f32(acc + i * kVec, ax, wide);
        }
        done = head + nv * kVec;
    }
    auto one = [&](int j) {
        float v = FIRST ? __fmul_rn(a.w[0], Grad<GDT>::ld1(g[0], j, gs(0)))
                        : __fmaf_rn(a.w[0], Grad<GDT>::ld1(g[0], j, gs(0)), acc0[j]);
#pragma unroll
        for (int q = 1; q < KM; ++q)
            if (q < kk) v = __fmaf_rn(a.w[q], Grad<GDT>::ld1(g[q], j, gs(q)), v);
        if (LAST) {
            v = __fmul_rn(v, inv_s);
            bad |= !isfinite(v);
            sq.one(v);
        }
        if (STORE) acc0[j] = v;
    };
    for (int j = t; j < head; j += NT) one(j);          // head
    // tail, or the whole segment without a vector part: with one or two lists,
    // S elements per thread loaded first, then finished in element order (more
    // lists already put that many loads in flight)
    constexpr int S = KM <= kFewLists ? (NT != 32 ? TL_SCALAR_FEW : TL_SCALAR_FEW_GROUP) : TL_SCALAR_MANY;
    int j = done + t;
    for (; S > 1 && j + (S - 1) * NT < len; j += S * NT) {
        float gx[S][KM], ax[S];
#pragma unroll
        for (int e = 0; e < S; ++e) {
#pragma unroll
            for (int q = 0; q < KM; ++q)
                if (q < kk) gx[e][q] = Grad<GDT>::ld1(g[q], j + e * NT, gs(q));
            if (!FIRST) ax[e] = acc0[j + e * NT];
        }
#pragma unroll
        for (int e = 0; e < S; ++e) {
            float v = FIRST ? __fmul_rn(a.w[0], gx[e][0]) : __fmaf_rn(a.w[0], gx[e][0], ax[e]);
#pragma unroll
            for (int q = 1; q < KM; ++q)
                if (q < kk) v = __fmaf_rn(a.w[q], gx[e][q], v);
            if (LAST) {
                v = __fmul_rn(v, inv_s);
                bad |= !isfinite(v);
                sq.one(v);
            }
            if (STORE) acc0[j + e * NT] = v;
        }
    }
    for (; j < len; j += NT) one(j);
}

// ROT: the form for lists of unequal element phase (rotated 16-bit loads; the
// registers they need cost it one resident CTA per SM).
template <int NT, int GDT, bool FIRST, bool LAST, int KM, bool STORE, bool ROT>
__global__ void __launch_bounds__(kThreads, NT == 32 ? (GDT == kF32 || KM > kFewLists ? 1 : GDT == kE4M3 ? TL_MINB_GROUP_FEW - 1 : TL_MINB_GROUP_FEW)
                                            : GDT == kF32 ? 2
                                            : KM <= kFewLists ? (GDT == kE4M3 || (LAST && !FIRST) || ROT ? TL_MINB_FEW - 1 : TL_MINB_FEW)
                                            : GDT == kE4M3 ? TL_MINB_MANY_E4M3 : TL_MINB_MANY)
k_accum_many(const Chunk* __restrict__ chunks, int64_t c0, int64_t c1, int run,
             const __grid_constant__ GradTableMany inl,
             const __grid_constant__ ManyArgs a, DevState* __restrict__ st, double* __restrict__ partials,
             int64_t fin) {
    const float inv_s = LAST ? __fdiv_rn(1.0f, st->S) : 1.0f;
    // (one accumulator structure in every partial-writing kernel: the passes that
    // reach the same u give the same norm bit for bit)
    SumSqT<TL_SQ_PAIRS != 0> sq;
    bool bad = false;
    int nrun = 0;   // runs finished by this CTA (the parity of finish_run's buffer)
    const bool run_slots = st->run_slots != 0;
    for_runs_nt<NT>(c0, c1, run, [&](int64_t c) {
        if (NT != 32)
            many_segment<NT, GDT, FIRST, LAST, KM, STORE, ROT>(chunks[c], threadIdx.x % NT, inl, a, inv_s, sq, bad);
        else
            many_segment<32, GDT, FIRST, LAST, KM, STORE, false>(group_segment(chunks, c0, c), threadIdx.x & 31, inl, a,
                                                          inv_s, sq, bad);
    }, [&](int64_t r0) {
        if (LAST) {
            if (run_slots) finish_run(sq, bad, r0, nrun++ & 1, st, partials);
            else finish_warp(sq, bad, r0, st, partials);
            sq = decltype(sq)();
            bad = false;
        }
    });
    if (LAST && fin > 0) finish_pass(st, partials, fin);
}

// ---------------------------------------------------------------------------
// a4: deterministic second stage.  [MEG] section 9: global_norm =
// sqrt(sum ||g||^2), clip_coef = max_norm / (global_norm + eps), applied only
// below 1 (eps = 1e-6).  kNormBlocks CTAs each reduce a fixed contiguous range
// of the partial slots (per thread eight interleaved accumulators, then a
// fixed butterfly and a fixed warp-order sum) into one slot.  Each CTA then
// takes a ticket; the CTA holding the last ticket of the launch adds the slots
// in slot order and finishes.  Nothing waits: the last CTA only runs after every
// other CTA has published its slot.  The ticket counter is never reset; the
// launch's last ticket is the one that is kNormBlocks - 1 modulo kNormBlocks.
// ---------------------------------------------------------------------------
__device__ __forceinline__ double block_sum(double s, double* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __dadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int k = 0; k < kNormThreads / 32; ++k) t = __dadd_rn(t, red[k]);
    }
    return t;
}

__global__ void __launch_bounds__(kNormThreads)
k_norm(const double* __restrict__ partials, int64_t n, double* __restrict__ slots, DevState* __restrict__ st,
       float max_norm) {
    __shared__ double red[kNormThreads / 32];
    __shared__ bool last;
    const int64_t per = (n + kNormBlocks - 1) / kNormBlocks;
    const int64_t lo = min(n, per * blockIdx.x);
    const int64_t hi = min(n, lo + per);
    double acc8[8] = {0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0};
    int64_t i = lo + threadIdx.x;
    for (; i + 7 * kNormThreads < hi; i += 8 * kNormThreads) {
        double x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = partials[i + q * kNormThreads];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc8[q] = __dadd_rn(acc8[q], x[q]);
    }
    double s = 0.0;
    for (; i < hi; i += kNormThreads) s = __dadd_rn(s, partials[i]);  // the last < 8 rounds
#pragma unroll
    for (int q = 0; q < 8; ++q) s = __dadd_rn(s, acc8[q]);
    s = block_sum(s, red);
    if (threadIdx.x == 0) {
        slots[blockIdx.x] = s;
        __threadfence();
        const uint32_t ticket = atomicAdd(&st->norm_ticket, 1u);
        last = (ticket % kNormBlocks) == kNormBlocks - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    double v = threadIdx.x < kNormBlocks ? __ldcg(slots + threadIdx.x) : 0.0;  // slots written by other SMs
    v = block_sum(v, red);
    if (threadIdx.x == 0) {
        st->sumsq = v;
        if (!isfinite(v)) st->found_inf = 1;   // an fp32 square overflowed: treated as an overflow
        const float norm = __double2float_rn(__dsqrt_rn(v));
        st->norm = norm;
        float coef = 1.0f;
        if (max_norm > 0.0f) {
            const float cc = __fdiv_rn(max_norm, __fadd_rn(norm, 1e-6f));
            if (cc < 1.0f) coef = cc;
        }
        st->coef = coef;
    }
}

// ---------------------------------------------------------------------------
// a5: clip + AdamW + recast.  [MEG] sections 7 and 9; [ZRO] "Why the optimizer
// state is the thing that overflows" (bias-corrected moments, eps outside the
// root); [RST] ch. 13 (decoupled weight decay, beta powers as state); [MP]
// section 2 "Why the weights stay float32" (only the model copy is rounded).
// A set overflow flag makes every CTA return before touching memory.
// ---------------------------------------------------------------------------
struct AdamConsts {
    float step, bc2s, lrwd, b1, omb1, b2, omb2, eps, coef;
};

__device__ __forceinline__ void adamw1(float u, float& w, float& m, float& v, const AdamConsts& k) {
    const float g = __fmul_rn(u, k.coef);
    m = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.omb1, g));
    v = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.omb2, __fmul_rn(g, g)));
    const float wd = __fsub_rn(w, __fmul_rn(k.lrwd, w));
    const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), k.bc2s), k.eps);
    w = __fsub_rn(wd, __fmul_rn(k.step, __fdiv_rn(m, denom)));
}

// Where a segment's u comes from.  UFromAcc: the accumulation buffer holds u
// (written by the unscale or many-list pass).  UFromLists: u is recomputed from
// the resident micro-batch gradient lists in the operations of the many-list
// pass (w_1 g_1, then fma(w_q, g_q, .) in list order, then times 1/S), so it is
// the same value bit for bit; nothing is read from the accumulation buffer.
struct UFromAcc {
    static constexpr int kUnroll = TL_ADAM_UNROLL;
    static constexpr bool kBlocked = false;
    static constexpr bool kEarly = true;   // edge elements loaded ahead of the vector loop
    static constexpr bool kClampTail = TL_ADAM_CLAMP != 0;  // the scalar path's last trip batched
    struct Raw {
        float x[8];
    };
    const float* __restrict__ u0;
    __device__ __forceinline__ explicit UFromAcc(const Chunk& ch) : u0(ch.acc) {}
    __device__ __forceinline__ bool aligned16_all() const { return aligned16(u0); }
    __device__ __forceinline__ bool aligned32_all() const { return aligned32(u0); }
    __device__ __forceinline__ bool phase_is(int r) const { return ephase<4>(u0) == r; }
    __device__ __forceinline__ void load(Raw& r, int o, bool wide) const { ld8_f32(u0 + o, r.x, wide); }
    __device__ __forceinline__ void value(const Raw& r, float (&u)[8]) const {
#pragma unroll
        for (int e = 0; e < 8; ++e) u[e] = r.x[e];
    }
    __device__ __forceinline__ float at(int j) const { return u0[j]; }
};

template <int GDT, int KM>
struct UFromLists {
    static constexpr int kUnroll = TL_REMAT_UNROLL;
    struct Raw {
        typename GradRaw<GDT>::T r[KM];
    };
    static constexpr bool kBlocked = GDT == kE4M3;  // vectors must start on multiples of 8 elements
    static constexpr bool kEarly = false;  // KM gradients per edge element would stay live across the loop
    static constexpr bool kClampTail = false;  // batched, its registers cost spills (1-5 % slower)
    const char* g[KM];
    const float* gs[KM];  // block scales (8-bit gradients)
    const float* w;  // micro-batch weights n_q / N
    int kk;
    float inv_s;
    __device__ __forceinline__ UFromLists(const Chunk& ch, const GradTableMany& inl, const ManyArgs& a, float is)
        : w(a.w), kk(a.k), inv_s(is) {
#pragma unroll
        for (int q = 0; q < KM; ++q) {
            if (q < kk) {
                const void* base = a.tabs[q] != nullptr ? a.tabs[q][ch.tensor] : inl.p[q * a.ntensors + ch.tensor];
                g[q] = static_cast<const char*>(base) + ch.start * Grad<GDT>::kBytes;
                gs[q] = grad_scales<GDT>(base, ch);
            } else {
                g[q] = nullptr;
                gs[q] = nullptr;
            }
        }
    }
    __device__ __forceinline__ bool aligned16_all() const {
        bool al = true;
#pragma unroll
        for (int q = 0; q < KM; ++q)
            if (q < kk) al = al && aligned16(g[q]);
        return al;
    }
    __device__ __forceinline__ bool aligned32_all() const { return true; }  // 16-byte accesses only
    __device__ __forceinline__ bool phase_is(int r) const {
        bool same = true;
#pragma unroll
        for (int q = 0; q < KM; ++q)
            if (q < kk) same = same && ephase<Grad<GDT>::kBytes>(g[q]) == r;
        return same;
    }
    __device__ __forceinline__ void load(Raw& r, int o, bool) const {
#pragma unroll
        for (int q = 0; q < KM; ++q)
            if (q < kk) r.r[q] = GradRaw<GDT>::ld(g[q], o, gs[q]);
    }
    __device__ __forceinline__ void value(const Raw& r, float (&u)[8]) const {
#pragma unroll
        for (int e = 0; e < 8; ++e) u[e] = __fmul_rn(w[0], GradRaw<GDT>::at(r.r[0], e));
#pragma unroll
        for (int q = 1; q < KM; ++q)
            if (q < kk) {
#pragma unroll
                for (int e = 0; e < 8; ++e) u[e] = __fmaf_rn(w[q], GradRaw<GDT>::at(r.r[q], e), u[e]);
            }
#pragma unroll
        for (int e = 0; e < 8; ++e) u[e] = __fmul_rn(u[e], inv_s);
    }
    __device__ __forceinline__ float at(int j) const {
        float v = __fmul_rn(w[0], Grad<GDT>::ld1(g[0], j, gs[0]));
#pragma unroll
        for (int q = 1; q < KM; ++q)
            if (q < kk) v = __fmaf_rn(w[q], Grad<GDT>::ld1(g[q], j, gs[q]), v);
        return __fmul_rn(v, inv_s);
    }
};

template <int NT, int PDT, class Src>
__device__ __forceinline__ void adamw_segment(const Chunk& ch, int t, const AdamConsts& k, const Src& src) {
    float* __restrict__ w0 = ch.master;
    float* __restrict__ m0 = ch.m;
    float* __restrict__ v0 = ch.v;
    unsigned short* p0 = static_cast<unsigned short*>(ch.param);
    const int len = ch.len;
    VecPlan pl{0, false, false};
    if (src.aligned16_all() && aligned16(w0) && aligned16(m0) && aligned16(v0) && aligned16(p0)) {
        pl = VecPlan{0, true, src.aligned32_all() && aligned32(w0) && aligned32(m0) && aligned32(v0)};
    } else {
        const int r = ephase<4>(w0);
        if (src.phase_is(r) && ephase<4>(m0) == r && ephase<4>(v0) == r && ephase<2>(p0) == r)
            pl = VecPlan{(8 - r) & 7, true, true};
    }
    if (Src::kBlocked && pl.head != 0) pl.vec = false;  // an 8-bit vector must not straddle two blocks
    int head = 0, done = 0;
    if (pl.vec) {
        head = min(pl.head, len);
        done = head + (len - head) / kVec * kVec;
    }
    // with Src::kEarly the edge elements' inputs are loaded before the vector
    // loop, so that their latency overlaps it, and finished after it
    const int ej = Src::kEarly && pl.vec ? edge_element(t, head, done, len) : -1;
    float eu = 0.0f, ew = 0.0f, em = 0.0f, ev = 0.0f;
    if (ej >= 0) {
        eu = src.at(ej);
        ew = w0[ej];
        em = m0[ej];
        ev = v0[ej];
    }
    if (pl.vec) {
        const bool wide = pl.wide;
        void* p = p0 + head;
        const int nv = (len - head) / kVec;
        constexpr int U = Src::kUnroll;
        int i = t;
        for (; i + (U - 1) * NT < nv; i += U * NT) {
            typename Src::Raw ur[U];
            float wx[U][8], mx[U][8], vx[U][8];
#pragma unroll
            for (int q = 0; q < U; ++q) {
                const int o = head + (i + q * NT) * kVec;
                src.load(ur[q], o, wide);
                ld8_f32(w0 + o, wx[q], wide);
                ld8_f32(m0 + o, mx[q], wide);
                ld8_f32(v0 + o, vx[q], wide);
            }
#pragma unroll
            for (int q = 0; q < U; ++q) {
                float ux[8];
                src.value(ur[q], ux);
#pragma unroll
                for (int e = 0; e < 8; ++e) adamw1(ux[e], wx[q][e], mx[q][e], vx[q][e], k);
                const int o = head + (i + q * NT) * kVec;
                st8_f32(w0 + o, wx[q], wide);
                st8_f32(m0 + o, mx[q], wide);
                st8_f32(v0 + o, vx[q], wide);
                st8_param<PDT>(p, (i + q * NT) * kVec, wx[q]);
            }
        }
        for (; i < nv; i += NT) {
            typename Src::Raw ur;
            float ux[8], wx[8], mx[8], vx[8];
            const int o = head + i * kVec;
            src.load(ur, o, wide);
            ld8_f32(w0 + o, wx, wide);
            ld8_f32(m0 + o, mx, wide);
            ld8_f32(v0 + o, vx, wide);
            src.value(ur, ux);
#pragma unroll
            for (int e = 0; e < 8; ++e) adamw1(ux[e], wx[e], mx[e], vx[e], k);
            st8_f32(w0 + o, wx, wide);
            st8_f32(m0 + o, mx, wide);
            st8_f32(v0 + o, vx, wide);
            st8_param<PDT>(p, i * kVec, wx);
        }
    }
    if (ej >= 0) {
        adamw1(eu, ew, em, ev, k);
        w0[ej] = ew;
        m0[ej] = em;
        v0[ej] = ev;
        Param<PDT>::st1(p0, ej, ew);
    }
    if (Src::kEarly && pl.vec) return;
    auto one = [&](int j) {
        float wj = w0[j], mj = m0[j], vj = v0[j];
        adamw1(src.at(j), wj, mj, vj, k);
        w0[j] = wj;
        m0[j] = mj;
        v0[j] = vj;
        Param<PDT>::st1(p0, j, wj);
    };
    for (int j = t; j < head; j += NT) one(j);          // head
    // tail, or the whole segment without a vector part: kScalar elements per
    // thread loaded before any is stored
    int j = done + t;
    for (; j + (kScalar - 1) * NT < len; j += kScalar * NT) {
        float ux[kScalar], wx[kScalar], mx[kScalar], vx[kScalar];
#pragma unroll
        for (int q = 0; q < kScalar; ++q) {
            const int o = j + q * NT;
            ux[q] = src.at(o);
            wx[q] = w0[o];
            mx[q] = m0[o];
            vx[q] = v0[o];
        }
#pragma unroll
        for (int q = 0; q < kScalar; ++q) {
            const int o = j + q * NT;
            adamw1(ux[q], wx[q], mx[q], vx[q], k);
            w0[o] = wx[q];
            m0[o] = mx[q];
            v0[o] = vx[q];
            Param<PDT>::st1(p0, o, wx[q]);
        }
    }
    if constexpr (Src::kClampTail) {
        // the last, partial trip batched as the others: its indices clamped to the
        // segment's last element, so that the loads stay unconditional and in flight
        // together, and only the stores of elements past the end left out
        if (j < len) {
            float ux[kScalar], wx[kScalar], mx[kScalar], vx[kScalar];
#pragma unroll
            for (int q = 0; q < kScalar; ++q) {
                const int o = min(j + q * NT, len - 1);
                ux[q] = src.at(o);
                wx[q] = w0[o];
                mx[q] = m0[o];
                vx[q] = v0[o];
            }
#pragma unroll
            for (int q = 0; q < kScalar; ++q) {
                const int o = j + q * NT;
                adamw1(ux[q], wx[q], mx[q], vx[q], k);
                if (o < len) {
                    w0[o] = wx[q];
                    m0[o] = mx[q];
                    v0[o] = vx[q];
                    Param<PDT>::st1(p0, o, wx[q]);
                }
            }
        }
        return;
    }
    for (; j < len; j += NT) one(j);
}

// The clip coefficient of [MEG] section 9 from the global norm: max_norm / (norm +
// 1e-6), applied only below 1; max_norm <= 0 disables clipping.
__device__ __forceinline__ float clip_coef(float norm, float max_norm) {
    float coef = 1.0f;
    if (max_norm > 0.0f) {
        const float cc = __fdiv_rn(max_norm, __fadd_rn(norm, 1e-6f));
        if (cc < 1.0f) coef = cc;
    }
    return coef;
}

// What the scaler needs at the end of an AdamW launch, kept in shared memory (so
// that nothing of it stays live in registers across the element loops).
struct AdamTail {
    double b1n, b2n;   // beta powers of the update in flight
    float coef;
    int skip;
};

__device__ __forceinline__ AdamTail& adam_tail() {
    __shared__ AdamTail t;
    return t;
}

// The per-step AdamW scalars (fp64 beta powers, bias corrections rounded to fp32
// once, the clip coefficient from the device norm), computed by one thread and
// shared through shared memory.  Returns true when the update is skipped (overflow
// flag set).  Thread 0 also leaves what the scaler needs in adam_tail().
__device__ __forceinline__ bool adam_consts(DevState* __restrict__ st, const AdamHP& hp, AdamConsts& out) {
    __shared__ AdamConsts sk;
    __shared__ int skip;
    if (threadIdx.x == 0) {
        const int f = st->found_inf;
        skip = f;
        const double b1n = __dmul_rn(st->b1p, static_cast<double>(hp.beta1));
        const double b2n = __dmul_rn(st->b2p, static_cast<double>(hp.beta2));
        // a schedule is indexed by the committed steps: a skipped attempt leaves
        // the next scheduled rate for the next one
        const int64_t t = st->t;
        const float lr = hp.lr_sched != nullptr ? hp.lr_sched[t < hp.lr_len ? t : hp.lr_len - 1] : hp.lr;
        AdamConsts k;
        k.step = __double2float_rn(__ddiv_rn(static_cast<double>(lr), __dadd_rn(1.0, -b1n)));
        k.bc2s = __double2float_rn(__dsqrt_rn(__dadd_rn(1.0, -b2n)));
        k.lrwd = __double2float_rn(__dmul_rn(static_cast<double>(lr), static_cast<double>(hp.wd)));
        k.b1 = hp.beta1;
        k.omb1 = __fsub_rn(1.0f, hp.beta1);
        k.b2 = hp.beta2;
        k.omb2 = __fsub_rn(1.0f, hp.beta2);
        k.eps = hp.eps;
        k.coef = clip_coef(st->norm, hp.max_norm);
        sk = k;
        adam_tail() = AdamTail{b1n, b2n, k.coef, f};
    }
    __syncthreads();
    out = sk;
    return skip != 0;
}

// ---------------------------------------------------------------------------
// a6: the scaler state machine, run by the last CTA of the update's last AdamW
// launch.  [MEG] section 5 (skip, back off to at least min_loss_scale, reset the
// tracker; or count a good step and grow after `interval` of them); [MP]
// "Dynamic scaling" (the count restarts after every overflow and every growth);
// [RST] ch. 13 "Discard a failed partial logical update" (a skipped attempt keeps
// t and the beta powers).  Every CTA takes a ticket when it is done (after its
// threads have read S and the flag); the CTA holding the last ticket has seen every
// other CTA finish, so it may change S, clear the flag and reset the ticket.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void scaler_step(DevState* __restrict__ st, const ScalerParams& sp, const AdamTail& tl_) {
    if (tl_.skip) {
        if (sp.enabled) {
            const float s = __fmul_rn(st->S, sp.backoff);
            st->S = s > sp.min_scale ? s : sp.min_scale;
        }
        st->count = 0;
        st->skipped = 1;
    } else {
        st->t += 1;
        st->b1p = tl_.b1n;
        st->b2p = tl_.b2n;
        if (sp.enabled) {
            st->count += 1;
            if (st->count == sp.interval) {
                const float s = __fmul_rn(st->S, sp.growth);
                st->S = s < sp.max_scale ? s : sp.max_scale;
                st->count = 0;
            }
        }
        st->skipped = 0;
    }
    st->coef = tl_.coef;
    st->found_inf = 0;
}

__device__ __noinline__ void adam_finish(DevState* __restrict__ st, const ScalerParams& sp) {
    __shared__ int last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t ticket = atomicAdd(&st->adam_ticket, 1u);
        last = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (threadIdx.x != 0 || !last) return;
    __threadfence();
    st->adam_ticket = 0;
    scaler_step(st, sp, adam_tail());
}

template <int NT, int PDT>
__global__ void __launch_bounds__(kThreads, NT == 32 ? TL_MINB_ADAM_GROUP : TL_MINB_ADAM)
k_adamw(const Chunk* __restrict__ chunks, int64_t c0, int64_t c1,
        DevState* __restrict__ st, AdamHP hp, ScalerParams sp) {
    AdamConsts k;
    if (!adam_consts(st, hp, k)) {
        if (NT == kThreads) {
            for_chunks<true>(chunks, c0, c1, [&](int64_t, const Chunk& ch) {
                adamw_segment<kThreads, PDT>(ch, threadIdx.x, k, UFromAcc(ch));
            });
        } else if (NT != 32) {
            for_split_chunks<NT>(c0, c1, [&](int64_t c) {
                const Chunk& ch = chunks[c];
                adamw_segment<NT, PDT>(ch, threadIdx.x % NT, k, UFromAcc(ch));
            });
        } else {
            for (int64_t c = c0 + blockIdx.x; c < c1; c += gridDim.x) {
                const Chunk& ch = group_segment(chunks, c0, c);
                adamw_segment<32, PDT>(ch, threadIdx.x & 31, k, UFromAcc(ch));
            }
        }
    }
    if (sp.run) adam_finish(st, sp);
}

// The re-materialising AdamW pass: u of every element recomputed from the
// resident gradient lists (at most KM <= kRematLists of them) instead of read.
template <int NT, int PDT, int GDT, int KM>
__global__ void __launch_bounds__(kThreads, NT == 32 && GDT == kF32 ? 1
                                            : KM <= kFewLists && GDT != kF32 ? TL_MINB_REMAT_FEW : TL_MINB_REMAT)
k_adamw_remat(const Chunk* __restrict__ chunks, int64_t c0, int64_t c1,
              DevState* __restrict__ st, AdamHP hp, ScalerParams sp, const __grid_constant__ GradTableMany inl,
              const __grid_constant__ ManyArgs a) {
    AdamConsts k;
    const float inv_s = __fdiv_rn(1.0f, st->S);
    if (!adam_consts(st, hp, k)) {
        if (NT == kThreads) {
            for_chunks<true>(chunks, c0, c1, [&](int64_t, const Chunk& ch) {
                adamw_segment<kThreads, PDT>(ch, threadIdx.x, k, UFromLists<GDT, KM>(ch, inl, a, inv_s));
            });
        } else if (NT != 32) {
            for_split_chunks<NT>(c0, c1, [&](int64_t c) {
                const Chunk& ch = chunks[c];
                adamw_segment<NT, PDT>(ch, threadIdx.x % NT, k, UFromLists<GDT, KM>(ch, inl, a, inv_s));
            });
        } else {
            for (int64_t c = c0 + blockIdx.x; c < c1; c += gridDim.x) {
                const Chunk& ch = group_segment(chunks, c0, c);
                adamw_segment<32, PDT>(ch, threadIdx.x & 31, k, UFromLists<GDT, KM>(ch, inl, a, inv_s));
            }
        }
    }
    if (sp.run) adam_finish(st, sp);
}

// ---------------------------------------------------------------------------
// Scalars of one update, one thread each: the clip coefficient from the device
// norm (for a status read before the AdamW launch has computed it); the local
// squared norm and overflow flag copied out to caller memory, and a global squared
// norm and flag (combined across the shards of a sharded update by the caller)
// taken in as the update's: [MEG] section 6 "Overflow must be global" (all ranks of
// one logical update take the same step-or-skip decision) and section 9 (local
// squared norms reduced before the root is taken); [ZRO] "Gradient clipping" (each
// device sums the squares of its own slice, the scalars are all-reduced, then the
// root is taken and the scale applied).
// ---------------------------------------------------------------------------
__global__ void k_coef(DevState* __restrict__ st, float max_norm) {
    if (threadIdx.x == 0 && blockIdx.x == 0) st->coef = clip_coef(st->norm, max_norm);
}

__global__ void k_export(const DevState* __restrict__ st, double* __restrict__ sumsq, int32_t* __restrict__ flag) {
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        sumsq[0] = st->sumsq;
        flag[0] = st->found_inf;
    }
}

__global__ void k_import(DevState* __restrict__ st, const double* __restrict__ sumsq,
                         const int32_t* __restrict__ flag, float max_norm) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const double v = sumsq[0];
    st->sumsq = v;
    if (flag[0] != 0 || !isfinite(v)) st->found_inf = 1;
    const float norm = __double2float_rn(__dsqrt_rn(v));
    st->norm = norm;
    st->coef = clip_coef(norm, max_norm);
}

// ---------------------------------------------------------------------------
// The backward seed S * w_i of a micro-batch ([RST] ch. 13: reverse mode seeded
// with S * n_i / N), read from the device scale at its point in the stream.
// ---------------------------------------------------------------------------
__global__ void k_seed(const DevState* __restrict__ st, float w, float* __restrict__ out) {
    if (threadIdx.x == 0 && blockIdx.x == 0) out[0] = __fmul_rn(st->S, w);
}

// ---------------------------------------------------------------------------
// dispatch tables.  `small` selects the instantiation for small-tensor groups
// (one warp per tensor) over whole-CTA segments; each has its own register
// budget.
// ---------------------------------------------------------------------------
using AccFn = void (*)(const Chunk*, int64_t, int64_t, const GradTable, const void* const*, float);
using UnsFn = void (*)(const Chunk*, int64_t, int64_t, int, const GradTable, const void* const*, float,
                       DevState*, double*, int64_t);
using ManyFn = void (*)(const Chunk*, int64_t, int64_t, int, const GradTableMany, const ManyArgs,
                        DevState*, double*, int64_t);
using AdamFn = void (*)(const Chunk*, int64_t, int64_t, DevState*, AdamHP, ScalerParams);

template <int NT>
AccFn acc_fn_nt(int gdt, bool first) {
    switch (gdt) {
        case kBF16: return first ? k_accumulate<NT, kBF16, true> : k_accumulate<NT, kBF16, false>;
        case kF16: return first ? k_accumulate<NT, kF16, true> : k_accumulate<NT, kF16, false>;
        case kF32: return first ? k_accumulate<NT, kF32, true> : k_accumulate<NT, kF32, false>;
        case kE4M3: return first ? k_accumulate<NT, kE4M3, true> : k_accumulate<NT, kE4M3, false>;
        default: return nullptr;
    }
}

#ifndef TL_SPLIT_TU
AccFn acc_fn(int gdt, bool first, bool small) { return small ? acc_fn_nt<32>(gdt, first) : acc_fn_nt<kThreads>(gdt, first); }
#endif

template <int NT, int GDT>
UnsFn uns_fn_dt(int mode) {
    switch (mode) {
        case kAccOnly: return k_unscale<NT, GDT, kAccOnly>;
        case kFirstOnly: return k_unscale<NT, GDT, kFirstOnly>;
        case kAccAndGrad: return k_unscale<NT, GDT, kAccAndGrad>;
        default: return nullptr;
    }
}

template <int NT>
UnsFn uns_fn_nt(int gdt, int mode) {
    switch (gdt) {
        case kBF16: return uns_fn_dt<NT, kBF16>(mode);
        case kF16: return uns_fn_dt<NT, kF16>(mode);
        case kF32: return uns_fn_dt<NT, kF32>(mode);
        case kE4M3: return uns_fn_dt<NT, kE4M3>(mode);
        default: return nullptr;
    }
}

#ifndef TL_SPLIT_TU
UnsFn uns_fn(int gdt, int mode, bool small) { return small ? uns_fn_nt<32>(gdt, mode) : uns_fn_nt<kThreads>(gdt, mode); }
#endif

template <int NT, int GDT, int KM, bool ROT>
ManyFn many_fn_km(bool first, bool last) {
    if (first)
        return last ? k_accum_many<NT, GDT, true, true, KM, true, ROT> : k_accum_many<NT, GDT, true, false, KM, true, ROT>;
    return last ? k_accum_many<NT, GDT, false, true, KM, true, ROT> : k_accum_many<NT, GDT, false, false, KM, true, ROT>;
}
// the rotated form exists for whole-CTA segments of one or two 16-bit lists only
template <int NT, int GDT>
constexpr bool has_rot() {
    return NT != 32 && (GDT == kBF16 || GDT == kF16);
}
template <int NT, int GDT>
ManyFn many_fn_dt(bool first, bool last, bool few, bool rot) {
    if (!few) return many_fn_km<NT, GDT, kMaxMany, false>(first, last);
    if constexpr (has_rot<NT, GDT>()) {
        if (rot) return many_fn_km<NT, GDT, kFewLists, true>(first, last);
    }
    return many_fn_km<NT, GDT, kFewLists, false>(first, last);
}

template <int NT>
ManyFn many_fn_nt(int gdt, bool first, bool last, bool few, bool rot) {
    switch (gdt) {
        case kBF16: return many_fn_dt<NT, kBF16>(first, last, few, rot);
        case kF16: return many_fn_dt<NT, kF16>(first, last, few, rot);
        case kF32: return many_fn_dt<NT, kF32>(first, last, few, rot);
        case kE4M3: return many_fn_dt<NT, kE4M3>(first, last, few, rot);
        default: return nullptr;
    }
}

#ifndef TL_SPLIT_TU
ManyFn many_fn(int gdt, bool first, bool last, bool small, bool few, bool rot) {
    return small ? many_fn_nt<32>(gdt, first, last, few, rot) : many_fn_nt<kThreads>(gdt, first, last, few, rot);
}
#endif

// the many-list pass without the store of u (first and last micro-batch at once)
template <int NT, int GDT>
ManyFn check_fn_dt(bool few, bool rot) {
    if (!few) return k_accum_many<NT, GDT, true, true, kMaxMany, false, false>;
    if constexpr (has_rot<NT, GDT>()) {
        if (rot) return k_accum_many<NT, GDT, true, true, kFewLists, false, true>;
    }
    return k_accum_many<NT, GDT, true, true, kFewLists, false, false>;
}
template <int NT>
ManyFn check_fn_nt(int gdt, bool few, bool rot) {
    switch (gdt) {
        case kBF16: return check_fn_dt<NT, kBF16>(few, rot);
        case kF16: return check_fn_dt<NT, kF16>(few, rot);
        case kF32: return check_fn_dt<NT, kF32>(few, rot);
        case kE4M3: return check_fn_dt<NT, kE4M3>(few, rot);
        default: return nullptr;
    }
}
#ifndef TL_SPLIT_TU
ManyFn check_fn(int gdt, bool small, bool few, bool rot) {
    return small ? check_fn_nt<32>(gdt, few, rot) : check_fn_nt<kThreads>(gdt, few, rot);
}
#endif

using RematFn = void (*)(const Chunk*, int64_t, int64_t, DevState*, AdamHP, ScalerParams, const GradTableMany,
                         const ManyArgs);

template <int NT, int PDT, int GDT>
RematFn remat_fn_gdt(bool few) {
    return few ? k_adamw_remat<NT, PDT, GDT, kFewLists> : k_adamw_remat<NT, PDT, GDT, kRematLists>;
}
template <int NT, int PDT>
RematFn remat_fn_pdt(int gdt, bool few) {
    switch (gdt) {
        case kBF16: return remat_fn_gdt<NT, PDT, kBF16>(few);
        case kF16: return remat_fn_gdt<NT, PDT, kF16>(few);
        case kF32: return remat_fn_gdt<NT, PDT, kF32>(few);
        case kE4M3: return remat_fn_gdt<NT, PDT, kE4M3>(few);
        default: return nullptr;
    }
}
template <int NT>
RematFn remat_fn_nt(int pdt, int gdt, bool few) {
    switch (pdt) {
        case kBF16: return remat_fn_pdt<NT, kBF16>(gdt, few);
        case kF16: return remat_fn_pdt<NT, kF16>(gdt, few);
        default: return nullptr;
    }
}
#ifndef TL_SPLIT_TU
RematFn remat_fn(int pdt, int gdt, bool small, bool few) {
    return small ? remat_fn_nt<32>(pdt, gdt, few) : remat_fn_nt<kThreads>(pdt, gdt, few);
}

AdamFn adam_fn(int pdt, bool small) {
    switch (pdt) {
        case kBF16: return small ? k_adamw<32, kBF16> : k_adamw<kThreads, kBF16>;
        case kF16: return small ? k_adamw<32, kF16> : k_adamw<kThreads, kF16>;
        default: return nullptr;
    }
}
#endif

int occupancy(const void* f) {
    int n = 0;
    if (f == nullptr || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kThreads, 0) != cudaSuccess || n < 1)
        return 1;
    return n;
}

}  // namespace

#ifdef TL_SPLIT_TU
// The split forms of the partial-writing passes (this file compiled a second
// time, by tl_kernels_split.cu): the launchers of tl_kernels.cu hand them the
// whole-CTA launches of contexts whose runs hold several chunks.
cudaError_t launch_unscale_split(int gdt, int mode, const Chunk* chunks, int64_t c0, int64_t c1, int run,
                                const GradTable& inl, const void* const* gtab, float w, DevState* st, double* partials,
                                int64_t fin, int grid, cudaStream_t s) {
    UnsFn f = uns_fn_nt<kSplitThreads>(gdt, mode);
    if (f == nullptr || run < 1) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, run, inl, gtab, w, st, partials, fin);
    return cudaGetLastError();
}

cudaError_t launch_accum_many_split(int gdt, bool first, bool last, bool rot, const Chunk* chunks, int64_t c0,
                                   int64_t c1, int run, const GradTableMany& inl, const ManyArgs& a, DevState* st,
                                   double* partials, int64_t fin, int grid, cudaStream_t s) {
    ManyFn f = many_fn_nt<kSplitThreads>(gdt, first, last, a.k <= kFewLists, rot);
    if (f == nullptr || a.k < 1 || a.k > kMaxMany || run < 1) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, run, inl, a, st, partials, last ? fin : 0);
    return cudaGetLastError();
}

cudaError_t launch_check_many_split(int gdt, bool rot, const Chunk* chunks, int64_t c0, int64_t c1, int run,
                                   const GradTableMany& inl, const ManyArgs& a, DevState* st, double* partials,
                                   int64_t fin, int grid, cudaStream_t s) {
    ManyFn f = check_fn_nt<kSplitThreads>(gdt, a.k <= kFewLists, rot);
    if (f == nullptr || a.k < 1 || a.k > kMaxMany || run < 1) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, run, inl, a, st, partials, fin);
    return cudaGetLastError();
}

cudaError_t launch_adamw_split(int pdt, const Chunk* chunks, int64_t c0, int64_t c1, DevState* st, AdamHP hp,
                               ScalerParams sp, int grid, cudaStream_t s) {
    AdamFn f = pdt == kBF16 ? k_adamw<kSplitThreads, kBF16> : pdt == kF16 ? k_adamw<kSplitThreads, kF16> : nullptr;
    if (f == nullptr) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, st, hp, sp);
    return cudaGetLastError();
}

cudaError_t launch_adamw_remat_split(int pdt, int gdt, const Chunk* chunks, int64_t c0, int64_t c1, DevState* st,
                                     AdamHP hp, ScalerParams sp, const GradTableMany& inl, const ManyArgs& a, int grid,
                                     cudaStream_t s) {
    RematFn f = remat_fn_nt<kSplitThreads>(pdt, gdt, a.k <= kFewLists);
    if (f == nullptr || a.k < 1 || a.k > kRematLists) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, st, hp, sp, inl, a);
    return cudaGetLastError();
}

int blocks_per_sm_split(int kind, int dt, int variant) {
    const void* f = nullptr;
    if (kind == 2)
        f = dt == kBF16 ? reinterpret_cast<const void*>(k_adamw<kSplitThreads, kBF16>)
            : dt == kF16 ? reinterpret_cast<const void*>(k_adamw<kSplitThreads, kF16>) : nullptr;
    else if (kind == 5) f = reinterpret_cast<const void*>(remat_fn_nt<kSplitThreads>(dt, variant & 3, (variant & 4) != 0));
    else if (kind == 1) f = reinterpret_cast<const void*>(uns_fn_nt<kSplitThreads>(dt, variant));
    else if (kind == 3)
        f = reinterpret_cast<const void*>(many_fn_nt<kSplitThreads>(dt, (variant & 1) != 0, (variant & 2) != 0,
                                                               (variant & 4) != 0, (variant & 8) != 0));
    else if (kind == 4) f = reinterpret_cast<const void*>(check_fn_nt<kSplitThreads>(dt, (variant & 4) != 0, (variant & 8) != 0));
    return occupancy(f);
}

#else  // the whole-CTA and group forms, and the other kernels

// Whole-CTA launches of the partial-writing passes over runs of several chunks go
// to the split forms.
bool split_form(bool small, int run) { return kPairSegs && !small && run > 1; }

cudaError_t launch_accumulate(int gdt, bool first, bool small, const Chunk* chunks, int64_t c0,
                              int64_t c1, const GradTable& inl, const void* const* gtab, float w, int grid,
                              cudaStream_t s) {
    AccFn f = acc_fn(gdt, first, small);
    if (f == nullptr) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, inl, gtab, w);
    return cudaGetLastError();
}

cudaError_t launch_unscale(int gdt, int mode, bool small, const Chunk* chunks, int64_t c0,
                           int64_t c1, int run, const GradTable& inl, const void* const* gtab, float w, DevState* st,
                           double* partials, int64_t fin, int grid, cudaStream_t s) {
    if (split_form(small, run))
        return launch_unscale_split(gdt, mode, chunks, c0, c1, run, inl, gtab, w, st, partials, fin, grid, s);
    UnsFn f = uns_fn(gdt, mode, small);
    if (f == nullptr || run < 1) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, run, inl, gtab, w, st, partials, fin);
    return cudaGetLastError();
}

cudaError_t launch_accum_many(int gdt, bool first, bool last, bool small, bool rot, const Chunk* chunks,
                              int64_t c0, int64_t c1, int run, const GradTableMany& inl, const ManyArgs& a,
                              DevState* st, double* partials, int64_t fin, int grid, cudaStream_t s) {
    if (split_form(small, run))
        return launch_accum_many_split(gdt, first, last, rot, chunks, c0, c1, run, inl, a, st, partials, fin, grid, s);
    ManyFn f = many_fn(gdt, first, last, small, a.k <= kFewLists, rot);
    if (f == nullptr || a.k < 1 || a.k > kMaxMany || run < 1) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, run, inl, a, st, partials, last ? fin : 0);
    return cudaGetLastError();
}

cudaError_t launch_norm(const double* partials, int64_t n, double* slots, DevState* st, float max_norm,
                        cudaStream_t s) {
    static_assert(kNormBlocks <= kNormThreads, "the last CTA reads one slot per thread");
    static_assert((kNormBlocks & (kNormBlocks - 1)) == 0, "the ticket counter wraps modulo a multiple of kNormBlocks");
    k_norm<<<kNormBlocks, kNormThreads, 0, s>>>(partials, n, slots, st, max_norm);
    return cudaGetLastError();
}

cudaError_t launch_check_many(int gdt, bool small, bool rot, const Chunk* chunks, int64_t c0, int64_t c1, int run,
                              const GradTableMany& inl, const ManyArgs& a, DevState* st, double* partials,
                              int64_t fin, int grid, cudaStream_t s) {
    if (split_form(small, run))
        return launch_check_many_split(gdt, rot, chunks, c0, c1, run, inl, a, st, partials, fin, grid, s);
    ManyFn f = check_fn(gdt, small, a.k <= kFewLists, rot);
    if (f == nullptr || a.k < 1 || a.k > kMaxMany || run < 1) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, run, inl, a, st, partials, fin);
    return cudaGetLastError();
}

cudaError_t launch_adamw_remat(int pdt, int gdt, bool small, int run, const Chunk* chunks, int64_t c0,
                               int64_t c1, DevState* st, AdamHP hp, ScalerParams sp, const GradTableMany& inl,
                               const ManyArgs& a, int grid, cudaStream_t s) {
    if (kSplitAdam && split_form(small, run))
        return launch_adamw_remat_split(pdt, gdt, chunks, c0, c1, st, hp, sp, inl, a, grid, s);
    RematFn f = remat_fn(pdt, gdt, small, a.k <= kFewLists);
    if (f == nullptr || a.k < 1 || a.k > kRematLists) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, st, hp, sp, inl, a);
    return cudaGetLastError();
}

cudaError_t launch_adamw(int pdt, bool small, int run, const Chunk* chunks, int64_t c0, int64_t c1,
                         DevState* st, AdamHP hp, ScalerParams sp, int grid, cudaStream_t s) {
    if (kSplitAdam && split_form(small, run)) return launch_adamw_split(pdt, chunks, c0, c1, st, hp, sp, grid, s);
    AdamFn f = adam_fn(pdt, small);
    if (f == nullptr) return cudaErrorInvalidValue;
    f<<<grid, kThreads, 0, s>>>(chunks, c0, c1, st, hp, sp);
    return cudaGetLastError();
}

cudaError_t launch_seed(const DevState* st, float w, float* out, cudaStream_t s) {
    k_seed<<<1, 32, 0, s>>>(st, w, out);
    return cudaGetLastError();
}

cudaError_t launch_coef(DevState* st, float max_norm, cudaStream_t s) {
    k_coef<<<1, 32, 0, s>>>(st, max_norm);
    return cudaGetLastError();
}

cudaError_t launch_export(const DevState* st, double* sumsq, int32_t* flag, cudaStream_t s) {
    k_export<<<1, 32, 0, s>>>(st, sumsq, flag);
    return cudaGetLastError();
}

cudaError_t launch_import(DevState* st, const double* sumsq, const int32_t* flag, float max_norm, cudaStream_t s) {
    k_import<<<1, 32, 0, s>>>(st, sumsq, flag, max_norm);
    return cudaGetLastError();
}

int blocks_per_sm(int kind, int dt, int variant, bool small) {
    if ((variant & 16) != 0 && kind >= 1 && kind <= 5 && (kSplitAdam || (kind != 2 && kind != 5)) &&
        split_form(small, 2))
        return blocks_per_sm_split(kind, dt, variant & 15);
    variant &= 15;
    const void* f = nullptr;
    if (kind == 0) f = reinterpret_cast<const void*>(acc_fn(dt, variant != 0, small));
    else if (kind == 1) f = reinterpret_cast<const void*>(uns_fn(dt, variant, small));
    else if (kind == 2) f = reinterpret_cast<const void*>(adam_fn(dt, small));
    else if (kind == 3)
        f = reinterpret_cast<const void*>(many_fn(dt, (variant & 1) != 0, (variant & 2) != 0, small, (variant & 4) != 0,
                                                  (variant & 8) != 0));
    else if (kind == 4) f = reinterpret_cast<const void*>(check_fn(dt, small, (variant & 4) != 0, (variant & 8) != 0));
    else if (kind == 5) f = reinterpret_cast<const void*>(remat_fn(dt, variant & 3, small, (variant & 4) != 0));
    return occupancy(f);
}

#endif  // TL_SPLIT_TU

}  // namespace tl
