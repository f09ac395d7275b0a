// Device helpers shared by the kernels of libar_gb300.so (sm_103a).
//
// The data path is HBM streaming: 16-byte vector loads and stores
// ("SGLang JIT custom all-reduce" notes, §1: one 128-bit access per thread
// per iteration), fp32 accumulation in rank order, one rounding at the end
// (same notes, §4).  There is no dense contraction, so no tensor cores.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace argb {

// ---- 16-byte global accesses ----------------------------------------------
// Loads skip L1 (each byte is read once); stores use the streaming hint.
// Plain weak accesses: ordering between calls comes from stream order.

__device__ __forceinline__ uint4 ld16(const void* p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st16(void* p, const uint4& v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// For a call of several launches, where one launch reads what the one before
// wrote (the ring's steps, the tree's levels, staged copies): the store keeps
// the default write-back policy, since st16's streaming hint marks its lines
// first to be evicted from L2 and the next launch would then read them from
// DRAM; and a load that is the last use of its data in the call takes the
// streaming hint, so its lines are the first to leave L2 and the lines the
// launch writes for the next one stay.
__device__ __forceinline__ void st16_next(void* p, const uint4& v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ld16_last(const void* p)
{
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Re-read for flag polling: a volatile load is never served from a stale
// register copy and is issued every time.
__device__ __forceinline__ uint4 ld16_volatile(const void* p)
{
    uint4 v;
    asm volatile("ld.volatile.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- payload types ---------------------------------------------------------
// Every payload type converts a 32-bit word holding 1 or 2 elements to fp32
// (exact) and back (round to nearest even).

template <int DT> struct Payload;

template <> struct Payload<AR_F32> {
    static constexpr int kPerWord = 1;
    using scalar_t = float;
    __device__ __forceinline__ static void widen(uint32_t w, float* f) { f[0] = __uint_as_float(w); }
    __device__ __forceinline__ static uint32_t narrow(const float* f) { return __float_as_uint(f[0]); }
    __device__ __forceinline__ static float widen1(scalar_t x) { return x; }
    __device__ __forceinline__ static scalar_t narrow1(float f) { return f; }
};

template <> struct Payload<AR_BF16> {
    static constexpr int kPerWord = 2;
    using scalar_t = __nv_bfloat16;
    __device__ __forceinline__ static void widen(uint32_t w, float* f)
    {
        __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w);
        float2 t = __bfloat1622float2(h);
        f[0] = t.x;
        f[1] = t.y;
    }
    __device__ __forceinline__ static uint32_t narrow(const float* f)
    {
        __nv_bfloat162 h = __float22bfloat162_rn(make_float2(f[0], f[1]));
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ __forceinline__ static float widen1(scalar_t x) { return __bfloat162float(x); }
    __device__ __forceinline__ static scalar_t narrow1(float f) { return __float2bfloat16_rn(f); }
};

template <> struct Payload<AR_F16> {
    static constexpr int kPerWord = 2;
    using scalar_t = __half;
    __device__ __forceinline__ static void widen(uint32_t w, float* f)
    {
        __half2 h = *reinterpret_cast<const __half2*>(&w);
        float2 t = __half22float2(h);
        f[0] = t.x;
        f[1] = t.y;
    }
    __device__ __forceinline__ static uint32_t narrow(const float* f)
    {
        __half2 h = __float22half2_rn(make_float2(f[0], f[1]));
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ __forceinline__ static float widen1(scalar_t x) { return __half2float(x); }
    __device__ __forceinline__ static scalar_t narrow1(float f) { return __float2half_rn(f); }
};

// Elements of the payload type in one 16-byte vector.
template <int DT> constexpr int kVecElems = 4 * Payload<DT>::kPerWord;

__device__ __forceinline__ uint32_t word(const uint4& v, int j)
{
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// acc[...] += widen(v), elementwise, for one 16-byte vector.
template <int DT>
__device__ __forceinline__ void accumulate(float* acc, const uint4& v)
{
    constexpr int P = Payload<DT>::kPerWord;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float f[P];
        Payload<DT>::widen(word(v, j), f);
#pragma unroll
        for (int k = 0; k < P; ++k) acc[j * P + k] = acc[j * P + k] + f[k];
    }
}

template <int DT>
__device__ __forceinline__ uint4 round_vec(const float* acc)
{
    constexpr int P = Payload<DT>::kPerWord;
    uint4 r;
    r.x = Payload<DT>::narrow(acc + 0 * P);
    r.y = Payload<DT>::narrow(acc + 1 * P);
    r.z = Payload<DT>::narrow(acc + 2 * P);
    r.w = Payload<DT>::narrow(acc + 3 * P);
    return r;
}

// Rank-order sum of NR vectors: acc = +0, then acc += x[0], ..., x[NR-1].
template <int DT, int NR>
__device__ __forceinline__ uint4 reduce_rank_order(const uint4 (&x)[NR])
{
    float acc[kVecElems<DT>];
#pragma unroll
    for (int k = 0; k < kVecElems<DT>; ++k) acc[k] = 0.0f;
#pragma unroll
    for (int q = 0; q < NR; ++q) accumulate<DT>(acc, x[q]);
    return round_vec<DT>(acc);
}

// ---- sticky status word ----------------------------------------------------

struct DevStatus {
    int code;
    int rank;
    unsigned long long line;
    unsigned long long skipped;
};

__device__ __forceinline__ void report_flag_timeout(DevStatus* st, int rank, unsigned long long line)
{
    if (atomicCAS(&st->code, 0, AR_ERR_FLAG_TIMEOUT) == 0) {
        st->rank = rank;
        st->line = line;
    }
    atomicAdd(&st->skipped, 1ull);
}

__device__ __forceinline__ void report_wait_timeout(DevStatus* st)
{
    atomicCAS(&st->code, 0, AR_ERR_WAIT_TIMEOUT);
}

// ---- programmatic dependent launch ------------------------------------------
// Every kernel is launched with programmatic stream serialization allowed
// (AR_OPT_PDL, default on), so the next kernel in the stream can be launched
// while this one drains.  Each kernel starts by waiting for its predecessor's
// completion and memory (griddepcontrol.wait, a hardware wait that returns at
// once when there is no programmatic predecessor) before it touches global
// memory, and lets its dependents launch once its own main loop is done
// (pdl_release): early enough to hide their launch, late enough that their
// CTAs, which wait on this grid, are spread over the SMs as this grid's tail
// frees them rather than packed onto the first SMs to free up.

__device__ __forceinline__ void pdl_acquire() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(const Handle& h, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, Args&&... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = h.pdl ? 1 : 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Rank pointer tables, passed by value in the kernel parameters.
template <int NR> struct CPtrs { const void* p[NR]; };
template <int NR> struct MPtrs { void* p[NR]; };

// Call f(std::integral_constant<int, n>) for n in [2, 16].
template <typename F>
inline int dispatch_ranks(int n, F&& f)
{
    switch (n) {
    case 2: return f(std::integral_constant<int, 2>{});
    case 3: return f(std::integral_constant<int, 3>{});
    case 4: return f(std::integral_constant<int, 4>{});
    case 5: return f(std::integral_constant<int, 5>{});
    case 6: return f(std::integral_constant<int, 6>{});
    case 7: return f(std::integral_constant<int, 7>{});
    case 8: return f(std::integral_constant<int, 8>{});
    case 9: return f(std::integral_constant<int, 9>{});
    case 10: return f(std::integral_constant<int, 10>{});
    case 11: return f(std::integral_constant<int, 11>{});
    case 12: return f(std::integral_constant<int, 12>{});
    case 13: return f(std::integral_constant<int, 13>{});
    case 14: return f(std::integral_constant<int, 14>{});
    case 15: return f(std::integral_constant<int, 15>{});
    case 16: return f(std::integral_constant<int, 16>{});
    default: return AR_ERR_INVALID;
    }
}

// Call f(std::integral_constant<int, dt>) for the three payload types.
template <typename F>
inline int dispatch_dtype(int dt, F&& f)
{
    switch (dt) {
    case AR_F32: return f(std::integral_constant<int, AR_F32>{});
    case AR_BF16: return f(std::integral_constant<int, AR_BF16>{});
    case AR_F16: return f(std::integral_constant<int, AR_F16>{});
    default: return AR_ERR_INVALID;
    }
}

inline int launch_status()
{
    return cudaGetLastError() == cudaSuccess ? AR_OK : AR_ERR_CUDA;
}

}  // namespace argb
