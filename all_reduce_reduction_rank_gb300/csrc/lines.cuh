// Device helpers shared by the two persistent rings (ring_persistent.cu,
// ring_cluster.cu): the LL128 line geometry and the element loads and stores
// of a rank's own chunk in that geometry.
//
// A line carries 30 fp32 words (elements 30 l .. 30 l + 29 of a chunk) in its
// first 120 bytes; 8 lanes move it, 16 bytes each, lane j holding elements
// 30 l + 4 j .. + 3 (lane 7: two, then the flag).  A batch is 32 lines (one
// flag per lane of a warp).
#pragma once

#include "common.cuh"

namespace argb {
namespace lines {

constexpr int kLineWords = 30;
constexpr int kBatchLines = 32;
constexpr size_t kBatchElems = (size_t)kLineWords * kBatchLines;   // 960

__device__ __forceinline__ void st8_plain(void* p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ uint2 ld8_plain(const void* p)
{
    uint2 v;
    asm volatile("ld.global.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld4_plain(const void* p)
{
    uint32_t v;
    asm volatile("ld.global.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Raw words of elements e .. e+nw-1 (zero past len): 4 fp32 words, or 2
// words of two 16-bit elements each.  Loads only; widen_raw converts later,
// so a warp can issue every load of a batch before it waits for any.
template <int DT> constexpr int kRawWords = DT == AR_F32 ? 4 : 2;

template <int DT>
__device__ __forceinline__ void load_raw(const void* chunk, size_t e, int nw, size_t len, uint32_t* w)
{
    using T = typename Payload<DT>::scalar_t;
    const T* x = static_cast<const T*>(chunk);
    if (e + (size_t)nw <= len) {
        if constexpr (DT == AR_F32) {
            const uint2 a = ld8_plain(x + e);
            w[0] = a.x;
            w[1] = a.y;
            w[2] = w[3] = 0u;
            if (nw == 4) {
                const uint2 b = ld8_plain(x + e + 2);
                w[2] = b.x;
                w[3] = b.y;
            }
        } else {
            w[0] = ld4_plain(x + e);
            w[1] = nw == 4 ? ld4_plain(x + e + 2) : 0u;
        }
    } else {
        const uint16_t* x16 = reinterpret_cast<const uint16_t*>(chunk);
        const uint32_t* x32 = reinterpret_cast<const uint32_t*>(chunk);
#pragma unroll
        for (int u = 0; u < kRawWords<DT>; ++u) w[u] = 0u;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (u < nw && e + u < len) {
                if constexpr (DT == AR_F32) w[u] = x32[e + u];
                else w[u >> 1] |= (uint32_t)x16[e + u] << (16 * (u & 1));
            }
        }
    }
}

template <int DT>
__device__ __forceinline__ void widen_raw(const uint32_t* w, float* f)
{
    if constexpr (DT == AR_F32) {
#pragma unroll
        for (int u = 0; u < 4; ++u) f[u] = __uint_as_float(w[u]);
    } else {
        Payload<DT>::widen(w[0], f);
        Payload<DT>::widen(w[1], f + 2);
    }
}

// Rounds f[0..nw) to the payload type and stores the elements below len.
template <int DT>
__device__ __forceinline__ void store_elems(void* chunk, size_t e, int nw, size_t len, const float* f)
{
    using T = typename Payload<DT>::scalar_t;
    T* y = static_cast<T*>(chunk);
    if (e + (size_t)nw <= len) {
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
            if (u >= nw) break;
            if constexpr (DT == AR_F32) {
                st8_plain(y + e + u, __float_as_uint(f[u]), __float_as_uint(f[u + 1]));
            } else {
                const uint32_t w = Payload<DT>::narrow(f + u);
                asm volatile("st.global.u32 [%0], %1;" ::"l"(y + e + u), "r"(w) : "memory");
            }
        }
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (u < nw && e + u < len) y[e + u] = Payload<DT>::narrow1(f[u]);
    }
}

}  // namespace lines
}  // namespace argb
