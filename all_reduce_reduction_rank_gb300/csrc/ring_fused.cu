// The ring's result in one pass over HBM.
//
// Handbook "多 GPU 与 NCCL", §ring all-reduce: in the reduce-scatter phase
// each chunk travels once around the ring and every rank it reaches adds its
// own copy of the chunk; the all-gather phase then only copies the completed
// chunk to the other ranks.  Per element that is a chain of additions in a
// fixed order: chunk c starts as rank c's value and takes in ranks c+1, ...,
// c+n-1 (mod n), one binary32 add per hop, with the partial kept in fp32 (as
// ar_ring) or rounded to the payload type after every hop (as
// ar_ring_rounded), and is rounded once into the rank that completes it; the
// copies change no bits.  No element depends on another, so one thread can
// load the n ranks' 16-byte vectors of chunk c once, run the chain in
// registers in the ring's order and store the result to all n outputs: the
// same bits as the step-by-step emulation, with HBM reading n S and writing
// n S, the bytes of one-shot, in one launch instead of 2 (n - 1).
#include "common.cuh"

namespace argb {
namespace {

// Vectors per thread per iteration, as the one-shot kernel.
template <int NR> __host__ __device__ constexpr int ring_fused_unroll() { return NR <= 4 ? 4 : NR <= 8 ? 2 : 1; }

// One hop's rounding of the partial to the payload type and back (identity
// for fp32).
template <int DT>
__device__ __forceinline__ void hop_round(float* a)
{
    constexpr int P = Payload<DT>::kPerWord;
#pragma unroll
    for (int j = 0; j < 4; ++j) Payload<DT>::widen(Payload<DT>::narrow(a + j * P), a + j * P);
}

// Grid: blockIdx.y = chunk c (block-uniform ring order), blockIdx.x strides
// over the chunk's 16-byte vectors, U per thread per iteration in CTAs of up
// to kThreads threads (U = 1 and narrower CTAs for calls too small to give
// every SM a full CTA).  HR: round the partial after every hop.  Three CTAs per SM
// at least: registers stay at or below 80, and no rank count spills.
template <int NR, int DT, bool HR, int U>
__global__ void __launch_bounds__(kThreads, 3)
ring_fused_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t C,
                  size_t count)
{
    pdl_acquire();
    using T = typename Payload<DT>::scalar_t;
    constexpr int VE = kVecElems<DT>;
    const int c = blockIdx.y;
    const size_t e_lo = (size_t)c * C;
    if (e_lo >= count) return;
    const size_t len = count - e_lo < C ? count - e_lo : C;   // elements of chunk c
    const size_t nv = len / VE;
    // src(k): chunk c of the rank the chain reaches after k hops
    auto src = [&](int k) { return static_cast<const T*>(in.p[c + k < NR ? c + k : c + k - NR]) + e_lo; };
    const size_t bs = U > 1 ? (size_t)kThreads : (size_t)blockDim.x, span = bs * U;  // U > 1: full CTAs only
    for (size_t base = (size_t)blockIdx.x * span; base < nv; base += (size_t)gridDim.x * span) {
        uint4 x[U][NR];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = base + (size_t)u * bs + threadIdx.x;
            if (v < nv) {
#pragma unroll
                for (int k = 0; k < NR; ++k) x[u][k] = ld16(src(k) + v * VE);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = base + (size_t)u * bs + threadIdx.x;
            if (v < nv) {
                float a[VE];
                // the chain starts from rank c's value itself (no zero start)
#pragma unroll
                for (int j = 0; j < 4; ++j) Payload<DT>::widen(word(x[u][0], j), a + j * Payload<DT>::kPerWord);
#pragma unroll
                for (int k = 1; k < NR; ++k) {
                    accumulate<DT>(a, x[u][k]);
                    if (HR && k < NR - 1) hop_round<DT>(a);
                }
                const uint4 y = round_vec<DT>(a);
#pragma unroll
                for (int q = 0; q < NR; ++q) st16(static_cast<T*>(out.p[q]) + e_lo + v * VE, y);
            }
        }
    }
    pdl_release();
    // the ragged end of the last chunk: one element per thread
    if (blockIdx.x == gridDim.x - 1) {
        const size_t j = nv * VE + threadIdx.x;
        if (j < len) {
            float a = Payload<DT>::widen1(src(0)[j]);
#pragma unroll
            for (int k = 1; k < NR; ++k) {
                a = a + Payload<DT>::widen1(src(k)[j]);
                if (HR && k < NR - 1) a = Payload<DT>::widen1(Payload<DT>::narrow1(a));
            }
            const T y = Payload<DT>::narrow1(a);
#pragma unroll
            for (int q = 0; q < NR; ++q) static_cast<T*>(out.p[q])[e_lo + j] = y;
        }
    }
}

template <bool HR>
int launch_ring_fused_impl(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                           cudaStream_t s, int* launches)
{
    return dispatch_dtype(dt, [&](auto dtc) -> int {
        constexpr int DT = decltype(dtc)::value;
        return dispatch_ranks(h.n, [&](auto nrc) -> int {
            constexpr int NR = decltype(nrc)::value;
            constexpr int U = ring_fused_unroll<NR>();
            CPtrs<NR> ip;
            MPtrs<NR> op;
            for (int q = 0; q < NR; ++q) {
                ip.p[q] = in[q];
                op.p[q] = out[q];
            }
            const size_t C = chunk_elems(NR, count, DT);
            const size_t cvec = C / kVecElems<DT>;
            const uint64_t S = (uint64_t)count * sizeof(typename Payload<DT>::scalar_t);
            const dim3 grid(grid_for_rows(h, (cvec + U - 1) / U, NR), NR);
            rec_begin(h, s);
            if (grid.x * grid.y < (unsigned)h.sm_count) {
                const Shape sh = narrow_shape(h, cvec, NR);
                launch_kernel(h, ring_fused_kernel<NR, DT, HR, 1>, dim3(sh.grid_x, NR), sh.block, 0, s, ip, op, C,
                              count);
            } else
                launch_kernel(h, ring_fused_kernel<NR, DT, HR, U>, grid, kThreads, 0, s, ip, op, C, count);
            rec_end(h, s, HR ? AR_K_RING_ROUNDED_FUSED : AR_K_RING_FUSED, 2ull * NR * S);
            *launches = 1;
            return launch_status();
        });
    });
}

}  // namespace

int launch_ring_fused(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                      int* launches)
{
    return launch_ring_fused_impl<false>(h, in, out, count, dt, s, launches);
}

int launch_ring_rounded_fused(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                              cudaStream_t s, int* launches)
{
    return launch_ring_fused_impl<true>(h, in, out, count, dt, s, launches);
}

}  // namespace argb
