// One-shot all-reduce of n rank buffers held in one GPU's HBM.
//
// "SGLang JIT custom all-reduce" notes: §1 each thread moves one 16-byte
// vector per rank per iteration; §2 grid-stride loop over 16-byte vectors,
// adjacent threads on adjacent vectors (coalesced); §3 the n loads are
// unrolled so all of them are in flight together; §4 fp32 accumulation from
// zero in rank order, one round-to-nearest; §5 the store.  The kBroadcast
// form (result written to every rank's output) is what an emulated
// all-reduce needs: the n outputs are all in this HBM.
//
// HBM traffic: each input vector is read once and each output vector
// written once, 2 n S bytes in all; the kernel is bound by HBM bandwidth.
#include "common.cuh"

namespace argb {
namespace {

// Vectors per thread per iteration: keeps about 128-256 B of loads in flight
// per thread without spilling at n = 16.
template <int NR> __host__ __device__ constexpr int one_shot_unroll() { return NR <= 4 ? 4 : NR <= 8 ? 2 : 1; }

template <int NR, int DT>
__global__ void __launch_bounds__(kThreads)
one_shot_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t nvec, size_t count)
{
    constexpr int U = one_shot_unroll<NR>();
    const size_t span = (size_t)kThreads * U;
    for (size_t base = (size_t)blockIdx.x * span; base < nvec; base += (size_t)gridDim.x * span) {
        uint4 x[U][NR];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = base + (size_t)u * kThreads + threadIdx.x;
            if (v < nvec) {
#pragma unroll
                for (int q = 0; q < NR; ++q) x[u][q] = ld16(static_cast<const uint4*>(in.p[q]) + v);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = base + (size_t)u * kThreads + threadIdx.x;
            if (v < nvec) {
                const uint4 r = reduce_rank_order<DT, NR>(x[u]);
#pragma unroll
                for (int q = 0; q < NR; ++q) st16(static_cast<uint4*>(out.p[q]) + v, r);
            }
        }
    }
    // Elements after the last whole vector: same arithmetic, one per thread.
    if (blockIdx.x == gridDim.x - 1) {
        using T = typename Payload<DT>::scalar_t;
        const size_t i = nvec * kVecElems<DT> + threadIdx.x;
        if (i < count) {
            float acc = 0.0f;
#pragma unroll
            for (int q = 0; q < NR; ++q) acc = acc + Payload<DT>::widen1(static_cast<const T*>(in.p[q])[i]);
            const T r = Payload<DT>::narrow1(acc);
#pragma unroll
            for (int q = 0; q < NR; ++q) static_cast<T*>(out.p[q])[i] = r;
        }
    }
}

}  // namespace

int launch_one_shot(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                    cudaStream_t s, int* launches)
{
    return dispatch_dtype(dt, [&](auto dtc) -> int {
        constexpr int DT = decltype(dtc)::value;
        return dispatch_ranks(h.n, [&](auto nrc) -> int {
            constexpr int NR = decltype(nrc)::value;
            CPtrs<NR> ip;
            MPtrs<NR> op;
            for (int q = 0; q < NR; ++q) {
                ip.p[q] = in[q];
                op.p[q] = out[q];
            }
            const size_t nvec = count / kVecElems<DT>;
            constexpr int U = one_shot_unroll<NR>();
            const unsigned grid = grid_for(h, (nvec + U - 1) / U);
            const uint64_t S = (uint64_t)count * sizeof(typename Payload<DT>::scalar_t);
            rec_begin(h, s);
            one_shot_kernel<NR, DT><<<grid, kThreads, 0, s>>>(ip, op, nvec, count);
            rec_end(h, s, AR_K_ONE_SHOT, 2ull * NR * S);
            *launches = 1;
            return launch_status();
        });
    });
}

}  // namespace argb
