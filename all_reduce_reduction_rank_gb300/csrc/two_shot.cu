// Two-shot all-reduce: a reduce-scatter phase, then an all-gather phase.
//
// Handbook "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce", §算法:
// in the first step each rank reads 1/n of every other rank's data and sums
// it (a reduce-scatter); in the second it reads the summed pieces back (an
// all-gather); two synchronizations.  "多 GPU 与 NCCL", §集合通信: all-reduce
// = reduce-scatter + all-gather.
//
// Chunk r is elements [rC, min((r+1)C, N)), C = ceil(N/n) rounded up to a
// whole 16-byte vector, so every chunk starts on a vector boundary.  The
// kernel boundary between the two launches is the synchronization.
//
// HBM traffic: phase 1 reads n S and writes S; phase 2 reads S and writes
// (n-1) S: (2n+1) S in all.
#include "common.cuh"

namespace argb {
namespace {

template <int NR> __host__ __device__ constexpr int rs_unroll() { return NR <= 4 ? 4 : NR <= 8 ? 2 : 1; }
// One vector per thread per iteration: measured best for the all-gather
// (n = 8 bf16, back-to-back calls: 23.2 vs 24.3 us at 8 MiB per rank, 169.0 vs
// 171.8 us at 64 MiB, against an unroll of 4).
constexpr int kAgUnroll = 1;

// Grid: blockIdx.y = chunk r (block-uniform output pointer, no per-vector
// division), blockIdx.x strides over the chunk's 16-byte vectors, in CTAs of
// up to kThreads threads (narrower ones, and U = 1, for calls too small to
// give every SM a full CTA; Small, compiled for three CTAs per SM as the
// one-shot kernel's small form, for latency).

// out[r][v] = rank-order sum of in[*][v] for v in chunk r.
template <int NR, int DT, int U, bool Small>
__global__ void __launch_bounds__(kThreads, Small ? 3 : 0)
reduce_scatter_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t nvec,
                      size_t count, size_t cvec)
{
    pdl_acquire();
    const int r = blockIdx.y;
    const size_t lo = (size_t)r * cvec;
    const size_t hi = lo + cvec < nvec ? lo + cvec : nvec;
    uint4* const dst = static_cast<uint4*>(out.p[r]);
    const size_t bs = U > 1 ? (size_t)kThreads : (size_t)blockDim.x, span = bs * U;  // U > 1: full CTAs only
    for (size_t base = lo + (size_t)blockIdx.x * span; base < hi; base += (size_t)gridDim.x * span) {
        uint4 x[U][NR];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = base + (size_t)u * bs + threadIdx.x;
            if (v < hi) {
#pragma unroll
                for (int q = 0; q < NR; ++q) x[u][q] = ld16(static_cast<const uint4*>(in.p[q]) + v);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = base + (size_t)u * bs + threadIdx.x;
            if (v < hi) st16(dst + v, reduce_rank_order<DT, NR>(x[u]));
        }
    }
    pdl_release();
    // elements past the last whole vector, handled once by the grid's last block
    if (blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1) {
        using T = typename Payload<DT>::scalar_t;
        const size_t i = nvec * kVecElems<DT> + threadIdx.x;
        if (i < count) {
            float acc = 0.0f;
#pragma unroll
            for (int q = 0; q < NR; ++q) acc = acc + Payload<DT>::widen1(static_cast<const T*>(in.p[q])[i]);
            static_cast<T*>(out.p[i / (cvec * kVecElems<DT>)])[i] = Payload<DT>::narrow1(acc);
        }
    }
}

// For v in chunk j: out[q][v] = out[j][v] for every q != j.
template <int NR, int DT, bool Small>
__global__ void __launch_bounds__(kThreads, Small ? 3 : 0)
all_gather_kernel(const __grid_constant__ MPtrs<NR> out, size_t nvec, size_t count, size_t cvec)
{
    pdl_acquire();
    constexpr int U = kAgUnroll;
    const int j = blockIdx.y;
    const size_t lo = (size_t)j * cvec;
    const size_t hi = lo + cvec < nvec ? lo + cvec : nvec;
    const uint4* const src = static_cast<const uint4*>(out.p[j]);
    const size_t bs = blockDim.x, span = bs * U;
    for (size_t base = lo + (size_t)blockIdx.x * span; base < hi; base += (size_t)gridDim.x * span) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = base + (size_t)u * bs + threadIdx.x;
            if (v < hi) x[u] = ld16(src + v);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = base + (size_t)u * bs + threadIdx.x;
            if (v < hi) {
#pragma unroll
                for (int q = 0; q < NR; ++q)
                    if (q != j) st16(static_cast<uint4*>(out.p[q]) + v, x[u]);
            }
        }
    }
    pdl_release();
    if (blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1) {
        using T = typename Payload<DT>::scalar_t;
        const size_t i = nvec * kVecElems<DT> + threadIdx.x;
        if (i < count) {
            const int jt = (int)(i / (cvec * kVecElems<DT>));
            const T x = static_cast<const T*>(out.p[jt])[i];
#pragma unroll
            for (int q = 0; q < NR; ++q)
                if (q != jt) static_cast<T*>(out.p[q])[i] = x;
        }
    }
}

}  // namespace

int launch_two_shot(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
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
            const size_t cvec = chunk_elems(NR, count, DT) / kVecElems<DT>;  // >= 1 for count >= 1
            constexpr int U = rs_unroll<NR>();
            const uint64_t S = (uint64_t)count * sizeof(typename Payload<DT>::scalar_t);
            const dim3 g_rs(grid_for_rows(h, (cvec + U - 1) / U, NR), NR);
            const dim3 g_ag(grid_for_rows(h, (cvec + kAgUnroll - 1) / kAgUnroll, NR), NR);
            // a call too small to give every SM a full CTA: narrower CTAs, one vector per thread
            const bool narrow = g_rs.x * NR < (unsigned)h.sm_count;
            const Shape sh = narrow_shape(h, cvec, NR);
            rec_begin(h, s);
            if (narrow)
                launch_kernel(h, reduce_scatter_kernel<NR, DT, 1, true>, dim3(sh.grid_x, NR), sh.block, 0, s, ip, op,
                              nvec, count, cvec);
            else
                launch_kernel(h, reduce_scatter_kernel<NR, DT, U, false>, g_rs, kThreads, 0, s, ip, op, nvec, count,
                              cvec);
            rec_end(h, s, AR_K_REDUCE_SCATTER, (uint64_t)(NR + 1) * S);
            if (launch_status() != AR_OK) return AR_ERR_CUDA;
            rec_begin(h, s);
            if (narrow)
                launch_kernel(h, all_gather_kernel<NR, DT, true>, dim3(sh.grid_x, NR), sh.block, 0, s, op, nvec, count,
                              cvec);
            else
                launch_kernel(h, all_gather_kernel<NR, DT, false>, g_ag, kThreads, 0, s, op, nvec, count, cvec);
            rec_end(h, s, AR_K_ALL_GATHER, (uint64_t)NR * S);
            *launches = 2;
            return launch_status();
        });
    });
}

}  // namespace argb
