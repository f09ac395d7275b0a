// Ring all-reduce, emulated step by step on one GPU.
//
// Handbook "多 GPU 与 NCCL", §ring all-reduce: p ranks form a ring and the
// data is cut into p chunks.  Reduce-scatter phase (p-1 steps): in each step
// every rank sends one chunk to the next rank, which adds the chunk it
// receives to its own copy of that chunk; after p-1 steps every rank holds
// the complete sum of one chunk.  All-gather phase (p-1 steps): every rank
// passes a completed chunk along the ring.  Each rank sends 2(p-1) S/p bytes
// over 2(p-1) steps.
//
// Emulation: one launch per step; one launch performs the n transfers of
// that step.  Reduce-scatter step s: rank r sends chunk c = (r - s) mod n to
// d = (r + 1) mod n.  The partial sums stay fp32 between hops, in the
// handle's scratch [2][n][C] (double-buffered by step parity, since in one
// step rank d both sends the partial it received in the step before and
// receives a new one).  At the last step the receiving rank rounds the
// completed chunk into its output.  All-gather step s: rank r passes chunk
// (r + 1 - s) mod n from its output to rank r + 1's output.
//
// HBM traffic per reduce-scatter step: n chunk reads of the sender's partial
// (payload at step 0), n of the receiver's payload, n partial writes
// (payload at the last step); per all-gather step n chunk reads and writes.
#include "common.cuh"

namespace argb {
namespace {

// Reduce-scatter step s of the ring.  Work item w = (r, k): vector k of the
// chunk that rank r sends.  p_read / p_write: fp32 partials, rank-major, C
// elements per rank.
template <int NR, int DT>
__global__ void __launch_bounds__(kThreads)
ring_rs_step_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, const float* __restrict__ p_read,
                    float* __restrict__ p_write, size_t C, size_t count, int s)
{
    constexpr int VE = kVecElems<DT>;
    using T = typename Payload<DT>::scalar_t;
    const bool first = (s == 0), last = (s == NR - 2);
    const size_t cvec = C / VE;
    const size_t total = (size_t)NR * cvec;
    for (size_t w = (size_t)blockIdx.x * kThreads + threadIdx.x; w < total;
         w += (size_t)gridDim.x * kThreads) {
        const int r = (int)(w / cvec);
        const size_t k = w - (size_t)r * cvec;
        const int d = (r + 1) % NR;
        const int c = (r - s + NR) % NR;
        const size_t e0 = (size_t)c * C + k * VE;  // first element of this vector
        if (e0 >= count) continue;
        const float* pr = p_read + (size_t)r * C + k * VE;
        float* pw = p_write + (size_t)d * C + k * VE;
        float a[VE];
        if (e0 + VE <= count) {
            // upstream partial (the sender's payload at step 0) ...
            if (first) {
                const uint4 xr = ld16(static_cast<const T*>(in.p[r]) + e0);
#pragma unroll
                for (int j = 0; j < VE; ++j) a[j] = 0.0f;
                // 0 + x is x except for -0: widen exactly instead of adding.
#pragma unroll
                for (int j = 0; j < 4; ++j) Payload<DT>::widen(word(xr, j), a + j * Payload<DT>::kPerWord);
            } else {
#pragma unroll
                for (int j = 0; j < VE / 4; ++j) {
                    const uint4 t = ld16(pr + 4 * j);
                    a[4 * j + 0] = __uint_as_float(t.x);
                    a[4 * j + 1] = __uint_as_float(t.y);
                    a[4 * j + 2] = __uint_as_float(t.z);
                    a[4 * j + 3] = __uint_as_float(t.w);
                }
            }
            // ... plus the receiver's own chunk
            const uint4 xd = ld16(static_cast<const T*>(in.p[d]) + e0);
            accumulate<DT>(a, xd);
            if (last) {
                st16(static_cast<T*>(out.p[d]) + e0, round_vec<DT>(a));
            } else {
#pragma unroll
                for (int j = 0; j < VE / 4; ++j)
                    st16(pw + 4 * j, make_uint4(__float_as_uint(a[4 * j]), __float_as_uint(a[4 * j + 1]),
                                                __float_as_uint(a[4 * j + 2]), __float_as_uint(a[4 * j + 3])));
            }
        } else {
            // the ragged end of the last chunk: element by element
            const size_t m = count - e0;
            for (size_t j = 0; j < m; ++j) {
                const float up = first ? Payload<DT>::widen1(static_cast<const T*>(in.p[r])[e0 + j]) : pr[j];
                const float sum = up + Payload<DT>::widen1(static_cast<const T*>(in.p[d])[e0 + j]);
                if (last) static_cast<T*>(out.p[d])[e0 + j] = Payload<DT>::narrow1(sum);
                else pw[j] = sum;
            }
        }
    }
}

// All-gather step s: out[r+1][chunk (r+1-s)] = out[r][chunk (r+1-s)].
template <int NR, int DT>
__global__ void __launch_bounds__(kThreads)
ring_ag_step_kernel(const __grid_constant__ MPtrs<NR> out, size_t C, size_t count, int s)
{
    constexpr int VE = kVecElems<DT>;
    using T = typename Payload<DT>::scalar_t;
    const size_t cvec = C / VE;
    const size_t total = (size_t)NR * cvec;
    for (size_t w = (size_t)blockIdx.x * kThreads + threadIdx.x; w < total;
         w += (size_t)gridDim.x * kThreads) {
        const int r = (int)(w / cvec);
        const size_t k = w - (size_t)r * cvec;
        const int d = (r + 1) % NR;
        const int c = (r + 1 - s + NR) % NR;
        const size_t e0 = (size_t)c * C + k * VE;
        if (e0 >= count) continue;
        const T* src = static_cast<const T*>(out.p[r]) + e0;
        T* dst = static_cast<T*>(out.p[d]) + e0;
        if (e0 + VE <= count) {
            st16(dst, ld16(src));
        } else {
            for (size_t j = 0; j < count - e0; ++j) dst[j] = src[j];
        }
    }
}

}  // namespace

int launch_ring(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
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
            const size_t C = chunk_elems(NR, count, DT);
            if (C > h.ring_chunk_max) return AR_ERR_TOO_LARGE;
            const unsigned grid = grid_for(h, (size_t)NR * (C / kVecElems<DT>));
            float* buf[2] = {h.ring_scratch, h.ring_scratch + (size_t)NR * C};
            int n_launch = 0;
            // per step every chunk moves once: N elements in all
            const uint64_t N = count, e = sizeof(typename Payload<DT>::scalar_t);
            for (int step = 0; step < NR - 1; ++step) {
                const uint64_t rd = (step == 0 ? e : 4) * N + e * N;
                const uint64_t wr = (step == NR - 2 ? e : 4) * N;
                rec_begin(h, s);
                ring_rs_step_kernel<NR, DT><<<grid, kThreads, 0, s>>>(
                    ip, op, buf[(step + 1) & 1], buf[step & 1], C, count, step);
                rec_end(h, s, AR_K_RING_RS_STEP, rd + wr);
                ++n_launch;
                if (launch_status() != AR_OK) return AR_ERR_CUDA;
            }
            for (int step = 0; step < NR - 1; ++step) {
                rec_begin(h, s);
                ring_ag_step_kernel<NR, DT><<<grid, kThreads, 0, s>>>(op, C, count, step);
                rec_end(h, s, AR_K_RING_AG_STEP, 2 * e * N);
                ++n_launch;
                if (launch_status() != AR_OK) return AR_ERR_CUDA;
            }
            *launches = n_launch;
            return AR_OK;
        });
    });
}

}  // namespace argb
