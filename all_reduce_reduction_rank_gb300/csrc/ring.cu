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
// that step.  A call whose step data (the n chunks' partials) is larger than
// half of L2 runs in pieces: each chunk is cut into P equal pieces (P = that
// data over half of L2, rounded), and the whole ring -- all reduce-scatter
// steps, then all all-gather steps -- runs on piece 0 of every chunk, then on
// piece 1, and so on, so one piece's partials stay in L2 from step to step
// (handbook "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce", §算法:
// a large message cut into blocks and pipelined; every element keeps its
// chunk and its order of summation, so the sums are the same).  Reduce-scatter step s: rank r sends chunk c = (r - s) mod n to
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
//
// ar_ring_rounded runs the same steps with the partials kept in the payload
// type, rounded at every hop (a library whose buffers hold the payload type
// adds each received chunk to its own copy that way): 2 e N read and e N
// written per reduce-scatter step.  Its partials sit in one buffer indexed by
// chunk and are rewritten in place, half the footprint of the double buffer:
// measured on GB300 (bf16, back to back) 215.0 against 228.5 us at n = 8,
// 64 MiB per rank and 1863 against 1976 us at n = 16, 256 MiB; the fp32
// ring laid out the same way was 1-3% slower, so it keeps the double buffer.
#include "common.cuh"

namespace argb {
namespace {

// Every store of a ring step is read by the next step (the partial the next
// hop adds to, the chunk the next all-gather hop passes on), so it keeps the
// default write-back policy (st16_next), and a reduce-scatter step's reads are
// each the last use of their data (the partial it adds to is dead once read,
// the payload chunk is read once), so they load with the streaming hint
// (ld16_last).  Measured on GB300 (n = 8 bf16, back-to-back calls): the stores
// took the ring from 421 to 385 us at 64 MiB per rank and the hop-rounded ring
// from 317 to 294 us (no change at 8 MiB); the loads then 380.6 -> 376.5 us at
// 64 MiB and 62.9 -> 60.8 us at 8 MiB.  Evict-last stores (an L2 cache
// policy), discarding the dead partial lines from L2 after their last read,
// and the streaming hint on the all-gather's reads were each no faster.
constexpr int kRsUnroll = 2;  // vectors per thread per iteration
// All-gather step: 8 vectors per thread, compiled for at least two CTAs per
// SM (GB300, n = 8 bf16, back to back: the ring 374.5 against 376.6 us at
// 64 MiB per rank and 58.6 against 60.7 us at 8 MiB with 4 vectors and the
// compiler's own bound; 2 vectors were 3% slower at 64 MiB).
constexpr int kAgUnroll = 8;

// The rank (row) r and the x position bx of this CTA in step g of the ring's
// 2(n-1) steps (g = s in the reduce-scatter, n - 1 + s in the all-gather).
// Every step reads what the step before wrote: row r reads the data row r - 1
// wrote.  When a step's data is larger than L2 (reorder), each step takes its
// tiles in the reverse of the order in which the step before wrote the data
// they read: CTAs are dispatched roughly in linear block order and L2 keeps
// the most recently written lines, so the first tiles a step reads are the
// last written, still in L2.  Hence odd steps reverse the block order (rows
// and x), and every step rotates its rows by g so that row r's reads follow
// row r - 1's writes.  Measured on GB300 (n = 8 bf16, 64 MiB per rank): 4.6%
// fewer DRAM bytes per reduce-scatter step, 29% fewer per all-gather step, the
// ring 3% faster; at 8 MiB (everything in L2) the plain order is 2% faster.
// Which CTA does which tile changes nothing in the sums.
// A template flag, not a runtime one: a runtime flag cost the step kernel 14
// registers and with them a CTA per SM.
template <int NR, bool RO>
__device__ __forceinline__ void ring_tile(int g, int& r, unsigned& bx)
{
    if constexpr (RO) {
        const bool rev = (g & 1) != 0;
        const int yb = rev ? NR - 1 - (int)blockIdx.y : (int)blockIdx.y;
        r = (yb + g) % NR;
        bx = rev ? gridDim.x - 1 - blockIdx.x : blockIdx.x;
    } else {
        r = (int)blockIdx.y;
        bx = blockIdx.x;
    }
}

// Reduce-scatter step s.  Grid: blockIdx.y gives the sending rank r
// (block-uniform chunk, pointers and step role; see ring_tile), blockIdx.x
// strides over the chunk's 16-byte vectors.  p_read / p_write: partials, rank-major, C elements per rank; fp32,
// or (HR, hop rounding) the payload type.  The fp32-partial step is compiled
// for three CTAs per SM (at most 80 registers; the ring measured 3% faster at
// 8 MiB per rank); the hop-rounded step keeps the compiler's own choice (a
// minimum of 0), which ran 10-16% faster at 8-64 MiB than that bound.
template <int NR, int DT, bool HR, bool RO>
__global__ void __launch_bounds__(kThreads, HR ? 0 : 3)
ring_rs_step_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out,
                    const float* __restrict__ p_read, float* __restrict__ p_write, size_t C, size_t count, int s,
                    size_t p_len)
{
    pdl_acquire();
    constexpr int VE = kVecElems<DT>;
    constexpr int PW = HR ? 1 : VE / 4;  // 16-byte words of partial per payload vector
    constexpr int U = kRsUnroll;
    using T = typename Payload<DT>::scalar_t;
    int r;
    unsigned bx;
    ring_tile<NR, RO>(s, r, bx);
    const int d = (r + 1) % NR;
    const int c = (r - s + NR) % NR;
    const bool first = (s == 0), last = (s == NR - 2);
    const size_t e_lo = (size_t)c * C;
    if (e_lo >= count) return;
    const size_t len = count - e_lo < p_len ? count - e_lo : p_len;   // elements of chunk c's piece
    const size_t nv = len / VE;                                 // whole vectors
    const T* const xr = static_cast<const T*>(in.p[r]) + e_lo;
    const T* const xd = static_cast<const T*>(in.p[d]) + e_lo;
    T* const od = static_cast<T*>(out.p[d]) + e_lo;
    const float* const pr = p_read + (size_t)r * C;
    float* const pw = p_write + (size_t)d * C;
    // hop-rounded partials: one buffer indexed by chunk, each partial read and rewritten in place
    // (a chunk's partial is held by one rank at a time, so no step reads what another writes);
    // read and written through p_write alone
    const T* const prh = reinterpret_cast<const T*>(p_write) + (size_t)c * C;
    T* const pwh = reinterpret_cast<T*>(p_write) + (size_t)c * C;
    const size_t span = (size_t)kThreads * U;
    for (size_t base = (size_t)bx * span; base < nv; base += (size_t)gridDim.x * span) {
        uint4 up[U][PW], own[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t k = base + (size_t)u * kThreads + threadIdx.x;
            if (k < nv) {
                // the partial rank r sends (its own payload at step 0) ...
                if (first) {
                    up[u][0] = ld16_last(xr + k * VE);
                } else if (HR) {
                    up[u][0] = ld16_last(prh + k * VE);
                } else {
#pragma unroll
                    for (int j = 0; j < PW; ++j) up[u][j] = ld16_last(pr + k * VE + 4 * j);
                }
                // ... and the receiver's own chunk
                own[u] = ld16_last(xd + k * VE);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t k = base + (size_t)u * kThreads + threadIdx.x;
            if (k < nv) {
                float a[VE];
                if (first || HR) {
                    // widen exactly (no zero start: the first hop adds two raw values)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        Payload<DT>::widen(word(up[u][0], j), a + j * Payload<DT>::kPerWord);
                } else {
#pragma unroll
                    for (int j = 0; j < PW; ++j) {
                        a[4 * j + 0] = __uint_as_float(up[u][j].x);
                        a[4 * j + 1] = __uint_as_float(up[u][j].y);
                        a[4 * j + 2] = __uint_as_float(up[u][j].z);
                        a[4 * j + 3] = __uint_as_float(up[u][j].w);
                    }
                }
                accumulate<DT>(a, own[u]);
                if (last) {
                    st16_next(od + k * VE, round_vec<DT>(a));
                } else if (HR) {
                    st16_next(pwh + k * VE, round_vec<DT>(a));
                } else {
#pragma unroll
                    for (int j = 0; j < PW; ++j)
                        st16_next(pw + k * VE + 4 * j,
                             make_uint4(__float_as_uint(a[4 * j]), __float_as_uint(a[4 * j + 1]),
                                        __float_as_uint(a[4 * j + 2]), __float_as_uint(a[4 * j + 3])));
                }
            }
        }
    }
    pdl_release();
    // the ragged end of the last chunk: one element per thread
    if (blockIdx.x == gridDim.x - 1) {
        const size_t j = nv * VE + threadIdx.x;
        if (j < len) {
            const float upv = first ? Payload<DT>::widen1(xr[j]) : HR ? Payload<DT>::widen1(prh[j]) : pr[j];
            const float sum = upv + Payload<DT>::widen1(xd[j]);
            if (last) od[j] = Payload<DT>::narrow1(sum);
            else if (HR) pwh[j] = Payload<DT>::narrow1(sum);
            else pw[j] = sum;
        }
    }
}

// All-gather step s: out[r+1][chunk (r+1-s)] = out[r][chunk (r+1-s)].
// Grid: blockIdx.y gives the sending rank r (see ring_tile).
template <int NR, int DT, bool RO>
__global__ void __launch_bounds__(kThreads, 2)
ring_ag_step_kernel(const __grid_constant__ MPtrs<NR> out, size_t C, size_t count, int s, size_t p_len)
{
    pdl_acquire();
    constexpr int VE = kVecElems<DT>;
    constexpr int U = kAgUnroll;
    using T = typename Payload<DT>::scalar_t;
    int r;
    unsigned bx;
    ring_tile<NR, RO>(NR - 1 + s, r, bx);
    const int d = (r + 1) % NR;
    const int c = (r + 1 - s + NR) % NR;
    const size_t e_lo = (size_t)c * C;
    if (e_lo >= count) return;
    const size_t len = count - e_lo < p_len ? count - e_lo : p_len;
    const size_t nv = len / VE;
    const T* const src = static_cast<const T*>(out.p[r]) + e_lo;
    T* const dst = static_cast<T*>(out.p[d]) + e_lo;
    const size_t span = (size_t)kThreads * U;
    for (size_t base = (size_t)bx * span; base < nv; base += (size_t)gridDim.x * span) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t k = base + (size_t)u * kThreads + threadIdx.x;
            if (k < nv) x[u] = ld16(src + k * VE);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t k = base + (size_t)u * kThreads + threadIdx.x;
            if (k < nv) st16_next(dst + k * VE, x[u]);
        }
    }
    pdl_release();
    if (blockIdx.x == gridDim.x - 1) {
        const size_t j = nv * VE + threadIdx.x;
        if (j < len) dst[j] = src[j];
    }
}

}  // namespace

template <bool HR>
int launch_ring_impl(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                     int* launches)
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
            const uint64_t e = sizeof(typename Payload<DT>::scalar_t);
            const uint64_t pe = HR ? e : 4;   // bytes of one partial
            // pieces: a step's partials over half of L2, rounded (measured on GB300, n = 8 bf16 and
            // n = 16: at 64 MiB per rank 2 pieces ran the ring 372 against 388 us at n = 8 and 809
            // against 853 us at n = 16; at 256 MiB and n = 16, 8 pieces 3313 against 3774 us and the
            // hop-rounded ring in 4 pieces 2224 against 2685 us; below half of L2 every extra
            // piece was slower, by about 1.4 us per added launch)
            const uint64_t half_l2 = h.l2_bytes / 2;
            // two streams (PieceStreams in internal.h) when a step's partials reach a tenth of L2.
            // Measured on GB300 (back to back; one stream -> two): n = 8 bf16 at 16 / 32 / 64 MiB per
            // rank 100.1 -> 88.8, 171.4 -> 157.5, 345.6 -> 312.6 us; n = 16 at 64 / 256 MiB 759 -> 666,
            // 3096 -> 2715; n = 4 at 64 MiB 147.6 -> 132.9; the hop-rounded ring 7-14% less (16 MiB:
            // 77.4 -> 70.3, 16.8 MB of step data); 58.8 -> 56.9 at 16.8 MB of fp32 partials (n = 8,
            // 8 MiB), slower at 8.4 MB and below (hop-rounded ring at 8 MiB: 45.9 -> 51.7; 1 MiB: 26.9
            // -> 49 us).  Twice the one-stream pieces was best at every size measured.
            const uint64_t step_data = (uint64_t)count * pe;
            const bool dual = two_streams(h, step_data, 10);
            size_t PL = piece_elems(h, step_data, C);
            if (dual) PL = half_piece(PL, C);
            const size_t cvec = (PL + kVecElems<DT> - 1) / kVecElems<DT>;
            const dim3 g_rs(grid_for_rows(h, (cvec + kRsUnroll - 1) / kRsUnroll, NR), NR);
            const dim3 g_ag(grid_for_rows(h, (cvec + kAgUnroll - 1) / kAgUnroll, NR), NR);
            float* buf[2] = {h.ring_scratch, h.ring_scratch + (size_t)NR * C};
            // a piece's step data (its partials) larger than half of L2: the reversed tile order
            const uint64_t step_bytes = (uint64_t)PL * NR * pe;
            const bool reorder = half_l2 > 0 && step_bytes > half_l2;
            int n_launch = 0, pieces = 0;
            PieceStreams streams{h, s, dual};
            if (streams.fork() != AR_OK) return AR_ERR_CUDA;
            // a piece is passed as every pointer moved to its first element and the count moved
            // with it, so the kernels' chunk arithmetic is the unpieced one (in-kernel piece offsets
            // cost the reduce-scatter step 19 registers and with them a CTA per SM)
            using T = typename Payload<DT>::scalar_t;
            auto shifted = [&](size_t p_lo, CPtrs<NR>& ipp, MPtrs<NR>& opp, float** bp) {
                for (int q = 0; q < NR; ++q) {
                    ipp.p[q] = static_cast<const T*>(ip.p[q]) + p_lo;
                    opp.p[q] = static_cast<T*>(op.p[q]) + p_lo;
                }
                for (int k = 0; k < 2; ++k)
                    bp[k] = HR ? reinterpret_cast<float*>(reinterpret_cast<T*>(buf[k]) + p_lo) : buf[k] + p_lo;
            };
            // piece by piece: its reduce-scatter steps, then its all-gather steps, whose first step
            // finds the chunk the last reduce-scatter step completed still in L2; one timing record
            // per piece and phase (the n-1 steps run back to back)
            int rc = AR_OK;
            for (size_t p_lo = 0; p_lo < C && rc == AR_OK; p_lo += PL) {
                const size_t p_len = C - p_lo < PL ? C - p_lo : PL;
                const cudaStream_t s = streams.next();   // this piece's stream
                ++pieces;
                uint64_t pn = 0;   // the piece's elements over all n chunks
                for (int c = 0; c < NR; ++c) {
                    const size_t lo = (size_t)c * C + p_lo;
                    if (lo < count) pn += count - lo < p_len ? count - lo : p_len;
                }
                uint64_t rs_bytes = 0;
                for (int step = 0; step < NR - 1; ++step)
                    rs_bytes += (step == 0 ? e : pe) * pn + e * pn + (step == NR - 2 ? e : pe) * pn;
                CPtrs<NR> ipp;
                MPtrs<NR> opp;
                float* bp[2];
                shifted(p_lo, ipp, opp, bp);
                rec_begin(h, s);
                for (int step = 0; step < NR - 1; ++step) {
                    if (reorder)
                        launch_kernel(h, ring_rs_step_kernel<NR, DT, HR, true>, g_rs, kThreads, 0, s, ipp, opp,
                                      bp[(step + 1) & 1], HR ? bp[0] : bp[step & 1], C, count - p_lo, step, p_len);
                    else
                        launch_kernel(h, ring_rs_step_kernel<NR, DT, HR, false>, g_rs, kThreads, 0, s, ipp, opp,
                                      bp[(step + 1) & 1], HR ? bp[0] : bp[step & 1], C, count - p_lo, step, p_len);
                    ++n_launch;
                    if (launch_status() != AR_OK) rc = AR_ERR_CUDA;
                }
                rec_end(h, s, HR ? AR_K_RING_RS_STEP_ROUNDED : AR_K_RING_RS_STEP, rs_bytes, NR - 1);
                rec_begin(h, s);
                for (int step = 0; step < NR - 1; ++step) {
                    if (reorder)
                        launch_kernel(h, ring_ag_step_kernel<NR, DT, true>, g_ag, kThreads, 0, s, opp, C, count - p_lo,
                                      step, p_len);
                    else
                        launch_kernel(h, ring_ag_step_kernel<NR, DT, false>, g_ag, kThreads, 0, s, opp, C, count - p_lo,
                                      step, p_len);
                    ++n_launch;
                    if (launch_status() != AR_OK) rc = AR_ERR_CUDA;
                }
                rec_end(h, s, AR_K_RING_AG_STEP, 2 * e * pn * (NR - 1), NR - 1);
            }
            if (streams.join() != AR_OK) rc = AR_ERR_CUDA;
            *launches = n_launch;
            return rc;
        });
    });
}

int launch_ring(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                int* launches)
{
    return launch_ring_impl<false>(h, in, out, count, dt, s, launches);
}

int launch_ring_rounded(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                        int* launches)
{
    return launch_ring_impl<true>(h, in, out, count, dt, s, launches);
}

}  // namespace argb
