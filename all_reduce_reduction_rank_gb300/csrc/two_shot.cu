// Two-shot all-reduce: a reduce-scatter phase, then an all-gather phase.
//
// Handbook "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce", §算法:
// in the first step each rank reads 1/n of every other rank's data and sums
// it (a reduce-scatter); in the second it reads the summed pieces back (an
// all-gather); two synchronizations.  "多 GPU 与 NCCL", §集合通信: all-reduce
// = reduce-scatter + all-gather.
//
// Chunk r is elements [rC, min((r+1)C, N)), C = ceil(N/n) rounded up to a
// whole 16-byte vector, so every chunk starts on a vector boundary.
//
// Three forms, the same bits and the same bytes (AR_OPT_TWO_SHOT_IMPL):
//   1  two launches: reduce_scatter_kernel, then all_gather_kernel; the
//      kernel boundary is the synchronization between the phases;
//   2  one launch (the default): two_shot_one_launch_kernel with the
//      synchronization per tile inside a CTA: the CTA that reduces tile k of
//      chunk r into out[r] then gathers that tile itself, a CTA barrier
//      ordering its phase-1 stores before it reads them back;
//   3  one launch with the synchronization per tile between CTAs: the CTA
//      that reduces a tile publishes a ready flag (release), and the CTA that
//      gathers it, a wave of CTAs later, waits for the flag (acquire,
//      bounded) before it reads the reduced tile back.
// Measured on GB300 (n = 8 bf16, 8 KiB - 64 MiB per rank), form 2 is the
// fastest at every size: one launch instead of two, and the re-read of the
// reduced tile comes from L2 right after its write.  Form 3 is slower than
// both (a ticket atomic, a release and an acquire per CTA); it is kept as the
// emulation of ranks that hand tiles to each other.
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
            if (v < hi) st16_next(dst + v, reduce_rank_order<DT, NR>(x[u]));   // the all-gather launch reads it
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


// ---- one launch: per-tile flags ----------------------------------------------
// Work items: phase-1 item i reduces tile k of chunk r (i = r * tpc + k, a
// tile = T = block x U vectors) into out[r]; phase-2 item i copies that tile
// of out[r] to every other rank.  Each CTA takes a ticket t from a counter in
// `sync` when it starts and does phase-1 item t (if t < R = n tpc), then
// phase-2 item t - L (if t >= L): the tile a CTA gathers was reduced by the
// CTA that took the ticket L earlier.  L = min(R, about one wave of CTAs), so
// that tile is normally done, and still in L2, when it is gathered.
//
// Progress: tickets go to CTAs in the order they start, and a CTA publishes
// its phase-1 tile before it waits for anything; it then waits only for the
// tile of a lower ticket, whose CTA has already started.  So the lowest
// waiting CTA always finds its tile coming, whatever the block scheduler
// does.  The wait is bounded all the same (AR_OPT_SPIN_NS): if it runs out
// the CTA records AR_ERR_WAIT_TIMEOUT, leaves that tile's outputs untouched
// and ends.
//
// sync (u32): [0] ticket counter, [1] CTAs finished, [2] epoch of the last
// finished call, [3] unused, [4 + i] ready flag of phase-1 item i.  A call's
// flags carry epoch = [2] + 1, so flags of earlier calls never match; the last
// CTA to finish zeroes the counters and advances [2] (read by the next call
// only after this grid has completed).

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u32(unsigned* p, unsigned v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Read of a tile another CTA reduced: cached in L2 only, never in this SM's L1.
__device__ __forceinline__ uint4 ld16_cg(const void* p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint64_t flag_polls(int64_t spin_ns) { return (uint64_t)spin_ns / 32u + 64u; }

// Vectors per thread per tile and the CTAs per SM the kernel is compiled for:
// about 128 KiB of loads in flight per SM at every n (4 CTAs of 256 threads
// x n ranks x U vectors x 16 B up to n = 8; 2 CTAs at n > 8).
template <int NR> __host__ __device__ constexpr int flagged_unroll() { return NR <= 2 ? 4 : NR <= 4 ? 2 : 1; }
template <int NR> __host__ __device__ constexpr int flagged_ctas_per_sm() { return NR <= 8 ? 4 : 2; }

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// lag > 0: the CTA of ticket t reduces tile t (if t < R) and gathers tile
// t - lag (if that is a tile), waiting for its flag.  lag == 0: no tickets
// and no flags; the CTA of block b reduces tile b and then gathers the same
// tile itself, a CTA barrier ordering its phase-1 stores before the re-read.
template <int NR, int DT, int U, bool Small>
__global__ void __launch_bounds__(kThreads, Small ? 3 : flagged_ctas_per_sm<NR>())
two_shot_one_launch_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t nvec,
                        size_t count, size_t cvec, unsigned tpc, unsigned lag, unsigned* __restrict__ sync,
                        DevStatus* st, int64_t spin_ns)
{
    pdl_acquire();
    __shared__ unsigned s_ticket, s_epoch;
    __shared__ int s_ready;
    unsigned* const flags = sync + 4;
    if (lag > 0) {
        if (threadIdx.x == 0) {
            s_ticket = atomicAdd(sync, 1u);
            s_epoch = ld_relaxed_u32(sync + 2) + 1u;
        }
        __syncthreads();
    }
    const unsigned t = lag > 0 ? s_ticket : blockIdx.x;
    const unsigned epoch = lag > 0 ? s_epoch : 0u;
    const unsigned R = (unsigned)NR * tpc;
    const size_t bs = U > 1 ? (size_t)kThreads : (size_t)blockDim.x, T = bs * U;  // U > 1: full CTAs only
    auto tile = [&](unsigned i, unsigned& r, size_t& lo, size_t& hi) {
        r = i / tpc;
        const size_t c_lo = (size_t)r * cvec;
        const size_t c_hi = c_lo + cvec < nvec ? c_lo + cvec : nvec;
        lo = c_lo + (size_t)(i - r * tpc) * T;
        hi = lo + T < c_hi ? lo + T : c_hi;
    };
    // phase 1's tile: issue its loads first
    unsigned r1 = 0;
    size_t lo1 = 0, hi1 = 0;
    if (t < R) tile(t, r1, lo1, hi1);
    uint4 x[U][NR];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const size_t v = lo1 + (size_t)u * bs + threadIdx.x;
        if (v < hi1) {
#pragma unroll
            for (int q = 0; q < NR; ++q) x[u][q] = ld16(static_cast<const uint4*>(in.p[q]) + v);
        }
    }
    // phase 2's tile (lag > 0): wait for its flag and load it while phase 1's loads are in flight
    unsigned r2 = 0;
    size_t lo2 = 0, hi2 = 0;
    if (lag > 0 && t >= lag && t - lag < R) tile(t - lag, r2, lo2, hi2);
    uint4 g[U];
    if (lo2 < hi2) {
        if (threadIdx.x == 0) {
            const unsigned* const f = flags + (t - lag);
            int ok = ld_acquire_u32(f) == epoch;
            if (!ok) {
                const uint64_t t0 = globaltimer_ns(), cap = flag_polls(spin_ns);
                for (uint64_t it = 0; it < cap && !ok; ++it) {
                    __nanosleep(32);
                    ok = ld_acquire_u32(f) == epoch;
                    if ((int64_t)(globaltimer_ns() - t0) > spin_ns) break;
                }
            }
            if (!ok) report_wait_timeout(st);
            s_ready = ok;
        }
        __syncthreads();
        if (!s_ready) hi2 = lo2;   // leave this tile's outputs untouched
        const uint4* const src = static_cast<const uint4*>(out.p[r2]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = lo2 + (size_t)u * bs + threadIdx.x;
            if (v < hi2) g[u] = ld16_cg(src + v);
        }
    }
    // phase 1: out[r1][tile] = rank-order sum of in[*][tile]
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const size_t v = lo1 + (size_t)u * bs + threadIdx.x;
        if (v < hi1) st16(static_cast<uint4*>(out.p[r1]) + v, reduce_rank_order<DT, NR>(x[u]));
    }
    if (lag == 0 && lo1 < hi1) {
        // the same tile gathered by this CTA: after its phase-1 stores
        __syncthreads();
        r2 = r1;
        lo2 = lo1;
        hi2 = hi1;
        const uint4* const src = static_cast<const uint4*>(out.p[r2]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = lo2 + (size_t)u * bs + threadIdx.x;
            if (v < hi2) g[u] = ld16_cg(src + v);
        }
    }
    // phase 2: out[q][tile] = out[r2][tile] for every q != r2
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const size_t v = lo2 + (size_t)u * bs + threadIdx.x;
        if (v < hi2) {
#pragma unroll
            for (int q = 0; q < NR; ++q)
                if (q != (int)r2) st16(static_cast<uint4*>(out.p[q]) + v, g[u]);
        }
    }
    // publish phase 1's tile
    if (lag > 0 && lo1 < hi1) {
        __syncthreads();  // every thread's stores of the tile come before the release
        if (threadIdx.x == 0) st_release_u32(flags + t, epoch);
    }
    pdl_release();
    // elements past the last whole vector: both phases by one thread each (same thread, program order)
    if (t == 0) {
        using T_ = typename Payload<DT>::scalar_t;
        const size_t i = nvec * kVecElems<DT> + threadIdx.x;
        if (i < count) {
            float acc = 0.0f;
#pragma unroll
            for (int q = 0; q < NR; ++q) acc = acc + Payload<DT>::widen1(static_cast<const T_*>(in.p[q])[i]);
            const int jt = (int)(i / (cvec * kVecElems<DT>));
            static_cast<T_*>(out.p[jt])[i] = Payload<DT>::narrow1(acc);
            const T_ y = static_cast<const T_*>(out.p[jt])[i];
#pragma unroll
            for (int q = 0; q < NR; ++q)
                if (q != jt) static_cast<T_*>(out.p[q])[i] = y;
        }
    }
    // the last CTA to finish (every CTA has taken its ticket) resets the counters
    if (lag > 0 && threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(sync + 1, 1u) == gridDim.x - 1) {
            st_relaxed_u32(sync, 0u);
            st_relaxed_u32(sync + 1, 0u);
            st_release_u32(sync + 2, epoch);
        }
    }
}

}  // namespace

// u32 words of the one-launch form's sync buffer for handles of n ranks and
// max_bytes per rank: 4 counters + one flag per phase-1 item at the smallest
// tile (one warp of one vector per thread).
size_t two_shot_sync_words(int n, size_t max_bytes)
{
    size_t most = 0;
    for (int dt = AR_F32; dt <= AR_F16; ++dt) {
        const size_t cvec = chunk_elems(n, max_bytes / elem_bytes(dt), dt) / (16u / elem_bytes(dt));
        const size_t items = (size_t)n * ((cvec + 31u) / 32u);
        if (items > most) most = items;
    }
    return 4u + most;
}

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
            // a call too small to give every SM a full CTA: narrower CTAs, one vector per thread
            const bool narrow = g_rs.x * NR < (unsigned)h.sm_count;
            const Shape sh = narrow_shape(h, cvec, NR);
            const bool one_launch = two_shot_one_launch(h.two_shot_impl);
            if (one_launch) {
                // one tile per CTA: phase 1 of tile t, then phase 2 of tile t (form 2) or of
                // the tile of ticket t - lag (form 3)
                constexpr int UF = flagged_unroll<NR>();
                const unsigned block = narrow ? sh.block : (unsigned)kThreads;
                const size_t T = (size_t)block * (narrow ? 1 : UF);
                const size_t tpc = (cvec + T - 1) / T;
                const size_t R = (size_t)NR * tpc;
                if (4 + R > h.two_shot_sync_words) return AR_ERR_TOO_LARGE;  // never: sized at create
                const int per_sm = narrow ? 3 * (kThreads / (int)block) : flagged_ctas_per_sm<NR>();
                size_t lag = h.two_shot_impl == 3 ? (size_t)h.sm_count * (size_t)per_sm : 0;
                if (lag > R) lag = R;
                const size_t grid = R + lag;
                rec_begin(h, s);
                if (narrow)
                    launch_kernel(h, two_shot_one_launch_kernel<NR, DT, 1, true>, dim3((unsigned)grid), block, 0, s, ip,
                                  op, nvec, count, cvec, (unsigned)tpc, (unsigned)lag, h.two_shot_sync, h.status,
                                  h.spin_ns);
                else
                    launch_kernel(h, two_shot_one_launch_kernel<NR, DT, UF, false>, dim3((unsigned)grid), kThreads, 0, s,
                                  ip, op, nvec, count, cvec, (unsigned)tpc, (unsigned)lag, h.two_shot_sync, h.status,
                                  h.spin_ns);
                rec_end(h, s, AR_K_TWO_SHOT, (uint64_t)(2 * NR + 1) * S);
                *launches = 1;
                return launch_status();
            }
            const dim3 g_ag(grid_for_rows(h, (cvec + kAgUnroll - 1) / kAgUnroll, NR), NR);
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
