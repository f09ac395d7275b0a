// Two other ways to run the one-shot all-reduce, both named by the pages.
//
// Push ("SGLang JIT custom all-reduce" notes, §实现: one-shot pull, one-shot
// push and two-shot pull): every rank writes its buffer into a staging slot
// of every peer, then every rank reduces its own staging slots locally.  The
// emulation keeps one staging slot per (receiving rank, sending rank) pair in
// the handle (n x n x max_bytes, allocated by AR_OPT_PUSH_STAGING).  Push
// phase: reads n S, writes n (n-1) S; reduce phase: every rank reads its n
// slots (its own input in place of its own slot) and writes its output:
// reads n^2 S, writes n S.
//
// Copy-in (same notes, §5 写回: outside graph capture the kernel reads a
// pre-registered pull buffer that cudaMemcpyAsync filled from the input, and
// the output may then be the input itself): each rank's input is copied into
// its registered buffer (AR_OPT_REGISTERED, n x max_bytes), then the one-shot
// kernel reads the registered buffers.  The pages issue one cudaMemcpyAsync
// per rank; here one launch copies all n buffers (blockIdx.y = rank), which
// costs one launch instead of n copies of a few microseconds each at decode
// sizes.  HBM: the copy reads n S and writes n S.
//
// Both give the one-shot result bit for bit: fp32 sums in rank order from +0,
// one rounding.
//
// Pieces: when the staged bytes (push: n (n-1) S; copy-in: n S) exceed half
// of L2, the buffers are cut into pieces that each go through both launches
// in turn, so the second launch reads the staging back from L2 (same bits,
// same HBM bytes, twice the launches per piece).
//
// Small: a call too small to give every SM a full CTA runs its kernels in
// narrower CTAs compiled for three CTAs per SM, as the one-shot kernel's small
// form (blockIdx.y = rank rows; one 16-byte vector per thread).
#include "common.cuh"

namespace argb {
namespace {

// stage[q][r] for r != q  <-  in[r].   Grid: blockIdx.y = sending rank r.
template <int NR, int DT, bool Small>
__global__ void __launch_bounds__(kThreads, Small ? 3 : 0)
push_kernel(const __grid_constant__ CPtrs<NR> in, uint8_t* __restrict__ stage, size_t slot_bytes, size_t nvec,
            size_t count)
{
    pdl_acquire();
    using T = typename Payload<DT>::scalar_t;
    const int r = blockIdx.y;
    const uint4* const src = static_cast<const uint4*>(in.p[r]);
    const size_t bs = Small ? (size_t)blockDim.x : (size_t)kThreads;
    for (size_t v = (size_t)blockIdx.x * bs + threadIdx.x; v < nvec; v += (size_t)gridDim.x * bs) {
        const uint4 x = ld16(src + v);
#pragma unroll
        for (int q = 0; q < NR; ++q)
            if (q != r) st16_next(reinterpret_cast<uint4*>(stage + ((size_t)q * NR + r) * slot_bytes) + v, x);
    }
    pdl_release();
    if (blockIdx.x == gridDim.x - 1) {
        const size_t i = nvec * kVecElems<DT> + threadIdx.x;
        if (i < count) {
            const T x = static_cast<const T*>(in.p[r])[i];
#pragma unroll
            for (int q = 0; q < NR; ++q)
                if (q != r) reinterpret_cast<T*>(stage + ((size_t)q * NR + r) * slot_bytes)[i] = x;
        }
    }
}

// out[q] = rank-order sum of stage[q][0..n-1], with in[q] as rank q's own term.
// Grid: blockIdx.y = receiving rank q.
template <int NR, int DT, bool Small>
__global__ void __launch_bounds__(kThreads, Small ? 3 : 0)
push_reduce_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out,
                   const uint8_t* __restrict__ stage, size_t slot_bytes, size_t nvec, size_t count)
{
    pdl_acquire();
    using T = typename Payload<DT>::scalar_t;
    const int q = blockIdx.y;
    auto slot = [&](int r) -> const void* {
        return r == q ? in.p[q] : static_cast<const void*>(stage + ((size_t)q * NR + r) * slot_bytes);
    };
    uint4* const dst = static_cast<uint4*>(out.p[q]);
    const size_t bs = Small ? (size_t)blockDim.x : (size_t)kThreads;
    for (size_t v = (size_t)blockIdx.x * bs + threadIdx.x; v < nvec; v += (size_t)gridDim.x * bs) {
        uint4 x[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) x[r] = ld16_last(static_cast<const uint4*>(slot(r)) + v);   // staged once
        st16(dst + v, reduce_rank_order<DT, NR>(x));
    }
    pdl_release();
    if (blockIdx.x == gridDim.x - 1) {
        const size_t i = nvec * kVecElems<DT> + threadIdx.x;
        if (i < count) {
            float acc = 0.0f;
#pragma unroll
            for (int r = 0; r < NR; ++r) acc = acc + Payload<DT>::widen1(static_cast<const T*>(slot(r))[i]);
            static_cast<T*>(out.p[q])[i] = Payload<DT>::narrow1(acc);
        }
    }
}

// reg[r] <- in[r] for every rank r.  Grid: blockIdx.y = rank.
template <int NR, int DT, bool Small>
__global__ void __launch_bounds__(kThreads, Small ? 3 : 0)
copyin_kernel(const __grid_constant__ CPtrs<NR> in, uint8_t* __restrict__ reg, size_t slot_bytes, size_t nvec,
              size_t count)
{
    pdl_acquire();
    using T = typename Payload<DT>::scalar_t;
    const int r = blockIdx.y;
    const uint4* const src = static_cast<const uint4*>(in.p[r]);
    uint4* const dst = reinterpret_cast<uint4*>(reg + (size_t)r * slot_bytes);
    const size_t bs = Small ? (size_t)blockDim.x : (size_t)kThreads;
    for (size_t v = (size_t)blockIdx.x * bs + threadIdx.x; v < nvec; v += (size_t)gridDim.x * bs)
        st16_next(dst + v, ld16(src + v));   // the one-shot launch after it reads it
    pdl_release();
    if (blockIdx.x == gridDim.x - 1) {
        const size_t i = nvec * kVecElems<DT> + threadIdx.x;
        if (i < count) reinterpret_cast<T*>(dst)[i] = static_cast<const T*>(in.p[r])[i];
    }
}

}  // namespace

int launch_one_shot_push(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
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
            using T = typename Payload<DT>::scalar_t;
            // pieces: the staged bytes, n (n - 1) S, over half of L2, rounded; each piece staged
            // and reduced in turn, so its staging is read back from L2.  Measured on GB300 (n = 8
            // bf16, back to back; pieces -> us): at 8 MiB per rank 1 -> 162.6, 4 -> 148.5,
            // 7 -> 143.4, 8 -> 142.4, 12 -> 156.0; at 64 MiB 1 -> 1357, 32 -> 1210, 57 -> 1150,
            // 64 -> 1152; at 2 MiB 1 -> 36.3, 2 -> 34.8; at 1 MiB one piece is fastest.  Two streams
            // (PieceStreams, twice the pieces) when the staged bytes exceed half of L2: at 2 / 8 /
            // 64 MiB 35.0 -> 33.6, 144 -> 125, 1168 -> 1012 us; at 1 MiB 16.0 -> 16.8 (one stream).
            const uint64_t staged = (uint64_t)NR * (NR - 1) * count * sizeof(T);
            const bool dual = two_streams(h, staged, 2);
            size_t PL = piece_elems(h, staged, count);
            if (dual) PL = half_piece(PL, count);
            const size_t pv = PL / kVecElems<DT>;
            const dim3 grid(grid_for_rows(h, pv ? pv : 1, NR), NR);
            const bool small = grid.x * NR < (unsigned)h.sm_count;   // narrower CTAs, as one-shot's small form
            const Shape sh = narrow_shape(h, pv ? pv : 1, NR);
            const dim3 g_small(sh.grid_x, NR);
            int nl = 0, rc = AR_OK;
            PieceStreams streams{h, s, dual};
            if (streams.fork() != AR_OK) return AR_ERR_CUDA;
            for (size_t p_lo = 0; p_lo < count && rc == AR_OK; p_lo += PL) {
                const size_t pc = count - p_lo < PL ? count - p_lo : PL;   // the piece's elements
                const uint64_t S = (uint64_t)pc * sizeof(T);
                const cudaStream_t s = streams.next();   // this piece's stream
                // the piece: every pointer moved to its first element (within each staging slot too)
                CPtrs<NR> ipp;
                MPtrs<NR> opp;
                for (int q = 0; q < NR; ++q) {
                    ipp.p[q] = static_cast<const T*>(in[q]) + p_lo;
                    opp.p[q] = static_cast<T*>(out[q]) + p_lo;
                }
                uint8_t* const st = h.push_stage + p_lo * sizeof(T);
                rec_begin(h, s);
                if (small)
                    launch_kernel(h, push_kernel<NR, DT, true>, g_small, sh.block, 0, s, ipp, st, h.stage_slot,
                                  pc / kVecElems<DT>, pc);
                else
                    launch_kernel(h, push_kernel<NR, DT, false>, grid, kThreads, 0, s, ipp, st, h.stage_slot,
                                  pc / kVecElems<DT>, pc);
                rec_end(h, s, AR_K_PUSH, (uint64_t)NR * S + (uint64_t)NR * (NR - 1) * S);
                if (launch_status() != AR_OK) {
                    rc = AR_ERR_CUDA;
                    break;
                }
                rec_begin(h, s);
                if (small)
                    launch_kernel(h, push_reduce_kernel<NR, DT, true>, g_small, sh.block, 0, s, ipp, opp,
                                  (const uint8_t*)st, h.stage_slot, pc / kVecElems<DT>, pc);
                else
                    launch_kernel(h, push_reduce_kernel<NR, DT, false>, grid, kThreads, 0, s, ipp, opp,
                                  (const uint8_t*)st, h.stage_slot, pc / kVecElems<DT>, pc);
                rec_end(h, s, AR_K_PUSH_REDUCE, (uint64_t)NR * NR * S + (uint64_t)NR * S);
                if (launch_status() != AR_OK) rc = AR_ERR_CUDA;
                nl += 2;
            }
            if (streams.join() != AR_OK) rc = AR_ERR_CUDA;
            *launches = nl;
            return rc;
        });
    });
}

int launch_one_shot_copyin(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                           cudaStream_t s, int* launches)
{
    // pieces: the registered copy, n S, over half of L2, rounded; each piece copied and then
    // reduced by the one-shot kernel, so the one-shot reads the copy back from L2.  Measured on
    // GB300 (n = 8 bf16, back to back; pieces -> us): at 64 MiB per rank 1 -> 308.4, 4 -> 286.0,
    // 8 -> 277.1, 12 -> 286.7; at 16 MiB 1 -> 71.8, 2 -> 68.2, 4 -> 76.4; at 8 MiB one piece is
    // fastest.  Two streams (PieceStreams, twice the pieces) when n S exceeds half of L2: at
    // 16 / 64 MiB 68.3 -> 67.0, 279 -> 260 us; equal at 8 MiB.
    const size_t e = elem_bytes(dt);
    const bool dual = two_streams(h, (uint64_t)h.n * count * e, 2);
    size_t PL = piece_elems(h, (uint64_t)h.n * count * e, count);
    if (dual) PL = half_piece(PL, count);
    PieceStreams streams{h, s, dual};
    if (streams.fork() != AR_OK) return AR_ERR_CUDA;
    int total = 0, rc_all = AR_OK;
    for (size_t p_lo = 0; p_lo < count && rc_all == AR_OK; p_lo += PL) {
        const size_t pc = count - p_lo < PL ? count - p_lo : PL;   // the piece's elements
        const cudaStream_t s = streams.next();   // this piece's stream
        const int rc = dispatch_dtype(dt, [&](auto dtc) -> int {
            constexpr int DT = decltype(dtc)::value;
            return dispatch_ranks(h.n, [&](auto nrc) -> int {
                constexpr int NR = decltype(nrc)::value;
                using T = typename Payload<DT>::scalar_t;
                CPtrs<NR> ip;
                for (int q = 0; q < NR; ++q) ip.p[q] = static_cast<const T*>(in[q]) + p_lo;
                const size_t nvec = pc / kVecElems<DT>;
                const uint64_t S = (uint64_t)pc * sizeof(T);
                const dim3 grid(grid_for_rows(h, nvec ? nvec : 1, NR), NR);
                const Shape sh = narrow_shape(h, nvec ? nvec : 1, NR);
                uint8_t* const reg = h.registered + p_lo * sizeof(T);
                rec_begin(h, s);
                if (grid.x * NR < (unsigned)h.sm_count)   // narrower CTAs, as one-shot's small form
                    launch_kernel(h, copyin_kernel<NR, DT, true>, dim3(sh.grid_x, NR), sh.block, 0, s, ip, reg,
                                  h.stage_slot, nvec, pc);
                else
                    launch_kernel(h, copyin_kernel<NR, DT, false>, grid, kThreads, 0, s, ip, reg, h.stage_slot,
                                  nvec, pc);
                rec_end(h, s, AR_K_COPYIN, 2ull * NR * S);
                return launch_status();
            });
        });
        if (rc != AR_OK) {
            rc_all = rc;
            break;
        }
        const void* reg[kMaxRanks];
        void* op[kMaxRanks];
        for (int r = 0; r < h.n; ++r) {
            reg[r] = h.registered + (size_t)r * h.stage_slot + p_lo * e;
            op[r] = static_cast<uint8_t*>(out[r]) + p_lo * e;
        }
        int one = 0;
        const int rc2 = launch_one_shot(h, reg, op, pc, dt, s, &one);
        if (rc2 != AR_OK) rc_all = rc2;
        total += 1 + one;
    }
    if (streams.join() != AR_OK) rc_all = AR_ERR_CUDA;
    *launches = total;
    return rc_all;
}

}  // namespace argb
