// Pairwise tree all-reduce (recursive doubling), emulated level by level.
//
// The PCIe-IPC blog post (bhfrc.com/news/61376, §3.1 算法骨架) pairs the
// ranks up: in each of log2(n) levels every rank reads its own data
// and its peer's, adds them, and writes the sum back to both.  At level l
// rank r pairs with r XOR 2^l, so n must be a power of two.  The buffers hold
// the payload type, so every level's sum is one binary32 add of the two
// widened values, rounded to the payload type.  Both members of a pair add the
// same two values, so one thread computes the sum once and writes it to both.
//
// Emulation: one launch per level.  Level 0 reads in[r], in[r ^ 1] and writes
// out[r], out[r ^ 1]; later levels work in place on out[].  Every element of
// every rank is read once and written once per level: HBM per level n S read,
// n S write.  A call whose level output (n S) is larger than half of L2 runs
// in pieces, each through all levels (handbook "集合通信：NCCL 的算法、协议与
// 推理框架的定制 all-reduce", §算法: a tree cuts a large message into blocks
// and pipelines them): P = n S over half of L2, rounded, so one piece's level
// output stays in L2 for the next level.  Same sums, same HBM bytes.
#include "common.cuh"

namespace argb {
namespace {

// One level.  Grid: blockIdx.y = pair j in [0, NR/2); its lower rank r has
// bit `d` clear, its upper rank is r | d.
template <int NR, int DT>
__global__ void __launch_bounds__(kThreads)
tree_level_kernel(const __grid_constant__ CPtrs<NR> src, const __grid_constant__ MPtrs<NR> dst, int d, size_t nvec,
                  size_t count)
{
    pdl_acquire();
    using T = typename Payload<DT>::scalar_t;
    constexpr int VE = kVecElems<DT>;
    const int j = blockIdx.y;
    const int r = ((j & ~(d - 1)) << 1) | (j & (d - 1));   // j with a 0 inserted at bit log2(d)
    const int p = r | d;
    const uint4* const a = static_cast<const uint4*>(src.p[r]);
    const uint4* const b = static_cast<const uint4*>(src.p[p]);
    uint4* const oa = static_cast<uint4*>(dst.p[r]);
    uint4* const ob = static_cast<uint4*>(dst.p[p]);
    for (size_t v = (size_t)blockIdx.x * kThreads + threadIdx.x; v < nvec; v += (size_t)gridDim.x * kThreads) {
        const uint4 xa = ld16(a + v), xb = ld16(b + v);
        float fa[VE], fb[VE];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            Payload<DT>::widen(word(xa, w), fa + w * Payload<DT>::kPerWord);
            Payload<DT>::widen(word(xb, w), fb + w * Payload<DT>::kPerWord);
        }
#pragma unroll
        for (int k = 0; k < VE; ++k) fa[k] = fa[k] + fb[k];
        const uint4 y = round_vec<DT>(fa);
        st16_next(oa + v, y);   // the next level reads it
        st16_next(ob + v, y);
    }
    pdl_release();
    if (blockIdx.x == gridDim.x - 1) {   // the ragged tail (< VE elements)
        const size_t i = nvec * VE + threadIdx.x;
        if (i < count) {
            const float y = Payload<DT>::widen1(static_cast<const T*>(src.p[r])[i]) +
                            Payload<DT>::widen1(static_cast<const T*>(src.p[p])[i]);
            static_cast<T*>(dst.p[r])[i] = Payload<DT>::narrow1(y);
            static_cast<T*>(dst.p[p])[i] = Payload<DT>::narrow1(y);
        }
    }
}

}  // namespace

int launch_tree(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                int* launches)
{
    if (h.n & (h.n - 1)) return AR_ERR_INVALID;
    return dispatch_dtype(dt, [&](auto dtc) -> int {
        constexpr int DT = decltype(dtc)::value;
        return dispatch_ranks(h.n, [&](auto nrc) -> int {
            constexpr int NR = decltype(nrc)::value;
            using T = typename Payload<DT>::scalar_t;
            const uint64_t S = (uint64_t)count * sizeof(T);
            // pieces: a level's output (n S) over half of L2, rounded.  Measured on GB300 (bf16,
            // back to back; pieces -> us): n = 8 at 64 MiB per rank 1 -> 472, 4 -> 444, 6 -> 381,
            // 8 -> 364, 12 -> 370, 16 -> 384; at 16 MiB 1 -> 112, 2 -> 89, 4 -> 96; at 8 MiB and
            // below one piece was fastest; n = 16 at 16 MiB 1 -> 317, 4 -> 226, 8 -> 244, and at
            // 64 MiB 1 -> 1258, 16 -> 959, 24 -> 939; n = 4 at 64 MiB 1 -> 159, 4 -> 131.  A piece
            // is passed as every pointer moved to its first element.  Two streams (PieceStreams,
            // twice the pieces) when the level output exceeds half of L2: n = 8 at 8 / 16 / 64 MiB
            // 44.9 -> 43.5, 89.2 -> 82.5, 364 -> 324 us; n = 16 at 16 / 64 MiB 225 -> 200, 961 ->
            // 848 us; equal at 4 MiB.
            const bool dual = two_streams(h, (uint64_t)NR * S, 2);
            size_t PL = piece_elems(h, (uint64_t)NR * S, count);
            if (dual) PL = half_piece(PL, count);
            PieceStreams streams{h, s, dual};
            if (streams.fork() != AR_OK) return AR_ERR_CUDA;
            int rc = AR_OK;
            const size_t pvec = PL / kVecElems<DT>;
            const dim3 grid(grid_for_rows(h, pvec ? pvec : 1, NR / 2), NR / 2);
            int levels = 0, n_launch = 0;
            rec_begin(h, s);
            for (size_t p_lo = 0; p_lo < count && rc == AR_OK; p_lo += PL) {
                const size_t pc = count - p_lo < PL ? count - p_lo : PL;   // the piece's elements
                const cudaStream_t ps = streams.next();   // this piece's stream
                CPtrs<NR> ipp, opc;
                MPtrs<NR> opp;
                for (int q = 0; q < NR; ++q) {
                    ipp.p[q] = static_cast<const T*>(in[q]) + p_lo;
                    opc.p[q] = static_cast<const T*>(out[q]) + p_lo;
                    opp.p[q] = static_cast<T*>(out[q]) + p_lo;
                }
                levels = 0;
                for (int d = 1; d < NR; d <<= 1, ++levels, ++n_launch) {
                    if (launch_kernel(h, tree_level_kernel<NR, DT>, grid, kThreads, 0, ps, d == 1 ? ipp : opc, opp, d,
                                      pc / kVecElems<DT>, pc) != cudaSuccess)
                        rc = AR_ERR_CUDA;
                }
            }
            if (streams.join() != AR_OK) rc = AR_ERR_CUDA;
            rec_end(h, s, AR_K_TREE_LEVEL, 2ull * NR * S * (uint64_t)levels, n_launch);
            *launches = n_launch;
            return rc != AR_OK ? rc : launch_status();
        });
    });
}

}  // namespace argb

// ---------------------------------------------------------------------------
// The same tree with every level done in registers, in one pass.
//
// The levels have no dependency across elements, so on one GPU a thread can
// load the n ranks' values of its 16-byte vector once, run all log2(n)
// pairwise levels on them (the same pairs, the same binary32 adds, the same
// rounding to the payload type after every level), and store the n results:
// HBM reads n S and writes n S, as one-shot does, instead of log2(n) times
// that.  Same bits as the level-by-level tree.
namespace argb {
namespace {

// Small: a call too small to give every SM a full CTA, in narrower CTAs and
// compiled for three CTAs per SM (for latency, as the one-shot kernel).
template <int NR, int DT, bool Small>
__global__ void __launch_bounds__(kThreads, Small ? 3 : 0)
tree_fused_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t nvec,
                  size_t count)
{
    pdl_acquire();
    using T = typename Payload<DT>::scalar_t;
    constexpr int P = Payload<DT>::kPerWord;   // elements per 32-bit word
    constexpr int VE = kVecElems<DT>;
    // all levels over one value per rank, rounded after each level
    auto levels = [](float (&f)[NR]) {
#pragma unroll
        for (int d = 1; d < NR; d <<= 1) {
            float g[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) g[r] = Payload<DT>::widen1(Payload<DT>::narrow1(f[r] + f[r ^ d]));
#pragma unroll
            for (int r = 0; r < NR; ++r) f[r] = g[r];
        }
    };
    const size_t bs = Small ? (size_t)blockDim.x : (size_t)kThreads;   // the full-size form: kThreads-thread CTAs
    for (size_t v = (size_t)blockIdx.x * bs + threadIdx.x; v < nvec; v += (size_t)gridDim.x * bs) {
        uint4 x[NR];
#pragma unroll
        for (int q = 0; q < NR; ++q) x[q] = ld16(static_cast<const uint4*>(in.p[q]) + v);
        uint32_t y[NR][4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            float e[NR][P];
#pragma unroll
            for (int q = 0; q < NR; ++q) Payload<DT>::widen(word(x[q], w), e[q]);
#pragma unroll
            for (int k = 0; k < P; ++k) {
                float f[NR];
#pragma unroll
                for (int q = 0; q < NR; ++q) f[q] = e[q][k];
                levels(f);
#pragma unroll
                for (int q = 0; q < NR; ++q) e[q][k] = f[q];
            }
#pragma unroll
            for (int q = 0; q < NR; ++q) y[q][w] = Payload<DT>::narrow(e[q]);
        }
#pragma unroll
        for (int q = 0; q < NR; ++q)
            st16(static_cast<uint4*>(out.p[q]) + v, make_uint4(y[q][0], y[q][1], y[q][2], y[q][3]));
    }
    pdl_release();
    if (blockIdx.x == gridDim.x - 1) {   // the ragged tail (< VE elements)
        const size_t i = nvec * VE + threadIdx.x;
        if (i < count) {
            float f[NR];
#pragma unroll
            for (int q = 0; q < NR; ++q) f[q] = Payload<DT>::widen1(static_cast<const T*>(in.p[q])[i]);
            levels(f);
#pragma unroll
            for (int q = 0; q < NR; ++q) static_cast<T*>(out.p[q])[i] = Payload<DT>::narrow1(f[q]);
        }
    }
}

}  // namespace

int launch_tree_fused(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                      int* launches)
{
    if (h.n & (h.n - 1)) return AR_ERR_INVALID;
    return dispatch_dtype(dt, [&](auto dtc) -> int {
        constexpr int DT = decltype(dtc)::value;
        return dispatch_ranks(h.n, [&](auto nrc) -> int {
            constexpr int NR = decltype(nrc)::value;
            if constexpr ((NR & (NR - 1)) != 0) {
                return AR_ERR_INVALID;
            } else {
                CPtrs<NR> ip;
                MPtrs<NR> op;
                for (int q = 0; q < NR; ++q) {
                    ip.p[q] = in[q];
                    op.p[q] = out[q];
                }
                const size_t nvec = count / kVecElems<DT>;
                const uint64_t S = (uint64_t)count * sizeof(typename Payload<DT>::scalar_t);
                // full CTAs, or narrower ones spread over more SMs for a small call
                const unsigned grid = grid_for(h, nvec);
                rec_begin(h, s);
                if (grid < (unsigned)h.sm_count) {
                    const Shape sh = narrow_shape(h, nvec);
                    launch_kernel(h, tree_fused_kernel<NR, DT, true>, sh.grid_x, sh.block, 0, s, ip, op, nvec, count);
                } else {
                    launch_kernel(h, tree_fused_kernel<NR, DT, false>, grid, kThreads, 0, s, ip, op, nvec, count);
                }
                rec_end(h, s, AR_K_TREE_FUSED, 2ull * NR * S);
                *launches = 1;
                return launch_status();
            }
        });
    });
}

}  // namespace argb
