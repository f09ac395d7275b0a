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
#include "bulk.cuh"
#include "common.cuh"

namespace argb {
namespace {

// Vectors per thread per iteration: keeps about 128-256 B of loads in flight
// per thread without spilling at n = 16.
template <int NR> __host__ __device__ constexpr int one_shot_unroll() { return NR <= 4 ? 4 : NR <= 8 ? 2 : 1; }

// U vectors per thread per iteration, in CTAs of up to kThreads threads.
// Small: a call too small to give every SM a full CTA, run with U = 1 and
// narrower CTAs, and compiled for three CTAs per SM (at most 80 registers;
// a minimum of 0 leaves the full-size form to the compiler's own choice).
// That bound matters for latency: measured on GB300 (n = 8 and 16 bf16,
// CUDA-graph replay), the compiler's own register choice ran calls of 8 KiB -
// 1 MiB per rank 0.2-1.9 us slower, while for full-size calls the bound
// gains nothing and costs up to 5% at 2 MiB.
template <int NR, int DT, int U, bool Small>
__global__ void __launch_bounds__(kThreads, Small ? 3 : 0)
one_shot_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t nvec, size_t count)
{
    pdl_acquire();
    const size_t bs = U > 1 ? (size_t)kThreads : (size_t)blockDim.x, span = bs * U;  // U > 1: full CTAs only
    for (size_t base = (size_t)blockIdx.x * span; base < nvec; base += (size_t)gridDim.x * span) {
        uint4 x[U][NR];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = base + (size_t)u * bs + threadIdx.x;
            if (v < nvec) {
#pragma unroll
                for (int q = 0; q < NR; ++q) x[u][q] = ld16(static_cast<const uint4*>(in.p[q]) + v);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t v = base + (size_t)u * bs + threadIdx.x;
            if (v < nvec) {
                const uint4 r = reduce_rank_order<DT, NR>(x[u]);
#pragma unroll
                for (int q = 0; q < NR; ++q) st16(static_cast<uint4*>(out.p[q]) + v, r);
            }
        }
    }
    pdl_release();
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

// ---- bulk-copy staging variant (AR_OPT_ONE_SHOT_IMPL = 2) -----------------
// Each CTA walks tiles of kBulkTile bytes per rank.  Thread 0 issues one
// cp.async.bulk load per rank into a pipeline stage (completion on the
// stage's mbarrier), all threads sum the stage from shared memory in rank
// order into a result tile, and thread 0 issues one bulk store of that tile
// per rank output: the n-way fan-out of the write is done by the copy
// engine from a single shared-memory tile.  Stages are refilled as soon as
// they are consumed; the result tile is double-buffered.

constexpr uint32_t kBulkTile = kThreads * 16;     // one 16-byte vector per thread per rank
constexpr int kBulkSmemBudget = 200 * 1024;

template <int NR> __host__ __device__ constexpr int bulk_stages()
{
    return (kBulkSmemBudget - 2 * (int)kBulkTile) / (NR * (int)kBulkTile) < 2   ? 2
           : (kBulkSmemBudget - 2 * (int)kBulkTile) / (NR * (int)kBulkTile) > 8 ? 8
           : (kBulkSmemBudget - 2 * (int)kBulkTile) / (NR * (int)kBulkTile);
}

template <int NR> __host__ __device__ constexpr int bulk_smem_bytes()
{
    return (bulk_stages<NR>() * NR + 2) * (int)kBulkTile;
}

template <int NR, int DT>
__global__ void __launch_bounds__(kThreads, 1)
one_shot_bulk_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t nvec,
                     size_t count, DevStatus* st)
{
    pdl_acquire();
    constexpr int P = bulk_stages<NR>();
    constexpr uint32_t T = kBulkTile;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bar[P];
    uint8_t* const res_base = smem + (size_t)P * NR * T;
    const int tid = threadIdx.x;
    const size_t nbytes = nvec * 16;
    const size_t ntiles = (nbytes + T - 1) / T;
    auto tile_bytes = [&](size_t t) -> uint32_t { return (uint32_t)(nbytes - t * T < T ? nbytes - t * T : T); };
    auto issue = [&](int s, size_t t) {
        const uint32_t b = tile_bytes(t);
        mbar_arrive_expect_tx(&bar[s], b * NR);
#pragma unroll
        for (int q = 0; q < NR; ++q)
            bulk_load(smem + ((size_t)s * NR + q) * T, static_cast<const uint8_t*>(in.p[q]) + t * T, b, &bar[s]);
    };

    if (tid == 0) {
        for (int s = 0; s < P; ++s) mbar_init(&bar[s], 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (tid == 0)
        for (int s = 0; s < P; ++s)
            if (blockIdx.x + (size_t)s * gridDim.x < ntiles) issue(s, blockIdx.x + (size_t)s * gridDim.x);

    size_t it = 0;
    bool failed = false;
    for (size_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int s = (int)(it % P);
        const bool ok = mbar_wait(&bar[s], (uint32_t)((it / P) & 1));
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        const uint32_t b = tile_bytes(t);
        uint8_t* const res = res_base + (it & 1) * T;
        if ((uint32_t)tid * 16 < b) {
            uint4 x[NR];
#pragma unroll
            for (int q = 0; q < NR; ++q) x[q] = lds16(smem + ((size_t)s * NR + q) * T + tid * 16);
            sts16(res + tid * 16, reduce_rank_order<DT, NR>(x));
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int q = 0; q < NR; ++q) bulk_store(static_cast<uint8_t*>(out.p[q]) + t * T, res, b);
            bulk_commit();
            const size_t tn = t + (size_t)P * gridDim.x;
            if (tn < ntiles) issue(s, tn);
            bulk_wait_read<1>();  // the other result tile is free again
        }
        __syncthreads();
    }
    pdl_release();
    if (tid == 0) {
        if (failed) {
            report_wait_timeout(st);
            // loads still in flight land in this CTA's shared memory: wait for
            // each issued stage (bounded) before the CTA exits
            for (int k = 0; k < P; ++k) {
                const size_t j = it + k;
                if (blockIdx.x + j * gridDim.x < ntiles) (void)mbar_wait(&bar[j % P], (uint32_t)((j / P) & 1));
            }
        }
        bulk_wait_all<0>();
    }
    if (blockIdx.x == gridDim.x - 1) {
        using T_ = typename Payload<DT>::scalar_t;
        const size_t i = nvec * kVecElems<DT> + tid;
        if (i < count) {
            float acc = 0.0f;
#pragma unroll
            for (int q = 0; q < NR; ++q) acc = acc + Payload<DT>::widen1(static_cast<const T_*>(in.p[q])[i]);
            const T_ r = Payload<DT>::narrow1(acc);
#pragma unroll
            for (int q = 0; q < NR; ++q) static_cast<T_*>(out.p[q])[i] = r;
        }
    }
}

// Opts the kernel into its shared-memory size on the current device (once per
// device).
template <int NR, int DT>
bool bulk_attributes()
{
    static std::atomic<uint32_t> done{0};
    return once_per_device(done, [] {
        return cudaFuncSetAttribute(one_shot_bulk_kernel<NR, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    bulk_smem_bytes<NR>()) == cudaSuccess;
    });
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
            const uint64_t S = (uint64_t)count * sizeof(typename Payload<DT>::scalar_t);
            if (h.one_shot_impl == 2) {
                constexpr int smem = bulk_smem_bytes<NR>();
                if (!bulk_attributes<NR, DT>()) return AR_ERR_CUDA;
                static const int per_sm = blocks_per_sm(one_shot_bulk_kernel<NR, DT>, smem);
                const size_t ntiles = (nvec * 16 + kBulkTile - 1) / kBulkTile;
                size_t grid = (size_t)h.sm_count * (size_t)(h.ctas_per_sm ? h.ctas_per_sm : per_sm);
                if (grid > ntiles) grid = ntiles;
                if (grid == 0) grid = 1;
                rec_begin(h, s);
                launch_kernel(h, one_shot_bulk_kernel<NR, DT>, (unsigned)grid, kThreads, smem, s, ip, op, nvec, count, h.status);
                rec_end(h, s, AR_K_ONE_SHOT, 2ull * NR * S);
            } else {
                constexpr int U = one_shot_unroll<NR>();
                const unsigned grid = grid_for(h, (nvec + U - 1) / U);
                rec_begin(h, s);
                if (grid < (unsigned)h.sm_count) {
                    const Shape sh = narrow_shape(h, nvec);
                    launch_kernel(h, one_shot_kernel<NR, DT, 1, true>, sh.grid_x, sh.block, 0, s, ip, op, nvec,
                                  count);
                } else
                    launch_kernel(h, one_shot_kernel<NR, DT, U, false>, grid, kThreads, 0, s, ip, op, nvec, count);
                rec_end(h, s, AR_K_ONE_SHOT, 2ull * NR * S);
            }
            *launches = 1;
            return launch_status();
        });
    });
}

}  // namespace argb
