// All-reduce fused with residual add and RMSNorm: the decode epilogue of a
// tensor-parallel layer in one launch.
//
// Handbook "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce",
// §源码对照, names such a fused all-reduce + RMSNorm kernel (FlashInfer's)
// without defining it; "多 GPU 与 NCCL", §为什么要多卡 puts the all-reduce at
// the end of every tensor-parallel attention and MLP block.  The result is
// that of the unfused chain:
//   a = all-reduce of in[*] (rank-order fp32 sum, rounded to the payload)
//   r = RN(a + residual)                          -> residual_out
//   y = RN(r * 1/sqrt(mean(r^2) + eps) * weight)  -> norm_out[0..n-1]
//
// Layout: one thread-block cluster of CL CTAs per token row (16, a
// non-portable cluster size, unless the row is too short to give each CTA 64
// vectors and the rows are many: then 8); CTA c of the cluster owns a
// contiguous slice of the row, and its TH threads (64 to 256, the slice
// rounded up) take one 16-byte vector each, further ones in turn.  Pass 1
// reads the n rank slices once, writes r, keeps r (fp32: a thread's first
// vector in registers, any further ones in shared memory) and accumulates its
// squares.  Each warp then sends its sum of squares straight into every CTA's
// shared memory (distributed shared memory) with an asynchronous store
// counted on the receiver's mbarrier; every thread waits only until the CL x
// warps partials have landed in its own CTA and adds them in one fixed order
// (no CTA-wide barrier anywhere), and pass 2 scales r and writes every rank's
// output.
// HBM: reads n S + S (+ the weight, H per launch), writes n S + S.
#include "common.cuh"

namespace argb {
namespace {

constexpr int kClusterCtas = 8;   // the smallest cluster: it sizes the longest slice a CTA keeps

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t to_cluster(const void* local, uint32_t cta)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(cta));
    return remote;
}

// Write v to CTA `cta`'s shared memory, at the offset of `local` in ours, and
// count its 4 bytes on that CTA's barrier at the offset of `bar` in ours.
__device__ __forceinline__ void st_async_cluster_f32(float* local, const uint64_t* bar, uint32_t cta, float v)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(to_cluster(local, cta)),
                 "r"(__float_as_uint(v)), "r"(to_cluster(bar, cta))
                 : "memory");
}

// Compiled for at least 512 threads per SM (at most 128 registers a thread,
// no spills at any n).
template <int NR, int DT, int CL, int TH>
__global__ void __launch_bounds__(TH, 512 / TH)
allreduce_rmsnorm_kernel(const __grid_constant__ CPtrs<NR> in, const void* __restrict__ residual,
                         const void* __restrict__ weight, float eps, const __grid_constant__ MPtrs<NR> out,
                         void* residual_out, size_t hidden, size_t slice_vecs, int early_release, DevStatus* st)
{
    constexpr int VE = kVecElems<DT>;
    constexpr int W = TH / 32;
    constexpr int NP = CL * W;                    // partial sums a CTA receives: every warp of the cluster's
    extern __shared__ float r_more[];             // r of the vectors after each thread's first
    __shared__ float parts[NP];                   // warp w of CTA k sends into parts[k * W + w]
    __shared__ __align__(8) uint64_t parts_bar;   // completes when the NP partials have landed
    if (threadIdx.x == 0) {
        // one arrival (this one, expecting the partials' bytes), then the bytes
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&parts_bar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(4u * NP) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the first half of a cluster barrier: its wait, before the partial sums
    // are sent, makes sure every CTA of the cluster has started and has set up
    // its barrier
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    pdl_acquire();
    if (early_release) pdl_release();
    const uint32_t c = cluster_ctarank();
    const size_t t = blockIdx.x / CL;                  // token row of this cluster
    const size_t nvec_row = hidden / VE;
    const size_t v_lo = (size_t)c * slice_vecs;
    const size_t v_hi = v_lo + slice_vecs < nvec_row ? v_lo + slice_vecs : nvec_row;
    const size_t row = t * nvec_row;                   // first 16-byte vector of the row
    const size_t v_first = v_lo + threadIdx.x;

    // pass 1: all-reduce, residual add, squares.  Every load of a vector --
    // the n ranks', the residual's and (for pass 2) the weight's -- is issued
    // before any is used, so the pass waits on memory once.
    float ss = 0.0f;
    uint4 w_first = make_uint4(0u, 0u, 0u, 0u);   // the weight of this thread's first vector
    float r_first[VE];                             // r of this thread's first vector
    for (size_t v = v_first; v < v_hi; v += TH) {
        uint4 x[NR];
#pragma unroll
        for (int q = 0; q < NR; ++q) x[q] = ld16(static_cast<const uint4*>(in.p[q]) + row + v);
        const uint4 res = ld16(static_cast<const uint4*>(residual) + row + v);
        if (v == v_first) w_first = ld16(static_cast<const uint4*>(weight) + v);
        const uint4 a = reduce_rank_order<DT, NR>(x);
        float af[VE], rf[VE];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            Payload<DT>::widen(word(a, j), af + j * Payload<DT>::kPerWord);
            Payload<DT>::widen(word(res, j), rf + j * Payload<DT>::kPerWord);
        }
#pragma unroll
        for (int k = 0; k < VE; ++k) rf[k] = af[k] + rf[k];
        const uint4 rr = round_vec<DT>(rf);
        st16(static_cast<uint4*>(residual_out) + row + v, rr);
        float rq[VE];
#pragma unroll
        for (int j = 0; j < 4; ++j) Payload<DT>::widen(word(rr, j), rq + j * Payload<DT>::kPerWord);
        if (v == v_first) {
#pragma unroll
            for (int k = 0; k < VE; ++k) r_first[k] = rq[k];
        } else {
            float* dst = r_more + (v - v_lo - TH) * VE;
#pragma unroll
            for (int k = 0; k < VE; ++k) dst[k] = rq[k];
        }
#pragma unroll
        for (int k = 0; k < VE; ++k) ss = ss + rq[k] * rq[k];
    }
    // the warp's sum of squares (lane 0's, in every lane), sent by lane k into CTA k
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = ss + __shfl_down_sync(0xffffffffu, ss, o);
    ss = __shfl_sync(0xffffffffu, ss, 0);
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (lane < CL) st_async_cluster_f32(&parts[c * W + w], &parts_bar, lane, ss);
    {
        // every thread waits (bounded) until all NP partials have landed here; a
        // CTA leaves only after that, so nothing is still landing in its shared
        // memory when it exits
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&parts_bar);
        uint32_t done = 0;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 0; it < (1u << 22) && !done; ++it) {
            asm volatile("{\n\t.reg .pred p;\n\t"
                         "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], 0;\n\t"
                         "selp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(done)
                         : "r"(bar)
                         : "memory");
            if (!done && (it & 255) == 255 && globaltimer_ns() - t0 > 100000000ull) break;   // 0.1 s
        }
        if (!done) report_wait_timeout(st);
    }
    // the row's sum, in the same order in every warp: lane j adds parts j, j + 32,
    // ..., then the lanes pairwise down to lane 0
    float t2 = 0.0f;
#pragma unroll
    for (int k = 0; k < NP; k += 32)
        if (k + (int)lane < NP) t2 = t2 + parts[k + lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t2 = t2 + __shfl_down_sync(0xffffffffu, t2, o);
    t2 = __shfl_sync(0xffffffffu, t2, 0);
    const float inv = 1.0f / sqrtf(t2 / (float)hidden + eps);
    if (!early_release) pdl_release();

    // pass 2: scale, weight, round, write every rank's output
    for (size_t v = v_first; v < v_hi; v += TH) {
        const uint4 wv = v == v_first ? w_first : ld16(static_cast<const uint4*>(weight) + v);
        float wf[VE], y[VE];
#pragma unroll
        for (int j = 0; j < 4; ++j) Payload<DT>::widen(word(wv, j), wf + j * Payload<DT>::kPerWord);
        const float* src = v == v_first ? r_first : r_more + (v - v_lo - TH) * VE;
#pragma unroll
        for (int k = 0; k < VE; ++k) y[k] = (src[k] * inv) * wf[k];
        const uint4 yo = round_vec<DT>(y);
#pragma unroll
        for (int q = 0; q < NR; ++q) st16(static_cast<uint4*>(out.p[q]) + row + v, yo);
    }
}

}  // namespace

// Largest slice of a row one CTA keeps in shared memory (fp32).
constexpr size_t kRmsnormMaxSliceBytes = 160u << 10;

size_t rmsnorm_slice_vecs(size_t hidden, int dt)
{
    const size_t ve = 16u / elem_bytes(dt);
    const size_t nvec = hidden / ve;
    return (nvec + kClusterCtas - 1) / kClusterCtas;
}

bool rmsnorm_fits(size_t hidden, int dt)
{
    const size_t ve = 16u / elem_bytes(dt);
    return rmsnorm_slice_vecs(hidden, dt) * ve * sizeof(float) <= kRmsnormMaxSliceBytes;
}

int launch_allreduce_rmsnorm(Handle& h, const void* const* in, const void* residual, const void* weight, float eps,
                             void* const* out, void* residual_out, size_t tokens, size_t hidden, int dt,
                             cudaStream_t s)
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
            const uint64_t S = (uint64_t)tokens * hidden * sizeof(typename Payload<DT>::scalar_t);
            const uint64_t W = (uint64_t)hidden * sizeof(typename Payload<DT>::scalar_t);
            auto run = [&](auto clc, auto thc) -> int {
                constexpr int CL = decltype(clc)::value;
                constexpr int TH = decltype(thc)::value;
                const size_t slice = (hidden / kVecElems<DT> + CL - 1) / CL;
                const size_t smem = slice > (size_t)TH ? (slice - TH) * kVecElems<DT> * sizeof(float) : 0;
                static std::atomic<uint32_t> attr_done{0};
                const bool attr_ok = once_per_device(attr_done, [&] {
                    return cudaFuncSetAttribute(allreduce_rmsnorm_kernel<NR, DT, CL, TH>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)kRmsnormMaxSliceBytes) == cudaSuccess &&
                           (CL <= 8 || cudaFuncSetAttribute(allreduce_rmsnorm_kernel<NR, DT, CL, TH>,
                                                            cudaFuncAttributeNonPortableClusterSizeAllowed,
                                                            1) == cudaSuccess);
                });
                if (!attr_ok) return AR_ERR_CUDA;
                cudaLaunchAttribute attr[2];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = CL;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                attr[1].val.programmaticStreamSerializationAllowed = h.pdl ? 1 : 0;
                cudaLaunchConfig_t cfg{};
                cfg.gridDim = dim3((unsigned)(tokens * CL));
                cfg.blockDim = dim3(TH);
                cfg.dynamicSmemBytes = smem;
                cfg.stream = s;
                cfg.attrs = attr;
                cfg.numAttrs = 2;
                // A grid of at most one CTA per SM lets the next launch in at once,
                // leaving every SM room for its CTAs: 2.16 against 2.25 us per call
                // at 1 x 4096 (n = 8 bf16, graph replay on GB300), no change at
                // 8 x 8192; at 64 x 8192 (1024 CTAs) the early CTAs cost 0.9 us.
                const int early = tokens * CL <= (size_t)h.sm_count ? 1 : 0;
                rec_begin(h, s);
                const cudaError_t e = cudaLaunchKernelEx(&cfg, allreduce_rmsnorm_kernel<NR, DT, CL, TH>, ip, residual,
                                                         weight, eps, op, residual_out, hidden, slice, early, h.status);
                rec_end(h, s, AR_K_ALLREDUCE_RMSNORM, 2ull * (NR + 1) * S + W);
                return e == cudaSuccess ? launch_status() : AR_ERR_CUDA;
            };
            using C8 = std::integral_constant<int, 8>;
            using C16 = std::integral_constant<int, 16>;
            using T64 = std::integral_constant<int, 64>;
            using T128 = std::integral_constant<int, 128>;
            using T256 = std::integral_constant<int, 256>;
            // Clusters of 16 (each row over twice the SMs) unless the row gives a
            // CTA fewer than 64 vectors and the rows fill more than a wave of
            // four CTAs per SM: then 8.  Threads: the slice rounded up to 64,
            // 128 or 256.  Measured on GB300 (n = 8 bf16, graph replay, every
            // (CL, threads) pair of {2, 4, 8, 16} x {32 ... 512}): the best or
            // within 0.01 us of it at 1 x 4096 to 64 x 8192; one vector a thread
            // beats a loop of two by 0.3-2 us, CTAs of 32 threads lose 0.1 us.
            const size_t nvec = hidden / kVecElems<DT>;
            if (nvec / 16 < 64 && tokens * 16 > 4 * (size_t)h.sm_count) {
                const size_t slice = (nvec + 7) / 8;
                return slice <= 64 ? run(C8{}, T64{}) : run(C8{}, T128{});
            }
            const size_t slice = (nvec + 15) / 16;
            return slice <= 64 ? run(C16{}, T64{}) : slice <= 128 ? run(C16{}, T128{}) : run(C16{}, T256{});
        });
    });
}

}  // namespace argb
