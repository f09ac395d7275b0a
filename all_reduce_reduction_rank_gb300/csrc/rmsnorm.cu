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
// Layout: one thread-block cluster of CL CTAs per token row (8; 16, a
// non-portable cluster size, while the CTAs of 16-CTA clusters fit in one
// wave); CTA c of the cluster owns a contiguous slice of the row.  Pass
// 1 reads the n rank slices once, writes r, keeps r (fp32: a thread's first
// vector in registers, any further ones in shared memory) and accumulates its
// squares; each CTA sends its partial sum into every
// CTA's shared memory (distributed shared memory) with an asynchronous store
// counted on the receiver's mbarrier, so each CTA waits only until the CL
// partials have landed in its own shared memory (no second cluster barrier),
// and adds them in the same fixed order; pass 2 scales r and writes every
// rank's output.
// HBM: reads n S + S (+ the weight, H per launch), writes n S + S.
#include "common.cuh"

namespace argb {
namespace {

constexpr int kClusterCtas = 8;   // the cluster size that sizes the shared-memory slice
constexpr int kNormThreads = 128;

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

// Compiled for at least four CTAs per SM (79 registers at n = 8, no spills at
// any n); a bound of four measured 1-3% less time per call at 1-64 tokens
// than the compiler's own choice (graph-replay A/B on GB300, n = 8 bf16).
template <int NR, int DT, int CL>
__global__ void __launch_bounds__(kNormThreads, 4)
allreduce_rmsnorm_kernel(const __grid_constant__ CPtrs<NR> in, const void* __restrict__ residual,
                         const void* __restrict__ weight, float eps, const __grid_constant__ MPtrs<NR> out,
                         void* residual_out, size_t hidden, size_t slice_vecs, DevStatus* st)
{
    constexpr int VE = kVecElems<DT>;
    extern __shared__ float r_slice[];                 // slice_vecs * VE floats
    __shared__ float warp_part[kNormThreads / 32];
    __shared__ float parts[CL];   // every CTA's sum of squares, sent by that CTA
    __shared__ __align__(8) uint64_t parts_bar;   // completes when the CL partials have landed
    __shared__ float row_inv;
    if (threadIdx.x == 0) {
        // one arrival (this one, expecting the CL partials' bytes), then the bytes
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&parts_bar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(4u * CL) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the first half of a cluster barrier: its wait, before the partial sums
    // are sent, makes sure every CTA of the cluster has started and has set up
    // its barrier
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    pdl_acquire();
    const uint32_t c = cluster_ctarank();
    const size_t t = blockIdx.x / CL;                  // token row of this cluster
    const size_t nvec_row = hidden / VE;
    const size_t v_lo = (size_t)c * slice_vecs;
    const size_t v_hi = v_lo + slice_vecs < nvec_row ? v_lo + slice_vecs : nvec_row;
    const size_t row = t * nvec_row;                   // first 16-byte vector of the row

    // pass 1: all-reduce, residual add, squares.  Every load of a vector --
    // the n ranks', the residual's and (for pass 2) the weight's -- is issued
    // before any is used, so the pass waits on memory once.
    float ss = 0.0f;
    uint4 w_first = make_uint4(0u, 0u, 0u, 0u);   // the weight of this thread's first vector
    float r_first[VE];                             // r of this thread's first vector (the rest in shared memory)
    for (size_t v = v_lo + threadIdx.x; v < v_hi; v += kNormThreads) {
        uint4 x[NR];
#pragma unroll
        for (int q = 0; q < NR; ++q) x[q] = ld16(static_cast<const uint4*>(in.p[q]) + row + v);
        const uint4 res = ld16(static_cast<const uint4*>(residual) + row + v);
        if (v == v_lo + threadIdx.x) w_first = ld16(static_cast<const uint4*>(weight) + v);
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
        if (v == v_lo + threadIdx.x) {
#pragma unroll
            for (int k = 0; k < VE; ++k) r_first[k] = rq[k];
        } else {
            float* dst = r_slice + (v - v_lo) * VE;
#pragma unroll
            for (int k = 0; k < VE; ++k) dst[k] = rq[k];
        }
#pragma unroll
        for (int k = 0; k < VE; ++k) ss = ss + rq[k] * rq[k];
    }
    // the CTA's sum of squares: warps, then the warps in order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = ss + __shfl_down_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = ss;
    __syncthreads();
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (threadIdx.x < CL) {   // this CTA's partial, sent into CTA k of the cluster by thread k
        float s = 0.0f;
        for (int w = 0; w < kNormThreads / 32; ++w) s = s + warp_part[w];
        st_async_cluster_f32(&parts[c], &parts_bar, threadIdx.x, s);
    }
    if (threadIdx.x == 0) {
        // wait (bounded) until all CL partials have landed here; a CTA leaves only
        // after that, so nothing is still landing in its shared memory when it exits
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
        // the row's: the cluster's CTAs in order
        float t2 = 0.0f;
        for (uint32_t k = 0; k < CL; ++k) t2 = t2 + parts[k];
        row_inv = 1.0f / sqrtf(t2 / (float)hidden + eps);
    }
    __syncthreads();
    pdl_release();
    const float inv = row_inv;

    // pass 2: scale, weight, round, write every rank's output
    for (size_t v = v_lo + threadIdx.x; v < v_hi; v += kNormThreads) {
        const uint4 wv = v == v_lo + threadIdx.x ? w_first : ld16(static_cast<const uint4*>(weight) + v);
        float wf[VE], y[VE];
#pragma unroll
        for (int j = 0; j < 4; ++j) Payload<DT>::widen(word(wv, j), wf + j * Payload<DT>::kPerWord);
        const float* src = v == v_lo + threadIdx.x ? r_first : r_slice + (v - v_lo) * VE;
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
            auto run = [&](auto clc) -> int {
                constexpr int CL = decltype(clc)::value;
                const size_t slice = (hidden / kVecElems<DT> + CL - 1) / CL;
                const size_t smem = slice * kVecElems<DT> * sizeof(float);
                static std::atomic<uint32_t> attr_done{0};
                const bool attr_ok = once_per_device(attr_done, [&] {
                    return cudaFuncSetAttribute(allreduce_rmsnorm_kernel<NR, DT, CL>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)kRmsnormMaxSliceBytes) == cudaSuccess &&
                           (CL <= 8 || cudaFuncSetAttribute(allreduce_rmsnorm_kernel<NR, DT, CL>,
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
                cfg.blockDim = dim3(kNormThreads);
                cfg.dynamicSmemBytes = smem;
                cfg.stream = s;
                cfg.attrs = attr;
                cfg.numAttrs = 2;
                rec_begin(h, s);
                const cudaError_t e = cudaLaunchKernelEx(&cfg, allreduce_rmsnorm_kernel<NR, DT, CL>, ip, residual,
                                                         weight, eps, op, residual_out, hidden, slice, h.status);
                rec_end(h, s, AR_K_ALLREDUCE_RMSNORM, 2ull * (NR + 1) * S + W);
                return e == cudaSuccess ? launch_status() : AR_ERR_CUDA;
            };
            // up to one wave of CTAs (four per SM), clusters of 16 spread each row over
            // twice the SMs: measured on GB300 (n = 8 bf16, graph replay), 3.92 against
            // 4.13 us at 32 x 8192; at 64 rows, where 16 would need more than a wave,
            // clusters of 8 (5.3 us) beat 16, 4 and 2 (7.2, 6.7, 6.3 us)
            if (tokens * 16 <= 4 * (size_t)h.sm_count) return run(std::integral_constant<int, 16>{});
            return run(std::integral_constant<int, kClusterCtas>{});
        });
    });
}

}  // namespace argb
