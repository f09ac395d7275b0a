// Persistent ring all-reduce over a thread-block cluster: the ranks are the
// CTAs of one cluster and a hop goes through distributed shared memory.
//
// The same protocol and sums as ring_persistent.cu (handbook "集合通信：NCCL
// 的算法、协议与推理框架的定制 all-reduce", §协议: LL128 lines of 120 bytes of
// data and an 8-byte flag, the receiver polling the flag; "多 GPU 与 NCCL",
// §ring all-reduce: the steps and chunk rotation; fp32 partials, chunk c
// summed from rank c, rounded once), so the result equals ar_ring's bit for
// bit.  What differs is where the receiving inbox lives: in the receiving
// CTA's shared memory, written by the sending CTA of the same cluster with
// st.shared::cluster.  On this GPU a flag round trip through distributed
// shared memory takes ~0.53 us against ~1.7 us through global memory, and
// the lines never touch L2 or HBM: HBM sees only the ranks' own elements and
// outputs, 2 n S per call, as one-shot does.
//
// Layout: cluster size n (one CTA per rank, cluster_ctarank = rank);
// cluster k owns slice [k E, (k+1) E) of every chunk (E a multiple of 960
// elements = 32 lines); clusters are independent, so the grid may run in any
// number of waves and needs no cooperative launch.  Warp w of rank r handles
// batches b = w, w+8, ... of the slice and exchanges lines only with warp w
// of ranks r-1 and r+1.
//
// Shared memory of a CTA: per warp kSlots inbox slots of 32 lines (one batch
// each), the per-warp count of batches its receiver has consumed, and an
// abort word.  The sender writes batch q into slot q % kSlots once the
// receiver has consumed batch q - kSlots; a line's flag is q + 1.  A warp
// walks its (step, batch) pairs in one software-pipelined loop: it issues
// the loads of the next pair's own elements before it sends the current
// one, and publishes a consumed slot after its own send (one fence serves
// both), which needs a step's batches to fit in kSlots - 1 slots.  Shared
// memory is zeroed at the start, behind a cluster barrier, so no flag of an
// earlier launch survives; a cluster barrier at the end keeps every CTA
// alive until no peer can still write into it.
//
// Ordering: data stores to the peer, __syncwarp, fence.acq_rel.cluster, flag
// stores; the receiver polls its flags with ld.acquire.cluster, __syncwarp,
// then reads the lines; the consumed count is a relaxed store after the
// same fence.  Every wait is bounded by spin_ns and a poll count; a
// wait that runs out records AR_ERR_FLAG_TIMEOUT (a line) or
// AR_ERR_WAIT_TIMEOUT (a slot) and raises the abort word of every CTA of the
// cluster, on which the other waits give up; all threads still reach the
// final cluster barrier.
#include "lines.cuh"

namespace argb {
namespace {

using namespace lines;

constexpr int kCWarps = kThreads / 32;
constexpr int kSlots = 3;                                                 // inbox slots per warp
constexpr unsigned kCFull = 0xffffffffu;
constexpr size_t kInboxBytes = (size_t)kCWarps * kSlots * kBatchLines * 128;
// inbox, then consumed[kCWarps] and the abort word, rounded to 16 bytes
constexpr size_t kClusterSmem = kInboxBytes + ((kCWarps + 1) * sizeof(uint64_t) + 15) / 16 * 16;

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t cta)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(cta));
    return a;
}

__device__ __forceinline__ void cluster_barrier()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint64_t ld_acq_local(uint32_t a)
{
    uint64_t v;
    asm volatile("ld.acquire.cluster.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_rlx_local(uint32_t a)
{
    uint64_t v;
    asm volatile("ld.relaxed.cluster.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld16_local(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st16_peer(uint32_t a, const uint4& v)
{
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st8_peer(uint32_t a, uint32_t x, uint32_t y)
{
    asm volatile("st.shared::cluster.v2.u32 [%0], {%1,%2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}

__device__ __forceinline__ void st_rlx_peer(uint32_t a, uint64_t v)
{
    asm volatile("st.relaxed.cluster.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}

__device__ __forceinline__ void fence_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

struct ClusterSmem {
    uint32_t inbox;      // shared address of this CTA's inbox
    uint32_t consumed;   // shared address of consumed[0]
    uint32_t abort;      // shared address of the abort word
};

// Raise the abort word of every CTA of the cluster.
template <int NR>
__device__ void raise_abort(const ClusterSmem& S)
{
#pragma unroll
    for (int q = 0; q < NR; ++q) st_rlx_peer(peer_addr(S.abort, (uint32_t)q), 1ull);
}

template <int NR, int DT>
__global__ void __launch_bounds__(kThreads, 2)
ring_cluster_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t C,
                    size_t count, size_t epc, int64_t spin_ns, int absent, DevStatus* st)
{
    using T = typename Payload<DT>::scalar_t;
    constexpr int kI = kBatchLines / 4;
    extern __shared__ __align__(128) unsigned char smem[];
    uint32_t crank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
    const int r = (int)crank;
    const size_t k = blockIdx.x / NR;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 3, j = lane & 7;
    const int nw = j < 7 ? 4 : 2;
    const int d = (r + 1) % NR, p = (r + NR - 1) % NR;   // next and previous rank
    ClusterSmem S;
    S.inbox = smem_addr(smem);
    S.consumed = S.inbox + (uint32_t)kInboxBytes;
    S.abort = S.consumed + kCWarps * 8;

    // zero the inbox flags, consumed counts and abort word, then let every
    // CTA of the cluster see that before any peer writes
    for (uint32_t o = threadIdx.x * 16; o < (uint32_t)kClusterSmem; o += kThreads * 16)
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(S.inbox + o), "r"(0u) : "memory");
    cluster_barrier();

    const size_t slice_lo = k * epc;
    const size_t line_lo = slice_lo / kLineWords;
    const uint32_t my_box = S.inbox + (uint32_t)(warp * kSlots * kBatchLines * 128);
    const uint32_t peer_box = peer_addr(my_box, (uint32_t)d);                    // the next rank's inbox for this warp
    const uint32_t my_consumed = S.consumed + 8 * warp;                            // written by the next rank
    const uint32_t prev_consumed = peer_addr(S.consumed + 8 * warp, (uint32_t)p);  // the previous rank's copy
    uint64_t q_recv = 0, q_send = 0;
    bool dead = (r == absent);   // a rank that never joins (failure emulation)

    // the warp's (step, batch) pairs in order: step t moves chunk c(t); the
    // warp's batches of it are b = warp, warp + 8, ... below nbatch(t)
    struct Geom {
        size_t len, slice_hi, nbatch;
        const T* x;
        T* y;
    };
    auto geom = [&](int t) -> Geom {
        const int c = t <= NR - 2 ? ((r - t) % NR + NR) % NR : ((r + NR - t) % NR + NR) % NR;
        const size_t lo = (size_t)c * C;
        Geom G;
        G.len = lo >= count ? 0 : (count - lo < C ? count - lo : C);
        G.slice_hi = slice_lo + epc < G.len ? slice_lo + epc : G.len;
        const size_t nlines = G.slice_hi > slice_lo ? (G.slice_hi - slice_lo + kLineWords - 1) / kLineWords : 0;
        G.nbatch = (nlines + kBatchLines - 1) / kBatchLines;
        G.x = static_cast<const T*>(in.p[r]) + lo;
        G.y = static_cast<T*>(out.p[r]) + lo;
        return G;
    };
    constexpr int kLast = 2 * NR - 2;   // t = 2n-2: only the last receive
    auto next_pair = [&](int& t, size_t& b, Geom& G) {   // the warp's next (step, batch), or t > kLast
        b += kCWarps;
        while (t <= kLast && b >= G.nbatch) {
            ++t;
            b = (size_t)warp;
            if (t <= kLast) G = geom(t);
        }
    };
    // the rank's own elements of a batch: issued early, used later
    uint32_t xr[kI][kRawWords<DT>];
    auto load_x = [&](int t, size_t b, const Geom& G) {
        if (t > NR - 1) return;
        const size_t base = line_lo + b * kBatchLines;
#pragma unroll
        for (int i = 0; i < kI; ++i) {
            const size_t l = base + 4 * i + g;
            load_raw<DT>(G.x, l * kLineWords + 4 * (size_t)j, nw, l * kLineWords < G.slice_hi ? G.len : 0, xr[i]);
        }
    };

    int t = 0;
    size_t b = (size_t)warp;
    Geom G = geom(0);
    if (b >= G.nbatch) {   // the warp's first pair
        b -= kCWarps;
        next_pair(t, b, G);
    }
    if (!dead && t <= kLast) load_x(t, b, G);
    while (!dead && t <= kLast) {
        const bool sends = t <= kLast - 1;
        const size_t base = line_lo + b * kBatchLines;
        uint4 w[kI];
#pragma unroll
        for (int i = 0; i < kI; ++i) w[i] = make_uint4(0u, 0u, 0u, 0u);
        if (t >= 1) {   // receive: wait for the 32 flags of this batch's slot
            const uint32_t slot = my_box + (uint32_t)((q_recv % kSlots) * kBatchLines * 128);
            const bool live = (base + lane) * kLineWords < G.slice_hi;
            const uint32_t flag = slot + lane * 128 + 120;
            bool ok = !live || ld_acq_local(flag) == q_recv + 1;
            if (!__all_sync(kCFull, ok)) {
                const uint64_t t0 = globaltimer_ns(), cap = (uint64_t)spin_ns / 16u + 4096u;
                bool stop = false;
                for (uint64_t it = 0; it < cap && !stop; ++it) {
                    if (it >= 1024) __nanosleep(32);
                    if (!ok) ok = ld_acq_local(flag) == q_recv + 1;
                    if (__all_sync(kCFull, ok)) break;
                    if ((it & 31) == 31)
                        stop = __any_sync(kCFull, (int64_t)(globaltimer_ns() - t0) > spin_ns ||
                                                      ld_rlx_local(S.abort) != 0);
                }
                if (!__all_sync(kCFull, ok)) {
                    if (ld_rlx_local(S.abort) == 0) {
                        if (!ok) report_flag_timeout(st, r, base + lane);
                        if (lane == 0) raise_abort<NR>(S);
                    }
                    dead = true;
                    break;
                }
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < kI; ++i) {
                const size_t l = base + 4 * i + g;
                if (l * kLineWords < G.slice_hi) w[i] = ld16_local(slot + (uint32_t)((4 * i + g) * 128 + 16 * j));
            }
        }
        float v[kI][4];
#pragma unroll
        for (int i = 0; i < kI; ++i) {
            v[i][0] = __uint_as_float(w[i].x);
            v[i][1] = __uint_as_float(w[i].y);
            v[i][2] = __uint_as_float(w[i].z);
            v[i][3] = __uint_as_float(w[i].w);
            if (t <= NR - 1) {
                float xv[4];
                widen_raw<DT>(xr[i], xv);
#pragma unroll
                for (int u = 0; u < 4; ++u) v[i][u] = t == 0 ? xv[u] : v[i][u] + xv[u];
            }
            if (t == NR - 1) {   // rounded once; the rounded value is passed on
#pragma unroll
                for (int u = 0; u < 4; ++u) v[i][u] = Payload<DT>::widen1(Payload<DT>::narrow1(v[i][u]));
            }
        }
        // the next pair's own elements now: their loads fly during the send
        int t2 = t;
        size_t b2 = b;
        Geom G2 = G;
        next_pair(t2, b2, G2);
        if (t2 <= kLast) load_x(t2, b2, G2);
        if (sends) {
            // the next rank must have consumed the batch that last used this slot
            if (q_send >= kSlots) {
                const uint64_t want = q_send - kSlots + 1;
                bool ok = ld_acq_local(my_consumed) >= want;
                if (!__all_sync(kCFull, ok)) {
                    const uint64_t t0 = globaltimer_ns(), cap = (uint64_t)spin_ns / 16u + 4096u;
                    bool stop = false;
                    for (uint64_t it = 0; it < cap && !stop; ++it) {
                        if (it >= 1024) __nanosleep(32);
                        ok = ld_acq_local(my_consumed) >= want;
                        if (__all_sync(kCFull, ok)) break;
                        if ((it & 31) == 31)
                            stop = __any_sync(kCFull, (int64_t)(globaltimer_ns() - t0) > spin_ns ||
                                                          ld_rlx_local(S.abort) != 0);
                    }
                    if (!__all_sync(kCFull, ok)) {
                        if (lane == 0 && ld_rlx_local(S.abort) == 0) {
                            report_wait_timeout(st);
                            raise_abort<NR>(S);
                        }
                        dead = true;
                        break;
                    }
                }
            }
            const uint32_t slot = peer_box + (uint32_t)((q_send % kSlots) * kBatchLines * 128);
#pragma unroll
            for (int i = 0; i < kI; ++i) {
                const size_t l = base + 4 * i + g;
                if (l * kLineWords >= G.slice_hi) continue;
                const uint32_t a = slot + (uint32_t)((4 * i + g) * 128 + 16 * j);
                if (j < 7)
                    st16_peer(a, make_uint4(__float_as_uint(v[i][0]), __float_as_uint(v[i][1]),
                                            __float_as_uint(v[i][2]), __float_as_uint(v[i][3])));
                else
                    st8_peer(a, __float_as_uint(v[i][0]), __float_as_uint(v[i][1]));
            }
            __syncwarp();
            fence_cluster();   // releases these lines; also orders this batch's inbox reads
            if ((base + lane) * kLineWords < G.slice_hi) st_rlx_peer(slot + lane * 128 + 120, q_send + 1);
            ++q_send;
            // this batch's inbox slot is free again (its reads precede the
            // fence): tell the previous rank.  Published after this rank's
            // own send, so a step's batches must fit in kSlots - 1 slots.
            if (t >= 1 && lane == 0) st_rlx_peer(prev_consumed, q_recv + 1);
        }
        if (t >= 1) ++q_recv;
        // this rank's output last, after the hop is on its way
        if (t >= NR - 1) {
#pragma unroll
            for (int i = 0; i < kI; ++i) {
                const size_t l = base + 4 * i + g;
                if (l * kLineWords < G.slice_hi) store_elems<DT>(G.y, l * kLineWords + 4 * (size_t)j, nw, G.len, v[i]);
            }
        }
        if (!dead && ld_rlx_local(S.abort) != 0) dead = true;
        dead = __any_sync(kCFull, dead);
        t = t2;
        b = b2;
        G = G2;
    }
    // no CTA leaves while a peer may still write into its shared memory
    cluster_barrier();
}

}  // namespace

int launch_ring_cluster(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
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
            static std::atomic<uint32_t> attr_done{0};
            const bool attr_ok = once_per_device(attr_done, [&] {
                return cudaFuncSetAttribute(ring_cluster_kernel<NR, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)kClusterSmem) == cudaSuccess &&
                       (NR <= 8 || cudaFuncSetAttribute(ring_cluster_kernel<NR, DT>,
                                                        cudaFuncAttributeNonPortableClusterSizeAllowed,
                                                        1) == cudaSuccess);
            });
            if (!attr_ok) return AR_ERR_CUDA;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = NR;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cudaLaunchConfig_t cfg{};
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = kClusterSmem;
            cfg.stream = s;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            // clusters that fit at once: one wave of them (computed once,
            // thread-safely, per kernel instantiation)
            static const int resident = [&] {
                cudaLaunchConfig_t q = cfg;
                q.gridDim = dim3((unsigned)(NR * 64));
                int nc = 0;
                if (cudaOccupancyMaxActiveClusters(&nc, ring_cluster_kernel<NR, DT>, &q) != cudaSuccess) nc = 0;
                cudaGetLastError();
                return nc;
            }();
            if (resident < 1) return AR_ERR_CUDA;
            const size_t C = chunk_elems(NR, count, DT);
            // slices of at least one batch per warp; one wave of clusters
            // unless that would give a warp more than kSlots - 1 batches per
            // step: at step 0 every rank sends without receiving, and a
            // receiver frees a slot only after its own send of the next
            // batch, so a step's batches must fit in kSlots - 1 slots
            // (otherwise every rank waits on its successor: a cycle)
            const size_t per_cta_min = kBatchElems * kCWarps;
            size_t K = (C + per_cta_min - 1) / per_cta_min;
            if (K > (size_t)resident) K = (size_t)resident;
            if (K < 1) K = 1;
            size_t epc = (C + K - 1) / K;
            epc = (epc + kBatchElems - 1) / kBatchElems * kBatchElems;
            if (epc > kBatchElems * kCWarps * (kSlots - 1)) epc = kBatchElems * kCWarps * (kSlots - 1);
            K = (C + epc - 1) / epc;
            if (K < 1) K = 1;
            cfg.gridDim = dim3((unsigned)(K * NR));
            const uint64_t S = (uint64_t)count * sizeof(typename Payload<DT>::scalar_t);
            rec_begin(h, s);
            const cudaError_t err = cudaLaunchKernelEx(&cfg, ring_cluster_kernel<NR, DT>, ip, op, C, count, epc,
                                                       h.spin_ns, h.persist_absent, h.status);
            rec_end(h, s, AR_K_RING_CLUSTER, 2ull * NR * S);
            *launches = 1;
            if (err != cudaSuccess) {
                cudaGetLastError();
                return AR_ERR_CUDA;
            }
            return launch_status();
        });
    });
}

}  // namespace argb
