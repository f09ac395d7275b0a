// Persistent ring all-reduce over a thread-block cluster: the ranks are the
// CTAs of one cluster and a hop goes through distributed shared memory.
//
// The same steps and sums as ar_ring (handbook "多 GPU 与 NCCL", §ring
// all-reduce: n-1 reduce-scatter steps then n-1 all-gather steps, chunk c
// summed from rank c; fp32 partials, rounded once), so the result equals
// ar_ring's bit for bit, in one launch.  A hop is a batch of 128-byte lines
// of fp32 words that the sending CTA writes straight into the receiving
// CTA's shared memory with asynchronous stores (st.async), each of which
// counts its bytes on the receiving slot's mbarrier (complete_tx).  The
// receiver waits on that one barrier; the sender neither waits for its
// stores nor fences them.  This is the handbook's Simple protocol shape
// ("集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce", §协议: data, plus
// a separate completion signal) rather than LL128's flag in every line:
// inside a cluster the barrier's byte count gives what the per-line flag
// gives over NVLink -- the data and its arrival in one operation -- without
// spending 8 bytes of every line on it.  For 16-bit payloads the all-gather
// hops carry the completed (already rounded) values in the payload type,
// half the bytes of fp32 lines.  HBM sees only the ranks' own elements and
// outputs: 2 n S per call.
//
// Layout: cluster size n (one CTA per rank, cluster_ctarank = rank);
// cluster k owns slice [k E, (k+1) E) of every chunk (E a multiple of one
// batch, 32 L elements); clusters are independent, so the grid may run in any
// number of waves and needs no cooperative launch.  Warp w of rank r handles
// batches b = w, w+8, ... of the slice and exchanges lines only with warp w
// of ranks r-1 and r+1.
//
// Shared memory of a CTA: per warp kSlots inbox slots of L lines; per slot a
// "full" mbarrier (the receiver's: one arrival, the sender's expect_tx, plus
// the slot's bytes) and an "empty" mbarrier (the sender's: one arrival by the
// receiver once it has read the slot); an abort word.  Batch q of a warp goes
// to slot q % kSlots; its use u = q / kSlots completes phase u of both
// barriers.  The receiver frees a slot as soon as it has read it, before its
// own send, so a step's batches may fill all kSlots slots: a warp's batches
// per step are capped at kSlots, or at step 0 (every rank sending, none
// receiving yet) every rank would wait on its successor.
//
// Every wait is bounded by spin_ns and a poll count.  A wait that runs out
// records AR_ERR_FLAG_TIMEOUT (a batch that never came) or
// AR_ERR_WAIT_TIMEOUT (a slot never freed) and raises the abort word of
// every CTA of the cluster, on which the other waits give up.  Before any CTA
// exits, a cluster barrier stops all sending; after an abort each CTA then
// waits (bounded) for the bytes of any batch already announced into its
// inbox, since an asynchronous store may still be landing; a second cluster
// barrier ends the kernel.
#include "lines.cuh"

namespace argb {
namespace {

using namespace lines;

constexpr int kCWarps = kThreads / 32;
constexpr int kCWords = 32;   // fp32 words per 128-byte line: 4 per lane, 8 lanes per line

// Four consecutive elements from e as raw words (zero past len).
template <int DT>
__device__ __forceinline__ void load4(const void* chunk, size_t e, size_t len, uint32_t* w)
{
    if (e + 4 <= len) {
        if constexpr (DT == AR_F32) {
            const uint4 v = ld16(static_cast<const float*>(chunk) + e);
            w[0] = v.x;
            w[1] = v.y;
            w[2] = v.z;
            w[3] = v.w;
        } else {
            const uint2 v = ld8_plain(static_cast<const uint16_t*>(chunk) + e);
            w[0] = v.x;
            w[1] = v.y;
        }
    } else {
        load_raw<DT>(chunk, e, 4, len, w);
    }
}

// Stores eight 16-bit elements (raw bits, one 16-byte vector) from e, those below len.
template <int DT>
__device__ __forceinline__ void store8_raw(void* chunk, size_t e, size_t len, const uint4& v)
{
    uint16_t* y = static_cast<uint16_t*>(chunk);
    if (e + 8 <= len) {
        st16(y + e, v);
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (e + u < len) y[e + u] = (uint16_t)(w[u >> 1] >> (16 * (u & 1)));
    }
}

// Rounds f[0..4) to the payload type and stores the elements below len.
template <int DT>
__device__ __forceinline__ void store4(void* chunk, size_t e, size_t len, const float* f)
{
    if (e + 4 <= len) {
        if constexpr (DT == AR_F32) {
            st16(static_cast<float*>(chunk) + e, make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                                                            __float_as_uint(f[2]), __float_as_uint(f[3])));
        } else {
            st8_plain(static_cast<uint16_t*>(chunk) + e, Payload<DT>::narrow(f), Payload<DT>::narrow(f + 2));
        }
    } else {
        store_elems<DT>(chunk, e, 4, len, f);
    }
}
// A warp's batch: L lines (L / 4 per lane group of 8 lanes), two forms.  A
// hop's latency is set by the instructions one warp issues for its batch,
// not by the transfer, so small calls use short batches (L = 8: a short
// chain per hop, a step spread over more warps); large calls, which are
// bound by instruction throughput, use long ones (L = 32: the per-batch work
// amortised over 4x the data).  kSlots batches per warp fit the inbox, and
// the kernel is compiled for kMinBlocks CTAs per SM.  Measured on GB300 (n = 8
// bf16, graph replay): 12.1 / 14.4 us at 64 KiB / 1 MiB per rank with short
// batches, 49.2 us at 8 MiB and 365 us at 64 MiB with long ones (the step
// ring: 19.0 / 23.2 / 58.6 / 435 us); 16- and 24-line batches, and three CTAs
// per SM for long ones, were slower.
template <int L> struct Geo {
    static constexpr int kLines = L;
    static constexpr int kSlots = L == 8 ? 6 : 3;   // inbox slots per warp
    static constexpr int kMinBlocks = 2;             // 4 for short batches measured 0.9-1.3 us slower
    static constexpr size_t kBatchElems = (size_t)kCWords * L;
    static constexpr size_t kSlotBytes = (size_t)L * 128;
    static constexpr size_t kInboxBytes = (size_t)kCWarps * kSlots * kSlotBytes;
    // inbox, then full[kCWarps][kSlots] and empty[kCWarps][kSlots] mbarriers and the abort word
    static constexpr size_t kSmem = kInboxBytes + (2 * kCWarps * kSlots + 2) * sizeof(uint64_t);
};
constexpr unsigned kCFull = 0xffffffffu;

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

__device__ __forceinline__ void st_rlx_peer(uint32_t a, uint64_t v)
{
    asm volatile("st.relaxed.cluster.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// One try of waiting for phase `parity` of a barrier of this CTA, acquiring
// at cluster scope what the phase's arrivals (and counted bytes) published.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Arrive on a barrier of another CTA of the cluster (relaxed: the caller has
// already consumed what the arrival releases).
__device__ __forceinline__ void mbar_arrive_peer(uint32_t bar)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on a barrier of another CTA, announcing `bytes` of asynchronous
// stores that will complete on it.
__device__ __forceinline__ void mbar_arrive_expect_tx_peer(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// 16 bytes into another CTA's shared memory, counted on its barrier `bar`.
__device__ __forceinline__ void st16_async_peer(uint32_t a, const uint4& v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1,%2,%3,%4}, [%5];" ::"r"(a),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
                 : "memory");
}

// 8 bytes into another CTA's shared memory, counted on its barrier `bar`.
__device__ __forceinline__ void st8_async_peer(uint32_t a, uint32_t x, uint32_t y, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1,%2}, [%3];" ::"r"(a),
                 "r"(x), "r"(y), "r"(bar)
                 : "memory");
}

struct ClusterSmem {
    uint32_t inbox;   // shared address of this CTA's inbox
    uint32_t full;    // full[0][0]
    uint32_t empty;   // empty[0][0]
    uint32_t abort;   // the abort word
};

// Raise the abort word of every CTA of the cluster.
template <int NR>
__device__ void raise_abort(const ClusterSmem& S)
{
#pragma unroll
    for (int q = 0; q < NR; ++q) st_rlx_peer(peer_addr(S.abort, (uint32_t)q), 1ull);
}

// Bounded wait of a whole warp on phase `parity` of a local barrier.  Returns
// false if spin_ns passed or the abort word was raised first.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint32_t abort, int64_t spin_ns)
{
    bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(kCFull, ok)) return true;
    const uint64_t t0 = globaltimer_ns(), cap = (uint64_t)spin_ns / 16u + 4096u;
    for (uint64_t it = 0; it < cap; ++it) {
        if (!ok) ok = mbar_try_wait(bar, parity);
        if (__all_sync(kCFull, ok)) return true;
        if ((it & 15) == 15 &&
            __any_sync(kCFull, (int64_t)(globaltimer_ns() - t0) > spin_ns || ld_rlx_local(abort) != 0))
            return false;
    }
    return false;
}

template <int NR, int DT, int L>
__global__ void __launch_bounds__(kThreads, Geo<L>::kMinBlocks)
ring_cluster_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t C,
                    size_t count, size_t epc, int64_t spin_ns, int absent, DevStatus* st)
{
    using T = typename Payload<DT>::scalar_t;
    constexpr int kCLines = Geo<L>::kLines, kSlots = Geo<L>::kSlots;
    constexpr size_t kSlotBytes = Geo<L>::kSlotBytes;
    constexpr int kI = kCLines / 4;
    // 16-bit payloads: the all-gather hops carry the completed values in the payload type (half the
    // bytes of fp32 lines); fp32 payloads keep fp32 lines throughout
    constexpr bool kNarrowGather = DT != AR_F32;
    constexpr int kV = kCLines / 8 > 0 ? kCLines / 8 : 1;   // 16-byte payload vectors per lane of a batch
    extern __shared__ __align__(128) unsigned char smem[];
    uint32_t crank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
    const int r = (int)crank;
    const size_t k = blockIdx.x / NR;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 3, j = lane & 7;
    const int d = (r + 1) % NR, p = (r + NR - 1) % NR;   // next and previous rank
    ClusterSmem S;
    S.inbox = smem_addr(smem);
    S.full = S.inbox + (uint32_t)Geo<L>::kInboxBytes;
    S.empty = S.full + (uint32_t)(kCWarps * kSlots * 8);
    S.abort = S.empty + (uint32_t)(kCWarps * kSlots * 8);

    // barriers and the abort word, initialised before any peer can use them
    if (threadIdx.x < kCWarps * kSlots) {
        mbar_init(S.full + 8 * threadIdx.x, 1);
        mbar_init(S.empty + 8 * threadIdx.x, 1);
    }
    if (threadIdx.x == 0) asm volatile("st.shared.u64 [%0], %1;" ::"r"(S.abort), "l"(0ull) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    cluster_barrier();

    const size_t slice_lo = k * epc;
    const size_t line_lo = slice_lo / kCWords;
    const uint32_t my_box = S.inbox + (uint32_t)(warp * kSlots * kSlotBytes);
    const uint32_t peer_box = peer_addr(my_box, (uint32_t)d);             // the next rank's inbox for this warp
    const uint32_t my_full = S.full + (uint32_t)(warp * kSlots * 8);      // + 8 s: slot s of my inbox
    const uint32_t peer_full = peer_addr(my_full, (uint32_t)d);           // the next rank's, for my sends
    const uint32_t my_empty = S.empty + (uint32_t)(warp * kSlots * 8);    // my sends' slots at the next rank
    const uint32_t prev_empty = peer_addr(my_empty, (uint32_t)p);         // the previous rank's, for my inbox
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
        const size_t nlines = G.slice_hi > slice_lo ? (G.slice_hi - slice_lo + kCWords - 1) / kCWords : 0;
        G.nbatch = (nlines + kCLines - 1) / kCLines;
        G.x = static_cast<const T*>(in.p[r]) + lo;
        G.y = static_cast<T*>(out.p[r]) + lo;
        return G;
    };
    // lines of batch b (from line_lo + 32 b) below the slice's end
    auto live_lines = [&](size_t base, const Geom& G) -> uint32_t {
        const size_t end = (G.slice_hi + kCWords - 1) / kCWords;
        return base >= end ? 0u : (uint32_t)(end - base < (size_t)kCLines ? end - base : kCLines);
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
        const size_t base = line_lo + b * kCLines;
#pragma unroll
        for (int i = 0; i < kI; ++i) {
            const size_t l = base + 4 * i + g;
            load4<DT>(G.x, l * kCWords + 4 * (size_t)j, l * kCWords < G.slice_hi ? G.len : 0, xr[i]);
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
        const size_t base = line_lo + b * kCLines;
        const uint32_t nlive = live_lines(base, G);
        if (kNarrowGather && t >= NR) {
            // an all-gather hop carries the completed values in the payload type: 16-byte
            // vectors of 8 elements, vector u = lane + 32 i of the batch (4 per 32-element line)
            const uint32_t nvec = 4 * nlive;
            const uint32_t s = (uint32_t)(q_recv % kSlots);
            const uint32_t slot = my_box + s * (uint32_t)kSlotBytes;
            if (!warp_wait(my_full + 8 * s, (uint32_t)((q_recv / kSlots) & 1), S.abort, spin_ns)) {
                if (lane == 0 && ld_rlx_local(S.abort) == 0) {
                    report_flag_timeout(st, r, base);
                    raise_abort<NR>(S);
                }
                dead = true;
                break;
            }
            uint4 pv[kV];
#pragma unroll
            for (int i = 0; i < kV; ++i) {
                const uint32_t u = (uint32_t)(lane + 32 * i);
                pv[i] = u < nvec ? ld16_local(slot + 16u * u) : make_uint4(0u, 0u, 0u, 0u);
            }
            // this rank's output first: the stores use the loaded vectors, so every load of
            // the slot has returned before the slot is freed below (elements past the slice's
            // end are neither stored nor read by anyone)
#pragma unroll
            for (int i = 0; i < kV; ++i) {
                const size_t e = base * kCWords + 8 * (size_t)(lane + 32 * i);
                if (e < G.slice_hi) store8_raw<DT>(G.y, e, G.len, pv[i]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_peer(prev_empty + 8 * s);
            ++q_recv;
            int t2 = t;
            size_t b2 = b;
            Geom G2 = G;
            next_pair(t2, b2, G2);
            if (sends) {
                const uint32_t so = (uint32_t)(q_send % kSlots);
                if (q_send >= kSlots &&
                    !warp_wait(my_empty + 8 * so, (uint32_t)((q_send / kSlots - 1) & 1), S.abort, spin_ns)) {
                    if (lane == 0 && ld_rlx_local(S.abort) == 0) {
                        report_wait_timeout(st);
                        raise_abort<NR>(S);
                    }
                    dead = true;
                    break;
                }
                const uint32_t oslot = peer_box + so * (uint32_t)kSlotBytes;
                const uint32_t bar = peer_full + 8 * so;
                if (lane == 0) mbar_arrive_expect_tx_peer(bar, nvec * 16u);
#pragma unroll
                for (int i = 0; i < kV; ++i) {
                    const uint32_t u = (uint32_t)(lane + 32 * i);
                    if (u < nvec) st16_async_peer(oslot + 16u * u, pv[i], bar);
                }
                ++q_send;
            }
            if (!dead && ld_rlx_local(S.abort) != 0) dead = true;
            dead = __any_sync(kCFull, dead);
            t = t2;
            b = b2;
            G = G2;
            continue;
        }
        uint4 w[kI];
#pragma unroll
        for (int i = 0; i < kI; ++i) w[i] = make_uint4(0u, 0u, 0u, 0u);
        if (t >= 1) {   // receive: batch q_recv in slot q_recv % kSlots
            const uint32_t s = (uint32_t)(q_recv % kSlots);
            const uint32_t slot = my_box + s * (uint32_t)kSlotBytes;
            if (!warp_wait(my_full + 8 * s, (uint32_t)((q_recv / kSlots) & 1), S.abort, spin_ns)) {
                if (lane == 0 && ld_rlx_local(S.abort) == 0) {
                    report_flag_timeout(st, r, base);
                    raise_abort<NR>(S);
                }
                dead = true;
                break;
            }
#pragma unroll
            for (int i = 0; i < kI; ++i)
                if ((uint32_t)(4 * i + g) < nlive) w[i] = ld16_local(slot + (uint32_t)((4 * i + g) * 128 + 16 * j));
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
        if (t >= NR) {
            // an all-gather hop in fp32 lines: nothing above used the loaded lines, so this
            // rank's output goes first -- its stores use them, so every load of the slot has
            // returned before the slot is freed below
#pragma unroll
            for (int i = 0; i < kI; ++i) {
                const size_t l = base + 4 * i + g;
                if (l * kCWords < G.slice_hi) store4<DT>(G.y, l * kCWords + 4 * (size_t)j, G.len, v[i]);
            }
        }
        if (t >= 1) {
            // the slot's lines are in registers and used: free it for the previous rank
            __syncwarp();
            if (lane == 0) mbar_arrive_peer(prev_empty + 8 * (uint32_t)(q_recv % kSlots));
            ++q_recv;
        }
        // the next pair's own elements now: their loads fly during the send
        int t2 = t;
        size_t b2 = b;
        Geom G2 = G;
        next_pair(t2, b2, G2);
        if (t2 <= kLast) load_x(t2, b2, G2);
        if (sends) {
            const uint32_t s = (uint32_t)(q_send % kSlots);
            // the next rank must have read the batch that last used this slot
            if (q_send >= kSlots &&
                !warp_wait(my_empty + 8 * s, (uint32_t)((q_send / kSlots - 1) & 1), S.abort, spin_ns)) {
                if (lane == 0 && ld_rlx_local(S.abort) == 0) {
                    report_wait_timeout(st);
                    raise_abort<NR>(S);
                }
                dead = true;
                break;
            }
            const uint32_t slot = peer_box + s * (uint32_t)kSlotBytes;
            const uint32_t bar = peer_full + 8 * s;
            if (kNarrowGather && t == NR - 1) {
                // the first all-gather hop: the rounded values in the payload type, 8 bytes a lane
                if (lane == 0) mbar_arrive_expect_tx_peer(bar, nlive * 64u);
#pragma unroll
                for (int i = 0; i < kI; ++i) {
                    if ((uint32_t)(4 * i + g) >= nlive) continue;
                    st8_async_peer(slot + (uint32_t)((4 * i + g) * 64 + 8 * j), Payload<DT>::narrow(v[i]),
                                   Payload<DT>::narrow(v[i] + 2), bar);
                }
            } else {
                if (lane == 0) mbar_arrive_expect_tx_peer(bar, nlive * 128u);
#pragma unroll
                for (int i = 0; i < kI; ++i) {
                    if ((uint32_t)(4 * i + g) >= nlive) continue;
                    const uint32_t a = slot + (uint32_t)((4 * i + g) * 128 + 16 * j);
                    st16_async_peer(a, make_uint4(__float_as_uint(v[i][0]), __float_as_uint(v[i][1]),
                                                  __float_as_uint(v[i][2]), __float_as_uint(v[i][3])), bar);
                }
            }
            ++q_send;
        }
        // the completing step's output last, after the hop is on its way
        if (t == NR - 1) {
#pragma unroll
            for (int i = 0; i < kI; ++i) {
                const size_t l = base + 4 * i + g;
                if (l * kCWords < G.slice_hi) store4<DT>(G.y, l * kCWords + 4 * (size_t)j, G.len, v[i]);
            }
        }
        if (!dead && ld_rlx_local(S.abort) != 0) dead = true;
        dead = __any_sync(kCFull, dead);
        t = t2;
        b = b2;
        G = G2;
    }
    // nothing is sent after this barrier
    cluster_barrier();
    if (ld_rlx_local(S.abort) != 0) {
        // after an abort an announced batch may still be landing in this
        // CTA's inbox: wait (bounded) for the next phase of every slot the
        // previous rank may have filled since this warp last read it
        const int64_t drain_ns = spin_ns < 100000 ? spin_ns : 100000;
        for (uint32_t s = 0; s < (uint32_t)kSlots; ++s) {
            const uint64_t used = q_recv > s ? (q_recv - s + kSlots - 1) / kSlots : 0;   // reads of slot s
            const uint32_t bar = my_full + 8 * s;
            const uint64_t t0 = globaltimer_ns();
            for (uint64_t it = 0; it < 65536; ++it) {
                if (mbar_try_wait(bar, (uint32_t)(used & 1))) break;
                if ((int64_t)(globaltimer_ns() - t0) > drain_ns) break;
            }
        }
    }
    // no CTA leaves while a peer may still touch its shared memory
    cluster_barrier();
}

// The kernel's attributes, set once per device, and the clusters of it that
// fit on the GPU at once (computed once per instantiation); 0 if the device
// cannot run a cluster of NR such CTAs.
template <int NR, int DT, int L>
int cluster_setup()
{
    static std::atomic<uint32_t> attr_done{0};
    const bool attr_ok = once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(ring_cluster_kernel<NR, DT, L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)Geo<L>::kSmem) == cudaSuccess &&
               (NR <= 8 || cudaFuncSetAttribute(ring_cluster_kernel<NR, DT, L>,
                                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess);
    });
    if (!attr_ok) return 0;
    static const int resident = [] {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = NR;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t q{};
        q.gridDim = dim3((unsigned)(NR * 64));
        q.blockDim = dim3(kThreads);
        q.dynamicSmemBytes = Geo<L>::kSmem;
        q.attrs = attr;
        q.numAttrs = 1;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, ring_cluster_kernel<NR, DT, L>, &q) != cudaSuccess) nc = 0;
        cudaGetLastError();
        return nc;
    }();
    return resident;
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
            const size_t C = chunk_elems(NR, count, DT);
            auto run = [&](auto lc) -> int {
                constexpr int L = decltype(lc)::value;
                using G = Geo<L>;
                const int resident = cluster_setup<NR, DT, L>();
                if (resident < 1) return AR_ERR_CUDA;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = NR;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cudaLaunchConfig_t cfg{};
                cfg.blockDim = dim3(kThreads);
                cfg.dynamicSmemBytes = G::kSmem;
                cfg.stream = s;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                // slices of at least one batch per warp; one wave of clusters
                // unless that would give a warp more than kSlots batches per step
                // (at step 0 every rank sends without receiving, so a step's
                // batches must fit the receiver's slots)
                const size_t per_cta_min = G::kBatchElems * kCWarps;
                size_t K = (C + per_cta_min - 1) / per_cta_min;
                if (K > (size_t)resident) K = (size_t)resident;
                if (K < 1) K = 1;
                size_t epc = (C + K - 1) / K;
                epc = (epc + G::kBatchElems - 1) / G::kBatchElems * G::kBatchElems;
                if (epc > G::kBatchElems * kCWarps * G::kSlots) epc = G::kBatchElems * kCWarps * G::kSlots;
                K = (C + epc - 1) / epc;
                if (K < 1) K = 1;
                cfg.gridDim = dim3((unsigned)(K * NR));
                const uint64_t S = (uint64_t)count * sizeof(typename Payload<DT>::scalar_t);
                rec_begin(h, s);
                const cudaError_t err = cudaLaunchKernelEx(&cfg, ring_cluster_kernel<NR, DT, L>, ip, op, C, count,
                                                           epc, h.spin_ns, h.persist_absent, h.status);
                rec_end(h, s, AR_K_RING_CLUSTER, 2ull * NR * S);
                *launches = 1;
                if (err != cudaSuccess) {
                    cudaGetLastError();
                    return AR_ERR_CUDA;
                }
                return launch_status();
            };
            // short batches while one wave of clusters gives every warp at most two
            // of them per step: small calls are latency-bound and gain from short
            // batches (14.6 against 30.6 us at 64 KiB, n = 8 bf16), large ones are
            // bound by instruction throughput and gain from long ones
            const int res8 = cluster_setup<NR, DT, 8>();
            if (res8 > 0 && C <= (size_t)res8 * kCWarps * Geo<8>::kBatchElems * 2)
                return run(std::integral_constant<int, 8>{});
            return run(std::integral_constant<int, 32>{});
        });
    });
}

}  // namespace argb
