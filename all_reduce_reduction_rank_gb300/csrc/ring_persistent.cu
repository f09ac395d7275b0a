// Persistent ring all-reduce: all 2(n-1) steps of the ring in one launch,
// every hop carried as LL128 lines with per-step flags.
//
// Handbook "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce", §协议:
// an LL128 line holds 120 bytes of data and an 8-byte flag, and the receiver
// polls the flag instead of waiting at a barrier, so a hop can start on a
// line as soon as that line has arrived.  "多 GPU 与 NCCL", §ring
// all-reduce: the reduce-scatter and all-gather steps and their chunk
// rotation.  The sums are those of ar_ring (fp32 partials; chunk c summed in
// the order c, c+1, ...; rounded once, at the last reduce-scatter hop), so
// the result equals ar_ring's bit for bit.
//
// One cooperative launch: blockIdx.y = rank r, blockIdx.x = CTA k of the
// rank.  CTA k of every rank owns the same slice [k E, (k+1) E) of whichever
// chunk a step moves (E a multiple of 960 elements = 32 lines), so CTA k of
// rank r exchanges lines only with CTA k of ranks r-1 and r+1.  Rank r sends
// at step t:
//   t = 0              its own chunk r, widened to fp32;
//   1 <= t <= n-2      received partial + own chunk (r - t) mod n;
//   t = n-1            received partial + own chunk r+1, rounded: written to
//                      out[r], then sent (the first all-gather hop);
//   n <= t <= 2n-3     the completed chunk received, written to out[r] and
//                      passed on;
// and after the last step writes the last completed chunk it receives.
//
// Inbox of rank q: two slots (step parity) of `lps` lines.  Line l of a slot
// holds elements 30 l .. 30 l + 29 of the chunk as fp32 words, and the flag
// F(t) = 64 seq + t + 1 of the step t that wrote it (seq is new for every
// call, so no line of an earlier call matches).
//
// Ordering follows the PTX memory model and does not assume that a 128-byte
// line is stored atomically: a warp writes the data of 32 lines, then
// __syncwarp, fence.acq_rel.gpu and one relaxed flag store per lane; a reader
// polls one flag per lane (relaxed loads), then fence.acq_rel.gpu and
// __syncwarp, and only then reads the data.
//
// Slot reuse: step t writes slot t % 2 of rank r+1, which step t-2 wrote
// last.  The receiving CTA publishes ack = F(t') (release) once it has
// consumed message t' of its slice; the sending CTA waits for
// ack >= F(t-2) before it writes.
//
// Every wait is bounded by spin_ns and a poll count.  A wait that runs out
// records AR_ERR_FLAG_TIMEOUT (a line) or AR_ERR_WAIT_TIMEOUT (an ack) in the
// status word and raises the call's abort word (= seq), on which every other
// wait gives up at once; each CTA then leaves its step loop at a barrier that
// all its threads reach.
#include "common.cuh"

namespace argb {
namespace {

constexpr int kPWarps = kThreads / 32;
constexpr int kLineWords = 30;
constexpr int kBatchLines = 32;                                      // one flag per lane
constexpr size_t kBatchElems = (size_t)kLineWords * kBatchLines;     // 960
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint64_t* p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Inbox data: cached in L2 only, never in the reading SM's L1.
__device__ __forceinline__ uint4 ld16_cg(const void* p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st16_plain(void* p, const uint4& v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st8_plain(void* p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ uint2 ld8_plain(const void* p)
{
    uint2 v;
    asm volatile("ld.global.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld4_plain(const void* p)
{
    uint32_t v;
    asm volatile("ld.global.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Elements e .. e+nw-1 (nw = 4 or 2) of a chunk of `len` elements, widened
// to fp32; elements at or past len read as 0.  e is a multiple of 2, so a
// pair of 16-bit elements is one aligned word and a pair of fp32 one aligned
// 8-byte load.
template <int DT>
__device__ __forceinline__ void load_elems(const void* chunk, size_t e, int nw, size_t len, float* f)
{
    using T = typename Payload<DT>::scalar_t;
    const T* x = static_cast<const T*>(chunk);
    if (e + (size_t)nw <= len) {
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
            if (u >= nw) break;
            if constexpr (DT == AR_F32) {
                const uint2 a = ld8_plain(x + e + u);
                f[u] = __uint_as_float(a.x);
                f[u + 1] = __uint_as_float(a.y);
            } else {
                Payload<DT>::widen(ld4_plain(x + e + u), f + u);
            }
        }
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) f[u] = u < nw && e + u < len ? Payload<DT>::widen1(x[e + u]) : 0.0f;
    }
}

// Rounds f[0..nw) to the payload type and stores the elements below len.
template <int DT>
__device__ __forceinline__ void store_elems(void* chunk, size_t e, int nw, size_t len, const float* f)
{
    using T = typename Payload<DT>::scalar_t;
    T* y = static_cast<T*>(chunk);
    if (e + (size_t)nw <= len) {
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
            if (u >= nw) break;
            if constexpr (DT == AR_F32) {
                st8_plain(y + e + u, __float_as_uint(f[u]), __float_as_uint(f[u + 1]));
            } else {
                const uint32_t w = Payload<DT>::narrow(f + u);
                asm volatile("st.global.u32 [%0], %1;" ::"l"(y + e + u), "r"(w) : "memory");
            }
        }
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (u < nw && e + u < len) y[e + u] = Payload<DT>::narrow1(f[u]);
    }
}

__device__ __forceinline__ uint64_t* flag_of(uint4* lines, size_t l)
{
    return reinterpret_cast<uint64_t*>(lines + 8 * l + 7) + 1;
}

struct Persist {
    uint4* inbox;        // [n][2][lps] lines
    uint64_t* acks;      // [n][kcap]
    uint64_t* abort_w;   // one word: == seq once a wait of this call gave up
    size_t lps;
    int kcap;
};

__device__ __forceinline__ bool aborted(const Persist& P, uint64_t seq) { return ld_relaxed(P.abort_w) == seq; }

// Every lane of the warp: wait until the flag of its line (if `valid`) reads
// `want`.  False (for the whole warp) if the wait ran out or the call was
// aborted.
__device__ bool wait_lines(const Persist& P, uint64_t seq, const uint64_t* flag, bool valid, uint64_t want,
                           int64_t spin_ns, DevStatus* st, int rank, size_t line)
{
    bool ok = !valid || ld_relaxed(flag) == want;
    if (__all_sync(kFull, ok)) return true;
    const uint64_t t0 = globaltimer_ns(), cap = (uint64_t)spin_ns / 32u + 64u;
    for (uint64_t it = 0; it < cap; ++it) {
        __nanosleep(32);
        if (!ok) ok = ld_relaxed(flag) == want;
        if (__all_sync(kFull, ok)) return true;
        const bool stop = (int64_t)(globaltimer_ns() - t0) > spin_ns || aborted(P, seq);
        if (__any_sync(kFull, stop)) break;
    }
    if (!ok && !aborted(P, seq)) {
        report_flag_timeout(st, rank, line);
        st_relaxed(P.abort_w, seq);
    }
    return false;
}

// One thread: wait until *ack >= want, then acquire.  False if the wait ran
// out or the call was aborted.
__device__ bool wait_ack(const Persist& P, uint64_t seq, const uint64_t* ack, uint64_t want, int64_t spin_ns,
                         DevStatus* st)
{
    if (ld_relaxed(ack) >= want) {
        fence_gpu();   // the block's later stores follow it through the barrier
        return true;
    }
    const uint64_t t0 = globaltimer_ns(), cap = (uint64_t)spin_ns / 32u + 64u;
    for (uint64_t it = 0; it < cap; ++it) {
        __nanosleep(32);
        if (ld_relaxed(ack) >= want) {
            fence_gpu();
            return true;
        }
        if (aborted(P, seq)) return false;
        if ((int64_t)(globaltimer_ns() - t0) > spin_ns) break;
    }
    if (!aborted(P, seq)) {
        report_wait_timeout(st);
        st_relaxed(P.abort_w, seq);
    }
    return false;
}

template <int NR, int DT>
__global__ void __launch_bounds__(kThreads)
ring_persistent_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out,
                       const __grid_constant__ Persist P, size_t C, size_t count, size_t epc, uint64_t seq,
                       int64_t spin_ns, int absent, DevStatus* st)
{
    using T = typename Payload<DT>::scalar_t;
    const int r = blockIdx.y;
    const int k = blockIdx.x;
    if (r == absent) return;  // a rank that never joins (failure emulation)
    const int d = (r + 1) % NR;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 3, j = lane & 7;
    const int nw = j < 7 ? 4 : 2;
    const size_t slice_lo = (size_t)k * epc;              // first element of the slice in a chunk
    const size_t line_lo = slice_lo / kLineWords;         // its first line
    uint64_t* const my_ack = P.acks + (size_t)r * P.kcap + k;
    const uint64_t* const next_ack = P.acks + (size_t)d * P.kcap + k;
    auto inbox = [&](int q, int slot) { return P.inbox + ((size_t)q * 2 + slot) * P.lps * 8; };
    auto chunk_len = [&](int c) -> size_t {
        const size_t lo = (size_t)c * C;
        return lo >= count ? 0 : (count - lo < C ? count - lo : C);
    };

    // t in [0, 2n-2): send step t; t = 2n-2: only the last receive.
    for (int t = 0; t <= 2 * NR - 2; ++t) {
        const bool sends = t <= 2 * NR - 3;
        bool fail = false;
        if (sends && t >= 2 && threadIdx.x == 0)
            fail = !wait_ack(P, seq, next_ack, 64 * seq + (uint64_t)(t - 2) + 1, spin_ns, st);
        if (__syncthreads_or(fail)) break;

        // the chunk this step moves (received at t-1 and sent at t: the same)
        const int c = t <= NR - 2 ? ((r - t) % NR + NR) % NR : ((r + NR - t) % NR + NR) % NR;
        const size_t len = chunk_len(c);
        const size_t slice_hi = slice_lo + epc < len ? slice_lo + epc : len;
        const size_t nlines = slice_hi > slice_lo ? (slice_hi - slice_lo + kLineWords - 1) / kLineWords : 0;
        const size_t nbatch = (nlines + kBatchLines - 1) / kBatchLines;
        const T* const x = static_cast<const T*>(in.p[r]) + (size_t)c * C;
        T* const y = static_cast<T*>(out.p[r]) + (size_t)c * C;
        uint4* const rx = inbox(r, (t + 1) & 1);   // slot of message t-1
        uint4* const tx = inbox(d, t & 1);         // slot of message t
        const uint64_t f_in = 64 * seq + (uint64_t)t;        // F(t-1)
        const uint64_t f_out = 64 * seq + (uint64_t)t + 1;   // F(t)

        for (size_t b = warp; b < nbatch; b += kPWarps) {
            const size_t base = line_lo + b * kBatchLines;   // first line of the batch
            if (t >= 1) {
                const size_t fl = base + lane;
                if (!wait_lines(P, seq, flag_of(rx, fl), fl * kLineWords < slice_hi, f_in, spin_ns, st, r, fl)) {
                    fail = true;
                    break;
                }
                fence_gpu();
                __syncwarp();
            }
#pragma unroll 2
            for (int i = 0; i < kBatchLines / 4; ++i) {
                const size_t l = base + 4 * i + g;
                const size_t e = l * kLineWords + 4 * (size_t)j;
                if (l * kLineWords >= slice_hi) continue;
                float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (t >= 1) {
                    const uint4 w = ld16_cg(rx + 8 * l + j);
                    v[0] = __uint_as_float(w.x);
                    v[1] = __uint_as_float(w.y);
                    v[2] = __uint_as_float(w.z);
                    v[3] = __uint_as_float(w.w);
                }
                if (t <= NR - 1) {   // reduce-scatter: add this rank's own chunk
                    float xv[4];
                    load_elems<DT>(x, e, nw, len, xv);
                    if (t == 0) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) v[u] = xv[u];
                    } else {
#pragma unroll
                        for (int u = 0; u < 4; ++u) v[u] = v[u] + xv[u];
                    }
                }
                if (t >= NR - 1) {   // a completed chunk: this rank's output
                    if (t == NR - 1) {   // rounded once; the rounded value is passed on
#pragma unroll
                        for (int u = 0; u < 4; ++u) v[u] = Payload<DT>::widen1(Payload<DT>::narrow1(v[u]));
                    }
                    store_elems<DT>(y, e, nw, len, v);
                }
                if (sends) {
                    if (j < 7)
                        st16_plain(tx + 8 * l + j, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                                                              __float_as_uint(v[2]), __float_as_uint(v[3])));
                    else
                        st8_plain(tx + 8 * l + j, __float_as_uint(v[0]), __float_as_uint(v[1]));
                }
            }
            if (sends) {
                __syncwarp();
                fence_gpu();
                const size_t fl = base + lane;
                if (fl * kLineWords < slice_hi) st_relaxed(flag_of(tx, fl), f_out);
            }
        }
        if (threadIdx.x == 0 && !fail) fail = aborted(P, seq);
        if (__syncthreads_or(fail)) break;
        if (t >= 1 && sends && threadIdx.x == 0) {   // message t-1 of this slice consumed
            fence_gpu();
            st_relaxed(my_ack, f_in);
        }
    }
}

}  // namespace

// CTAs per SM the inboxes are sized for; launches never use more.
constexpr int kPersistCtasPerSm = 8;

static int persist_kcap(int n, int sm_count) { return (kPersistCtasPerSm * sm_count + n - 1) / n; }

static size_t persist_lps(int n, size_t max_bytes, int sm_count)
{
    // the largest chunk (16-bit payloads give the most elements), plus one
    // batch of slack for every CTA's rounded-up slice
    const size_t cmax = chunk_elems(n, max_bytes / 2, AR_BF16);
    return (cmax + kLineWords - 1) / kLineWords + (size_t)kBatchLines * (size_t)persist_kcap(n, sm_count);
}

size_t persist_bytes(int n, size_t max_bytes, int sm_count)
{
    return (size_t)n * 2 * persist_lps(n, max_bytes, sm_count) * 128 +
           (size_t)n * (size_t)persist_kcap(n, sm_count) * sizeof(uint64_t) + 256;
}

// Lines moved per step over all ranks: the sum over chunks of ceil(len / 30).
uint64_t persist_lines_per_step(int n, size_t count, int dt)
{
    const size_t C = chunk_elems(n, count, dt);
    uint64_t lines = 0;
    for (int c = 0; c < n; ++c) {
        const size_t lo = (size_t)c * C;
        const size_t len = lo >= count ? 0 : (count - lo < C ? count - lo : C);
        lines += (len + kLineWords - 1) / kLineWords;
    }
    return lines;
}

int launch_ring_persistent(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                           cudaStream_t s, int* launches)
{
    if (!h.persist) return AR_ERR_INVALID;
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
            static const int occ = blocks_per_sm(ring_persistent_kernel<NR, DT>);
            const int per_sm = h.ctas_per_sm ? (h.ctas_per_sm < occ ? h.ctas_per_sm : occ) : occ;
            const int cap_sm = per_sm < kPersistCtasPerSm ? per_sm : kPersistCtasPerSm;
            const int kmax = cap_sm * h.sm_count / NR;
            if (kmax < 1) return AR_ERR_CUDA;
            const size_t C = chunk_elems(NR, count, DT);
            // every warp of a CTA gets at least one batch of 32 lines
            const size_t per_cta_min = kBatchElems * kPWarps;
            size_t K = (C + per_cta_min - 1) / per_cta_min;
            if (K > (size_t)kmax) K = (size_t)kmax;
            if (K < 1) K = 1;
            size_t epc = (C + K - 1) / K;
            epc = (epc + kBatchElems - 1) / kBatchElems * kBatchElems;
            K = (C + epc - 1) / epc;
            if (K < 1) K = 1;
            const size_t lps = persist_lps(h.n, h.max_bytes, h.sm_count);
            if (K * epc / kLineWords > lps || (int)K > persist_kcap(h.n, h.sm_count)) return AR_ERR_CUDA;
            Persist P;
            P.inbox = reinterpret_cast<uint4*>(h.persist);
            P.lps = lps;
            P.kcap = persist_kcap(h.n, h.sm_count);
            P.acks = reinterpret_cast<uint64_t*>(h.persist + (size_t)h.n * 2 * lps * 128);
            P.abort_w = P.acks + (size_t)h.n * P.kcap;
            const uint64_t seq = ++h.persist_seq;

            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeCooperative;
            attr[0].val.cooperative = 1;
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = dim3((unsigned)K, NR);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = 0;
            cfg.stream = s;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            const uint64_t e = sizeof(typename Payload<DT>::scalar_t);
            const uint64_t L = persist_lines_per_step(NR, count, DT);
            const uint64_t bytes = 2ull * ((uint64_t)NR * e * count + (uint64_t)(2 * NR - 2) * 128ull * L);
            rec_begin(h, s);
            const cudaError_t err = cudaLaunchKernelEx(&cfg, ring_persistent_kernel<NR, DT>, ip, op, P, C, count,
                                                       epc, seq, h.spin_ns, h.persist_absent, h.status);
            rec_end(h, s, AR_K_RING_PERSISTENT, bytes);
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
