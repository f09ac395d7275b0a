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
// Pieces: a CTA takes its slice in P pieces of sp elements (a multiple of 32
// lines) and runs all 2(n-1) steps of the ring on one piece before the next,
// so that what is in flight is one piece's messages.  P is the two inbox
// slots of a whole step (all ranks' lines) over half of L2, rounded: large
// calls then keep their messages in L2 instead of sending every line through
// DRAM; small calls run in one piece (each piece pays the ring's hop latency
// 2(n-1) times).  Message m = q (2n-2) + t is step t of piece q.
//
// Inbox of rank q: two slots (message parity) of `lps` lines.  Piece q of
// CTA k uses lines [k sp/30, (k+1) sp/30) of a slot, the same lines for every
// piece; line i of them holds elements 30 i .. 30 i + 29 of the piece's part
// of the chunk as fp32 words, and the flag F(m) = 4096 seq + m + 1 of the
// message m that wrote it.  seq is a call number kept in device memory: every
// warp reads it at the start, and the call's last warp to finish advances it,
// so each call -- also each replay of a captured CUDA graph -- has its own,
// and no line of an earlier call or piece matches.
//
// Ordering follows the PTX memory model and does not assume that a 128-byte
// line is stored atomically: a warp writes the data of 32 lines, then
// __syncwarp, fence.acq_rel.gpu and one relaxed flag store per lane; a reader
// polls one flag per lane with acquire loads, then __syncwarp, and only then
// reads the data.  A warp issues all loads of its 32 lines (and of the rank's
// own elements) before it uses any, so a batch costs about one memory latency.
//
// Slot reuse: message m goes to slot m % 2 of rank r+1, which message m-2
// used last.  Each receiving warp publishes ack = F(m') (release) once it has
// consumed its batches of message m'; the sending warp waits for
// ack >= F(m-2) before it writes.
//
// Every wait is bounded by spin_ns and a poll count.  A wait that runs out
// records AR_ERR_FLAG_TIMEOUT (a line) or AR_ERR_WAIT_TIMEOUT (an ack) in the
// status word and raises the call's abort word (= seq), on which every other
// wait gives up at once; a warp whose wait gave up returns (there is no
// block-wide barrier to leave unmatched).
#include "lines.cuh"

namespace argb {
namespace {

using namespace lines;

constexpr int kPWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint64_t* p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
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

__device__ __forceinline__ uint64_t* flag_of(uint4* lines, size_t l)
{
    return reinterpret_cast<uint64_t*>(lines + 8 * l + 7) + 1;
}

struct Persist {
    uint4* inbox;        // [n][2][lps] lines
    uint64_t* acks;      // [n][kcap][warps per CTA]
    uint64_t* abort_w;   // one word: == seq once a wait of this call gave up
    uint64_t* epoch_w;   // the last finished call's seq
    unsigned* done_w;    // warps of the current call that have finished
    size_t lps;
    int kcap;
};

__device__ __forceinline__ bool aborted(const Persist& P, uint64_t seq) { return ld_relaxed(P.abort_w) == seq; }

// Every lane of the warp: wait until the flag of its line (if `valid`) reads
// `want` (acquire).  False (for the whole warp) if the wait ran out or the
// call was aborted.  The first polls spin; later ones sleep between reads.
__device__ bool wait_lines(const Persist& P, uint64_t seq, const uint64_t* flag, bool valid, uint64_t want,
                           int64_t spin_ns, DevStatus* st, int rank, size_t line)
{
    bool ok = !valid || ld_acquire(flag) == want;
    if (__all_sync(kFull, ok)) return true;
    const uint64_t t0 = globaltimer_ns(), cap = (uint64_t)spin_ns / 32u + 1024u;
    for (uint64_t it = 0; it < cap; ++it) {
        if (it >= 256) __nanosleep(64);
        if (!ok) ok = ld_acquire(flag) == want;
        if (__all_sync(kFull, ok)) return true;
        if ((it & 15) == 15) {
            const bool stop = (int64_t)(globaltimer_ns() - t0) > spin_ns || aborted(P, seq);
            if (__any_sync(kFull, stop)) break;
        }
    }
    if (!ok && !aborted(P, seq)) {
        report_flag_timeout(st, rank, line);
        st_relaxed(P.abort_w, seq);
    }
    return false;
}

// Every lane of the warp: wait until *ack >= want (acquire).  False (for
// the whole warp) if the wait ran out or the call was aborted.
__device__ bool wait_ack(const Persist& P, uint64_t seq, const uint64_t* ack, uint64_t want, int64_t spin_ns,
                         DevStatus* st)
{
    if (__all_sync(kFull, ld_acquire(ack) >= want)) return true;
    const uint64_t t0 = globaltimer_ns(), cap = (uint64_t)spin_ns / 32u + 1024u;
    for (uint64_t it = 0; it < cap; ++it) {
        if (it >= 256) __nanosleep(64);
        if (__all_sync(kFull, ld_acquire(ack) >= want)) return true;
        if ((it & 15) == 15) {
            const bool stop = (int64_t)(globaltimer_ns() - t0) > spin_ns || aborted(P, seq);
            if (__any_sync(kFull, stop)) break;
        }
    }
    if ((threadIdx.x & 31) == 0 && !aborted(P, seq)) {
        report_wait_timeout(st);
        st_relaxed(P.abort_w, seq);
    }
    return false;
}

// Flags of a call: F(m) = kMsgBase seq + m + 1, with m < kMsgBase.
constexpr uint64_t kMsgBase = 4096;
static_assert(kMaxPieces * 30 < kMsgBase, "messages of a call must stay below kMsgBase");

// Work of one warp, piece by piece: batches b = warp, warp + 8, ... of its
// CTA's piece, the same batches on every rank, so warp w of CTA k of rank r exchanges lines and
// acknowledgements only with warp w of CTA k of ranks r-1 and r+1: the step
// loop has no block-wide barrier.  Per batch, software-pipelined: add and
// store the batch (next rank's lines, outputs), acquire the next batch's
// flags and issue its loads, then release this batch (fence, flags) while
// those loads are in flight.  A wait that gives up returns at once.
template <int NR, int DT>
__device__ __forceinline__ void persist_warp(const CPtrs<NR>& in, const MPtrs<NR>& out, const Persist& P, size_t C,
                                             size_t count, size_t epc, size_t sp, uint64_t seq, int64_t spin_ns,
                                             int absent, int prefetch, DevStatus* st)
{
    using T = typename Payload<DT>::scalar_t;
    constexpr int kI = kBatchLines / 4;   // lines per lane group per batch
    const int r = blockIdx.y;
    const int k = blockIdx.x;
    if (r == absent) return;  // a rank that never joins (failure emulation)
    const int d = (r + 1) % NR;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 3, j = lane & 7;
    const int nw = j < 7 ? 4 : 2;
    const size_t slice_end = (size_t)k * epc + epc;       // end of the CTA's slice in a chunk
    const int npieces = (int)((epc + sp - 1) / sp);
    uint64_t* const my_ack = P.acks + ((size_t)r * P.kcap + k) * kPWarps + warp;
    const uint64_t* const next_ack = P.acks + ((size_t)d * P.kcap + k) * kPWarps + warp;
    auto inbox = [&](int rank, int slot) { return P.inbox + ((size_t)rank * 2 + slot) * P.lps * 8; };

    for (int q = 0; q < npieces; ++q) {
        const size_t slice_lo = (size_t)k * epc + (size_t)q * sp;   // first element of the piece in a chunk
        const size_t piece_end = slice_lo + sp < slice_end ? slice_lo + sp : slice_end;
        const size_t line_lo = slice_lo / kLineWords;               // its first line
        // inbox lines are indexed by the chunk's line numbers l, shifted so that
        // this piece's lines land on the CTA's lines [k sp/30, (k+1) sp/30)
        const ptrdiff_t shift = 8 * ((ptrdiff_t)((size_t)k * (sp / kLineWords)) - (ptrdiff_t)line_lo);
        // t in [0, 2n-2): send step t; t = 2n-2: only the last receive.
        for (int t = 0; t <= 2 * NR - 2; ++t) {
            const bool sends = t <= 2 * NR - 3;
            const uint64_t m = (uint64_t)q * (2 * NR - 2) + (uint64_t)t;   // the message this iteration sends
            // the chunk this step moves (received at t-1 and sent at t: the same)
            const int c = t <= NR - 2 ? ((r - t) % NR + NR) % NR : ((r + NR - t) % NR + NR) % NR;
            const size_t lo = (size_t)c * C;
            const size_t len = lo >= count ? 0 : (count - lo < C ? count - lo : C);
            const size_t slice_hi = piece_end < len ? piece_end : len;
            const size_t nlines = slice_hi > slice_lo ? (slice_hi - slice_lo + kLineWords - 1) / kLineWords : 0;
            const size_t nbatch = (nlines + kBatchLines - 1) / kBatchLines;
            const T* const x = static_cast<const T*>(in.p[r]) + lo;
            T* const y = static_cast<T*>(out.p[r]) + lo;
            uint4* const rx = inbox(r, (t + 1) & 1) + shift;   // slot of message m-1 (2n-2 is even)
            uint4* const tx = inbox(d, t & 1) + shift;         // slot of message m
            const uint64_t f_in = kMsgBase * seq + m;        // F(m-1)
            const uint64_t f_out = kMsgBase * seq + m + 1;   // F(m)
            auto flag_ptr = [&](size_t bb) { return flag_of(rx, line_lo + bb * kBatchLines + lane); };
            auto flag_live = [&](size_t bb) { return (line_lo + bb * kBatchLines + lane) * kLineWords < slice_hi; };

            // the rank's own elements of this step, pulled into L2 while the
            // warp waits for the lines (small calls, whose steps are latency-bound)
            if (prefetch && t >= 1 && t <= NR - 1) {
                for (size_t bb = warp; bb < nbatch; bb += kPWarps) {
                    const size_t e0 = (line_lo + bb * kBatchLines) * kLineWords + (size_t)lane * (128 / sizeof(T));
                    if (e0 < slice_hi) prefetch_l2(x + e0);
                }
            }
            // step prologue: the receiver's acknowledgement of message m-2 (slot
            // reuse) and the first batch's flags, polled together, one acquire
            size_t b = warp;
            {
                const bool need_ack = sends && m >= 2, need_fl = t >= 1 && b < nbatch;
                const uint64_t want_ack = kMsgBase * seq + m - 1;   // F(m-2)
                bool ok_ack = !need_ack || ld_relaxed(next_ack) >= want_ack;
                bool ok_fl = !need_fl || !flag_live(b) || ld_relaxed(flag_ptr(b)) == f_in;
                if (!__all_sync(kFull, ok_ack && ok_fl)) {
                    if (!__all_sync(kFull, ok_ack) && !wait_ack(P, seq, next_ack, want_ack, spin_ns, st)) return;
                    if (need_fl && !wait_lines(P, seq, flag_ptr(b), flag_live(b), f_in, spin_ns, st, r,
                                               line_lo + b * kBatchLines + lane))
                        return;
                }
                fence_gpu();
                __syncwarp();
            }
            // a batch's loads: 8 lines and the rank's own elements, all issued
            // before any is used
            uint4 w[kI];
            uint32_t xr[kI][kRawWords<DT>];
            auto load_batch = [&](size_t bb) {
                const size_t base = line_lo + bb * kBatchLines;
#pragma unroll
                for (int i = 0; i < kI; ++i) {
                    const size_t l = base + 4 * i + g;
                    w[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (t >= 1 && l * kLineWords < slice_hi) w[i] = ld16_cg(rx + 8 * l + j);
                }
                if (t <= NR - 1) {
#pragma unroll
                    for (int i = 0; i < kI; ++i) {
                        const size_t l = base + 4 * i + g;
                        load_raw<DT>(x, l * kLineWords + 4 * (size_t)j, nw, l * kLineWords < slice_hi ? len : 0, xr[i]);
                    }
                }
            };
            if (b < nbatch) load_batch(b);
            while (b < nbatch) {
                const size_t base = line_lo + b * kBatchLines;   // first line of the batch
#pragma unroll
                for (int i = 0; i < kI; ++i) {
                    const size_t l = base + 4 * i + g;
                    const size_t e = l * kLineWords + 4 * (size_t)j;
                    if (l * kLineWords >= slice_hi) continue;
                    float v[4] = {__uint_as_float(w[i].x), __uint_as_float(w[i].y), __uint_as_float(w[i].z),
                                  __uint_as_float(w[i].w)};
                    if (t <= NR - 1) {   // reduce-scatter: add this rank's own chunk
                        float xv[4];
                        widen_raw<DT>(xr[i], xv);
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
                // the next batch: acquire its flags and issue its loads before
                // this batch's release, so that they are in flight while this
                // batch's stores drain
                const size_t nb = b + kPWarps;
                if (t >= 1 && nb < nbatch) {
                    const bool ok = __all_sync(kFull, !flag_live(nb) || ld_acquire(flag_ptr(nb)) == f_in);
                    if (!ok && !wait_lines(P, seq, flag_ptr(nb), flag_live(nb), f_in, spin_ns, st, r,
                                           line_lo + nb * kBatchLines + lane))
                        return;
                    __syncwarp();
                }
                if (nb < nbatch) load_batch(nb);
                if (sends) {
                    __syncwarp();
                    fence_gpu();
                    const size_t fl = base + lane;
                    if (fl * kLineWords < slice_hi) st_relaxed(flag_of(tx, fl), f_out);
                }
                b = nb;
            }
            // message m-1 of this warp's batches is consumed (its last batch's
            // values were used before the last fence; a step that sends nothing
            // or had no batch fences here): acknowledge it for the sender's slot
            // reuse.  The last message of the call needs none.
            if (t >= 1 && (sends || q + 1 < npieces) && lane == 0) {
                if (!sends || nbatch <= (size_t)warp) fence_gpu();
                st_relaxed(my_ack, f_in);
            }
        }
    }
}

template <int NR, int DT>
__global__ void __launch_bounds__(kThreads, 2)   // two CTAs per SM: 128 registers, no spills
ring_persistent_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out,
                       const __grid_constant__ Persist P, size_t C, size_t count, size_t epc, size_t sp,
                       int64_t spin_ns, int absent, int prefetch, DevStatus* st)
{
    // the same for every warp: only this call's last warp advances it
    const uint64_t seq = ld_relaxed(P.epoch_w) + 1;
    persist_warp<NR, DT>(in, out, P, C, count, epc, sp, seq, spin_ns, absent, prefetch, st);
    if ((threadIdx.x & 31) == 0) {
        fence_gpu();
        const unsigned total = gridDim.x * gridDim.y * (unsigned)kPWarps;
        if (atomicAdd(P.done_w, 1u) == total - 1) {   // every other warp of the call is done
            *P.done_w = 0u;
            st_relaxed(P.epoch_w, seq);
        }
    }
}

}  // namespace

// Calls up to this many bytes per rank prefetch each step's own elements
// into L2 (the step's elements of all ranks then take at most this much L2).
constexpr uint64_t kPersistPrefetchBytes = 32ull << 20;

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
           (size_t)n * (size_t)persist_kcap(n, sm_count) * kPWarps * sizeof(uint64_t) + 256;
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

// Elements of a CTA's slice per piece: P = the two inbox slots of a step
// (2 x 128 B x L lines) over half of L2, rounded, at most kMaxPieces; sp a
// multiple of 32 lines.  Measured on GB300 (n = 8 bf16, one launch, µs;
// pieces 1 / 2 / 4 / 8): 8 MiB per rank 129 / 173 / 275 / 491, 32 MiB 555 /
// 441 / 469 / 659, 64 MiB 1111 / 1079 / 861 / 968; the rule gives 1, 2, 4.
static size_t persist_piece_elems(const Handle& h, uint64_t L, size_t epc)
{
    const uint64_t half = (uint64_t)h.l2_bytes / 2, live = 2ull * 128ull * L;
    uint64_t P = half ? (live + half / 2) / half : 1;
    if (P < 1) P = 1;
    if (P > kMaxPieces) P = kMaxPieces;
    size_t sp = (epc + P - 1) / P;
    sp = (sp + kBatchElems - 1) / kBatchElems * kBatchElems;
    return sp < epc ? sp : epc;
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
            const uint64_t L = persist_lines_per_step(NR, count, DT);
            const size_t sp = persist_piece_elems(h, L, epc);
            if (K * epc / kLineWords > lps || (int)K > persist_kcap(h.n, h.sm_count)) return AR_ERR_CUDA;
            Persist P;
            P.inbox = reinterpret_cast<uint4*>(h.persist);
            P.lps = lps;
            P.kcap = persist_kcap(h.n, h.sm_count);
            P.acks = reinterpret_cast<uint64_t*>(h.persist + (size_t)h.n * 2 * lps * 128);
            P.abort_w = P.acks + (size_t)h.n * P.kcap * kPWarps;
            P.epoch_w = P.abort_w + 1;
            P.done_w = reinterpret_cast<unsigned*>(P.abort_w + 2);

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
            const uint64_t bytes = 2ull * ((uint64_t)NR * e * count + (uint64_t)(2 * NR - 2) * 128ull * L);
            rec_begin(h, s);
            const cudaError_t err = cudaLaunchKernelEx(&cfg, ring_persistent_kernel<NR, DT>, ip, op, P, C, count,
                                                       epc, sp, h.spin_ns, h.persist_absent,
                                                       (int)(count * e <= kPersistPrefetchBytes), h.status);
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
