// Host-side internals of libar_gb300.so: the handle, the launch plan and the
// per-file launchers.  Not part of the C-ABI (that is include/ar.h).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <type_traits>
#include <vector>

#include <cuda_runtime.h>

#include "ar.h"

namespace argb {

constexpr int kMaxRanks = 16;
constexpr int kThreads = 256;  // threads per CTA of the streaming kernels

struct DevStatus;

// Optional per-launch timing (AR_OPT_TIMING): a ring of event pairs created
// when the option is set; recording costs two cudaEventRecord calls per
// launch and allocates nothing.
struct Timing {
    int capacity = 0;
    std::vector<cudaEvent_t> start, stop;
    std::vector<ar_launch_time_t> rec;
    size_t head = 0, count = 0;
    int op = 0;      // the call being recorded
    int paused = 0;  // AR_OPT_TIMING_PAUSE: keep the events, record nothing
};

struct Handle {
    int n = 0;
    size_t max_bytes = 0;
    int device = 0;
    int sm_count = 0;
    int l2_bytes = 0;   // the device's L2 size
    int ctas_per_sm = 0;  // 0: one full wave, from each kernel's occupancy
    int64_t spin_ns = 1000000;
    int one_shot_impl = 0;
    int pdl = 1;  // programmatic dependent launch between consecutive kernels
    int auto_policy = AR_AUTO_MODEL;
    int64_t auto_alpha_ns = 1500;
    int64_t auto_beta_mbs = 450000;
    int64_t auto_handoff = 8 << 20;
    uint8_t* push_stage = nullptr;  // [n][n][stage_slot] (AR_OPT_PUSH_STAGING)
    uint8_t* registered = nullptr;  // [n][stage_slot] (AR_OPT_REGISTERED)
    size_t stage_slot = 0;          // max_bytes rounded up to 256
    uint8_t* persist = nullptr;     // ar_ring_persistent's inboxes, acks, abort word (AR_OPT_PERSISTENT)
    int persist_absent = -1;        // AR_OPT_ABSENT_RANK
    int two_shot_impl = 0;          // AR_OPT_TWO_SHOT_IMPL
    unsigned* two_shot_sync = nullptr;  // the one-launch two-shot's counters and tile flags
    size_t two_shot_sync_words = 0;
    float* ring_scratch = nullptr;  // [2][n][ring_chunk_max] fp32 partials
    size_t ring_chunk_max = 0;      // elements
    // a second stream for the ring's pieces, forked from and joined to the
    // caller's stream by these events within each call
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    DevStatus* status = nullptr;    // device
    cudaStream_t last_stream = nullptr;
    ar_traffic_t last{};
    Timing timing;
};

// Bracket one launch, or a run of consecutive launches of one kernel, with the
// timing events (no-ops when timing is off).
inline void rec_begin(Handle& h, cudaStream_t s)
{
    Timing& t = h.timing;
    if (t.capacity && !t.paused) cudaEventRecord(t.start[t.head], s);
}

inline void rec_end(Handle& h, cudaStream_t s, int kernel, uint64_t hbm_bytes, int launches = 1)
{
    Timing& t = h.timing;
    if (!t.capacity || t.paused) return;
    cudaEventRecord(t.stop[t.head], s);
    t.rec[t.head] = ar_launch_time_t{kernel, t.op, 0.0f, hbm_bytes, launches};
    t.head = (t.head + 1) % (size_t)t.capacity;
    if (t.count < (size_t)t.capacity) ++t.count;
}

inline size_t elem_bytes(int dt) { return dt == AR_F32 ? 4u : 2u; }

// Two-shot / ring chunk: ceil(N/n) rounded up to a whole 16-byte vector.
inline size_t chunk_elems(int n, size_t N, int dt)
{
    size_t per = (N + (size_t)n - 1) / (size_t)n;
    size_t q = 16u / elem_bytes(dt);
    return (per + q - 1) / q * q;
}

// ar_two_shot's form: AR_OPT_TWO_SHOT_IMPL 1 = two launches, 2 = one launch
// (per-tile CTA barrier), 3 = one launch (per-tile flags between CTAs);
// 0 (auto) = form 2, measured fastest at every size on GB300.
inline bool two_shot_one_launch(int impl) { return impl != 1; }

// CTAs of `kernel` (kThreads threads, no dynamic shared memory) that fit on
// one SM at once.  Callers cache it in a function-local static per kernel
// instantiation.
template <typename K>
inline int blocks_per_sm(K kernel, size_t dyn_smem = 0)
{
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, dyn_smem) != cudaSuccess || b < 1) {
        cudaGetLastError();
        b = 1;
    }
    return b;
}

// Grid sizing of the streaming kernels.  Measured on GB300 (n = 8 bf16,
// 8 and 64 MiB per rank, CTAs/SM swept 1..1024): many short-lived CTAs, up
// to about one tile each, beat one resident wave of grid-striding CTAs by
// 5-14% (the block scheduler balances the SMs; a static split does not), and
// the gain is flat from 32 to 1024 CTAs/SM.  So the default caps the grid at
// kAutoCtasPerSm CTAs per SM and the kernels grid-stride past that.
constexpr int kAutoCtasPerSm = 64;

// CTAs for a streaming kernel that needs `work` thread-iterations.
inline unsigned grid_for(const Handle& h, size_t work)
{
    size_t want = (work + kThreads - 1) / kThreads;
    size_t cap = (size_t)h.sm_count * (size_t)(h.ctas_per_sm ? h.ctas_per_sm : kAutoCtasPerSm);
    if (want > cap) want = cap;
    return want ? (unsigned)want : 1u;
}

// Piece length (elements) for a call of several launches that hands
// `handed_bytes` from one launch to the next over a range of `len` elements:
// the range is cut into P = handed_bytes over half of L2, rounded (at least
// 1, at most kMaxPieces), equal pieces of whole 256-element blocks (whole
// 16-byte vectors of every payload type), so that what one launch hands the
// next stays in L2; each piece then goes through all of the call's launches
// in turn.  `len` when the device's L2 size is unknown or one piece is
// enough.  The cap: every piece adds its launches' ramp and drain (about
// 1.4 us each on GB300), and the largest count measured to help was 57 (push,
// n = 8 bf16, 64 MiB per rank: 57 and 64 pieces took the same time).
constexpr uint64_t kMaxPieces = 64;
inline size_t piece_elems(const Handle& h, uint64_t handed_bytes, size_t len)
{
    const uint64_t half = h.l2_bytes / 2;
    if (half == 0) return len;
    uint64_t P = (handed_bytes + half / 2) / half;
    if (P <= 1) return len;
    if (P > kMaxPieces) P = kMaxPieces;
    size_t pl = (size_t)((len + P - 1) / P);
    pl = (pl + 255) / 256 * 256;
    return pl < len ? pl : len;
}

// Independent pieces on two streams.  A call's pieces do not depend on each
// other, so when it has many the call runs twice as many, half as long,
// alternately on the caller's stream and on the handle's side stream (forked
// from the caller's stream by an event at the start, joined back by another
// at the end, so the call stays stream-ordered and capturable in a CUDA
// graph): one stream's launches fill the other's ramp and drain, and two
// half-length pieces in flight hold in L2 what one piece did.  A call made
// while timing records are taken stays on one stream, so that each record
// times its own launches.
inline bool recording(const Handle& h) { return h.timing.capacity && !h.timing.paused; }

inline bool two_streams(const Handle& h, uint64_t handed_bytes, uint64_t l2_fraction)
{
    return h.side && h.l2_bytes > 0 && handed_bytes * l2_fraction >= (uint64_t)h.l2_bytes && !recording(h);
}

// Half a piece length, in whole 256-element blocks, at most `len`.
inline size_t half_piece(size_t pl, size_t len)
{
    pl = (pl + 1) / 2;
    pl = (pl + 255) / 256 * 256;
    return pl < len ? pl : len;
}

struct PieceStreams {
    Handle& h;
    cudaStream_t main;
    bool on;
    int k = 0;
    int fork() const
    {
        return on && (cudaEventRecord(h.ev_fork, main) != cudaSuccess ||
                      cudaStreamWaitEvent(h.side, h.ev_fork, 0) != cudaSuccess)
                   ? AR_ERR_CUDA
                   : AR_OK;
    }
    cudaStream_t next() { return on && (k++ & 1) ? h.side : main; }   // the next piece's stream
    int join() const   // also after a failed launch, so a stream capture is never left forked
    {
        return on && (cudaEventRecord(h.ev_join, h.side) != cudaSuccess ||
                      cudaStreamWaitEvent(main, h.ev_join, 0) != cudaSuccess)
                   ? AR_ERR_CUDA
                   : AR_OK;
    }
};

// blockIdx.x extent for a 2-D grid of `rows` rows (blockIdx.y) that each need
// `work` thread-iterations, within the same CTA budget.
inline unsigned grid_for_rows(const Handle& h, size_t work, int rows)
{
    size_t want = (work + kThreads - 1) / kThreads;
    size_t total = (size_t)h.sm_count * (size_t)(h.ctas_per_sm ? h.ctas_per_sm : kAutoCtasPerSm);
    size_t cap = total / (size_t)rows;
    if (cap == 0) cap = 1;
    if (want > cap) want = cap;
    return want ? (unsigned)want : 1u;
}

// Launch shape for a call too small to give every SM a full CTA: `work`
// thread-iterations in each of `rows` rows (blockIdx.y), one per thread,
// with the CTAs narrowed (down to one warp) until the grid covers the SMs or
// cannot grow further.  Measured on GB300 (n = 8 bf16, 8 KiB - 1 MiB per
// rank): a small call's time is set by how many SMs move its bytes, not by
// how many threads each SM runs, so narrow CTAs on many SMs beat one wide CTA.
struct Shape {
    unsigned grid_x, block;
};
inline Shape narrow_shape(const Handle& h, size_t work, int rows = 1)
{
    // never more CTAs than the launch cap (AR_OPT_CTAS_PER_SM) allows
    const size_t cap = (size_t)h.sm_count * (size_t)(h.ctas_per_sm ? h.ctas_per_sm : kAutoCtasPerSm);
    unsigned block = kThreads;
    while (block > 32 && ((work + block - 1) / block) * (size_t)rows < (size_t)h.sm_count &&
           ((work + block / 2 - 1) / (block / 2)) * (size_t)rows <= cap)
        block >>= 1;
    size_t want = (work + block - 1) / block;
    return Shape{want ? (unsigned)want : 1u, block};
}

// Kernel attributes (dynamic shared memory size, non-portable cluster size)
// belong to the device they are set on: a launcher sets them through this,
// once per device (a bit per device in `done`), with that device current.
template <typename F>
inline bool once_per_device(std::atomic<uint32_t>& done, F&& set)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 32) return false;
    const uint32_t bit = 1u << dev;
    if (done.load(std::memory_order_acquire) & bit) return true;
    if (!set()) {
        cudaGetLastError();
        return false;
    }
    done.fetch_or(bit, std::memory_order_acq_rel);
    return true;
}

// Launchers: argument checks are done by the caller; these only launch.
int launch_one_shot(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                    cudaStream_t s, int* launches);
int launch_two_shot(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                    cudaStream_t s, int* launches);
size_t two_shot_sync_words(int n, size_t max_bytes);
int launch_ring(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                cudaStream_t s, int* launches);
int launch_ring_rounded(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                        int* launches);
int launch_one_shot_push(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                         int* launches);
int launch_one_shot_copyin(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                           cudaStream_t s, int* launches);
int launch_tree(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                int* launches);
int launch_ring_persistent(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                           cudaStream_t s, int* launches);
size_t persist_bytes(int n, size_t max_bytes, int sm_count);
int launch_tree_fused(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                      int* launches);
int launch_ring_cluster(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                        int* launches);
int launch_ring_fused(Handle& h, const void* const* in, void* const* out, size_t count, int dt, cudaStream_t s,
                      int* launches);
int launch_ring_rounded_fused(Handle& h, const void* const* in, void* const* out, size_t count, int dt,
                              cudaStream_t s, int* launches);
uint64_t persist_lines_per_step(int n, size_t count, int dt);
int launch_ll_pack(Handle& h, int nb, const float* const* src, void* const* lines, size_t count, uint32_t step,
                   cudaStream_t s);
int launch_ll_unpack(Handle& h, int nb, const void* const* lines, float* const* dst, size_t count, uint32_t step,
                     cudaStream_t s);
int launch_ll_reduce(Handle& h, const void* const* in, void* const* out, size_t count,
                     uint32_t step, cudaStream_t s);
int launch_ll128_pack(Handle& h, int nb, const float* const* src, void* const* lines, size_t count, uint64_t step,
                      cudaStream_t s);
int launch_ll128_unpack(Handle& h, int nb, const void* const* lines, float* const* dst, size_t count,
                        uint64_t step, cudaStream_t s);
size_t rmsnorm_slice_vecs(size_t hidden, int dt);
bool rmsnorm_fits(size_t hidden, int dt);
int launch_allreduce_rmsnorm(Handle& h, const void* const* in, const void* residual, const void* weight, float eps,
                             void* const* out, void* residual_out, size_t tokens, size_t hidden, int dt,
                             cudaStream_t s);
int launch_ll128_reduce(Handle& h, const void* const* in, void* const* out, size_t count,
                        uint64_t step, cudaStream_t s);

}  // namespace argb
