// LL and LL128 protocol lines: pack, flag-checked unpack, flag-checked reduce.
//
// Handbook "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce", §协议
// table: LL puts 4 bytes of data and a 4-byte flag in every 8 bytes and the
// receiver polls the flag (about 50% efficiency, lowest latency); LL128 puts
// 120 bytes of data and an 8-byte flag in every 128 bytes (about 94%).
//
// Layout (a reading; the pages give no byte positions):
//   LL line i    = { u32 payload word i, u32 flag }                  (8 B)
//   LL128 line k = { u32 payload words 30k..30k+29, u64 flag }       (128 B)
// An LL128 line is moved by 8 lanes, 16 bytes each; lane 7 of the group
// holds the last two payload words and the flag, so a group votes on lane
// 7's flag.  The flag is the step id.
//
// Consumers check every flag.  A missing flag is re-read (volatile) for at
// most `spin_ns` nanoseconds and a bounded number of polls; a line that never
// shows its flag is not consumed (its output is left untouched) and the
// handle's sticky status records AR_ERR_FLAG_TIMEOUT.  No wait is unbounded.
#include "common.cuh"

namespace argb {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint2 ld8(const void* p)
{
    uint2 v;
    asm volatile("ld.global.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ void st8(void* p, uint2 v)
{
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ uint2 ld8_volatile(const void* p)
{
    uint2 v;
    asm volatile("ld.volatile.global.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// Bound on polls: the time limit normally ends the wait; the poll count ends
// it even if the timer did not advance (each poll is a global round trip of
// well over 32 ns).
__device__ __forceinline__ uint64_t max_polls(int64_t spin_ns) { return (uint64_t)spin_ns / 32u + 64u; }

// ---------------------------------------------------------------- LL -------

// Pack / unpack kernels take a table of buffers; blockIdx.y picks one, so a
// single launch serves one buffer or all n ranks' buffers.  Every LL kernel
// runs in CTAs of up to kThreads threads, narrower (whole warps) for a call
// too small to give every SM a full CTA.
struct SrcTable { const void* p[kMaxRanks]; };
struct DstTable { void* p[kMaxRanks]; };

__global__ void __launch_bounds__(kThreads)
ll_pack_kernel(const __grid_constant__ SrcTable srcs, const __grid_constant__ DstTable outs, size_t count,
               uint32_t step)
{
    pdl_acquire();
    const float* const src = static_cast<const float*>(srcs.p[blockIdx.y]);
    uint4* const lines = static_cast<uint4*>(outs.p[blockIdx.y]);
    const size_t nq = count / 4;  // 4 payload words -> 2 x 16 B of lines
    for (size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x; v < nq; v += (size_t)gridDim.x * blockDim.x) {
        const uint4 x = ld16(src + 4 * v);
        st16(lines + 2 * v, make_uint4(x.x, step, x.y, step));
        st16(lines + 2 * v + 1, make_uint4(x.z, step, x.w, step));
    }
    pdl_release();
    if (blockIdx.x == gridDim.x - 1) {
        const size_t i = nq * 4 + threadIdx.x;
        if (i < count) reinterpret_cast<uint2*>(lines)[i] = make_uint2(__float_as_uint(src[i]), step);
    }
}

__global__ void __launch_bounds__(kThreads)
ll_unpack_kernel(const __grid_constant__ SrcTable ins, const __grid_constant__ DstTable dsts, size_t count,
                 uint32_t step, int64_t spin_ns, DevStatus* st)
{
    pdl_acquire();
    const int rank = blockIdx.y;
    const uint4* const lines = static_cast<const uint4*>(ins.p[rank]);
    float* const dst = static_cast<float*>(dsts.p[rank]);
    const size_t nq = count / 4;
    for (size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x; v < nq; v += (size_t)gridDim.x * blockDim.x) {
        uint4 a = ld16(lines + 2 * v), b = ld16(lines + 2 * v + 1);
        bool ok = a.y == step && a.w == step && b.y == step && b.w == step;
        if (!ok) {
            const uint64_t t0 = globaltimer_ns(), cap = max_polls(spin_ns);
            for (uint64_t it = 0; it < cap && !ok; ++it) {
                __nanosleep(64);
                a = ld16_volatile(lines + 2 * v);
                b = ld16_volatile(lines + 2 * v + 1);
                ok = a.y == step && a.w == step && b.y == step && b.w == step;
                if ((int64_t)(globaltimer_ns() - t0) > spin_ns) break;
            }
        }
        if (ok) {
            st16(dst + 4 * v, make_uint4(a.x, a.z, b.x, b.z));
        } else {
            const uint32_t d[4] = {a.x, a.z, b.x, b.z}, f[4] = {a.y, a.w, b.y, b.w};
            for (int j = 0; j < 4; ++j) {
                if (f[j] == step) dst[4 * v + j] = __uint_as_float(d[j]);
                else report_flag_timeout(st, rank, 4 * v + j);
            }
        }
    }
    pdl_release();
    if (blockIdx.x == gridDim.x - 1) {
        const size_t i = nq * 4 + threadIdx.x;
        if (i < count) {
            const uint2* line = reinterpret_cast<const uint2*>(lines) + i;
            uint2 x = *line;
            const uint64_t t0 = globaltimer_ns(), cap = max_polls(spin_ns);
            for (uint64_t it = 0; it < cap && x.y != step; ++it) {
                __nanosleep(64);
                x = ld8_volatile(line);
                if ((int64_t)(globaltimer_ns() - t0) > spin_ns) break;
            }
            if (x.y == step) dst[i] = __uint_as_float(x.x);
            else report_flag_timeout(st, rank, i);
        }
    }
}

// Two lines (16 B) per rank per thread.  A line is consumed only when all NR
// ranks' copies carry the step.  The flags are checked at warp level first:
// one vote over the warp's lanes decides whether any of them must poll, so
// the common case (every flag there) is a warp-uniform branch past the poll;
// measured on GB300 (n = 8 fp32, graph replay, A/B in one process pair) the
// 1 MiB LL pass ran 4% faster with the vote than with a per-thread branch.
// A lane whose lines lack a flag then polls its own lines (bounded).  A form
// in which the whole warp polled as one (lanes past the end idle, votes
// ending the poll) ran 0.2-0.45 us slower per pass and was not kept.
template <int NR>
__global__ void __launch_bounds__(kThreads)
ll_reduce_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t count, uint32_t step, int64_t spin_ns, DevStatus* st)
{
    pdl_acquire();
    const size_t np = (count + 1) / 2;  // 16-byte pairs of lines, the last one maybe half used
    const size_t bs = blockDim.x;
    for (size_t v = (size_t)blockIdx.x * bs + threadIdx.x; v < np; v += (size_t)gridDim.x * bs) {
        const bool two = 2 * v + 1 < count;
        uint4 x[NR];
#pragma unroll
        for (int q = 0; q < NR; ++q) {
            if (two) {
                x[q] = ld16(static_cast<const uint4*>(in.p[q]) + v);
            } else {
                const uint2 h = ld8(static_cast<const uint2*>(in.p[q]) + 2 * v);
                x[q] = make_uint4(h.x, h.y, 0u, step);
            }
        }
        bool ok0 = true, ok1 = true;
#pragma unroll
        for (int q = 0; q < NR; ++q) {
            ok0 = ok0 && x[q].y == step;
            ok1 = ok1 && x[q].w == step;
        }
        if (!__all_sync(__activemask(), ok0 && ok1) && !(ok0 && ok1)) {   // warp vote, then this lane
            const uint64_t t0 = globaltimer_ns(), cap = max_polls(spin_ns);
            for (uint64_t it = 0; it < cap && !(ok0 && ok1); ++it) {
                __nanosleep(64);
                ok0 = ok1 = true;
#pragma unroll
                for (int q = 0; q < NR; ++q) {
                    if (x[q].y != step || x[q].w != step) {
                        if (two) {
                            x[q] = ld16_volatile(static_cast<const uint4*>(in.p[q]) + v);
                        } else {
                            const uint2 h = ld8_volatile(static_cast<const uint2*>(in.p[q]) + 2 * v);
                            x[q] = make_uint4(h.x, h.y, 0u, step);
                        }
                    }
                    ok0 = ok0 && x[q].y == step;
                    ok1 = ok1 && x[q].w == step;
                }
                if ((int64_t)(globaltimer_ns() - t0) > spin_ns) break;
            }
        }
        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
        for (int q = 0; q < NR; ++q) {
            s0 = s0 + __uint_as_float(x[q].x);
            s1 = s1 + __uint_as_float(x[q].z);
        }
        const uint4 r = make_uint4(__float_as_uint(s0), step, __float_as_uint(s1), step);
        if (ok0 && ok1 && two) {
#pragma unroll
            for (int q = 0; q < NR; ++q) st16(static_cast<uint4*>(out.p[q]) + v, r);
        } else {
            if (ok0) {
#pragma unroll
                for (int q = 0; q < NR; ++q) st8(static_cast<uint2*>(out.p[q]) + 2 * v, make_uint2(r.x, r.y));
            }
            if (two && ok1) {
#pragma unroll
                for (int q = 0; q < NR; ++q) st8(static_cast<uint2*>(out.p[q]) + 2 * v + 1, make_uint2(r.z, r.w));
            }
            for (int q = 0; q < NR; ++q) {
                if (!ok0 && x[q].y != step) { report_flag_timeout(st, q, 2 * v); break; }
            }
            for (int q = 0; q < NR && two; ++q) {
                if (!ok1 && x[q].w != step) { report_flag_timeout(st, q, 2 * v + 1); break; }
            }
        }
    }
    pdl_release();
}

// -------------------------------------------------------------- LL128 ------
// Warp w handles lines 4w..4w+3 per iteration; lane l moves bytes
// 16 (l % 8) .. 16 (l % 8) + 15 of line 4w + l / 8.

struct Lane128 {
    size_t k;     // line index
    int j;        // 16-byte slot in the line, 0..7
    int leader;   // lane holding the group's flag (slot 7)
};

__device__ __forceinline__ Lane128 lane128(size_t kb)
{
    const int lane = threadIdx.x & 31;
    return Lane128{kb + (size_t)(lane >> 3), lane & 7, (lane & ~7) | 7};
}

__device__ __forceinline__ uint64_t group_flag(const uint4& v, int leader)
{
    const uint32_t lo = __shfl_sync(kFull, v.z, leader);
    const uint32_t hi = __shfl_sync(kFull, v.w, leader);
    return ((uint64_t)hi << 32) | lo;
}

__global__ void __launch_bounds__(kThreads)
ll128_pack_kernel(const __grid_constant__ SrcTable srcs, const __grid_constant__ DstTable outs, size_t count,
                  uint64_t step)
{
    pdl_acquire();
    const float* const src = static_cast<const float*>(srcs.p[blockIdx.y]);
    uint4* const lines = static_cast<uint4*>(outs.p[blockIdx.y]);
    const size_t L = (count + 29) / 30;
    const size_t warp = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
    for (size_t kb = warp * 4; kb < L; kb += nwarps * 4) {
        const Lane128 ln = lane128(kb);
        if (ln.k >= L) continue;
        const size_t e0 = 30 * ln.k + 4 * (size_t)ln.j;  // first payload word of this slot
        const int words = ln.j < 7 ? 4 : 2;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (30 * ln.k + 30 <= count) {
            const uint2 a = ld8(src + e0);
            w[0] = a.x;
            w[1] = a.y;
            if (words == 4) {
                const uint2 b = ld8(src + e0 + 2);
                w[2] = b.x;
                w[3] = b.y;
            }
        } else {
            for (int t = 0; t < words; ++t)
                if (e0 + t < count) w[t] = __float_as_uint(src[e0 + t]);
        }
        if (ln.j == 7) {
            w[2] = (uint32_t)step;
            w[3] = (uint32_t)(step >> 32);
        }
        st16(lines + 8 * ln.k + ln.j, make_uint4(w[0], w[1], w[2], w[3]));
    }
    pdl_release();
}

__global__ void __launch_bounds__(kThreads)
ll128_unpack_kernel(const __grid_constant__ SrcTable ins, const __grid_constant__ DstTable dsts, size_t count,
                    uint64_t step, int64_t spin_ns, DevStatus* st)
{
    pdl_acquire();
    const int rank = blockIdx.y;
    const uint4* const lines = static_cast<const uint4*>(ins.p[rank]);
    float* const dst = static_cast<float*>(dsts.p[rank]);
    const size_t L = (count + 29) / 30;
    const size_t warp = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
    for (size_t kb = warp * 4; kb < L; kb += nwarps * 4) {  // warp-uniform loop
        const Lane128 ln = lane128(kb);
        const bool active = ln.k < L;
        const uint4* p = lines + 8 * ln.k + ln.j;
        uint4 v = active ? ld16(p) : make_uint4(0u, 0u, 0u, 0u);
        const uint64_t f0 = group_flag(v, ln.leader);  // every lane shuffles
        bool ok = !active || f0 == step;
        if (!__all_sync(kFull, ok)) {
            const uint64_t t0 = globaltimer_ns(), cap = max_polls(spin_ns);
            for (uint64_t it = 0; it < cap; ++it) {
                __nanosleep(64);
                if (!ok) v = ld16_volatile(p);
                const uint64_t f = group_flag(v, ln.leader);
                ok = !active || f == step;
                const bool late = (int64_t)(globaltimer_ns() - t0) > spin_ns;
                if (__all_sync(kFull, ok) || __any_sync(kFull, late)) break;
            }
        }
        if (!active) continue;
        if (ok) {
            const size_t e0 = 30 * ln.k + 4 * (size_t)ln.j;
            const int words = ln.j < 7 ? 4 : 2;
            if (30 * ln.k + 30 <= count) {
                st8(dst + e0, make_uint2(v.x, v.y));
                if (words == 4) st8(dst + e0 + 2, make_uint2(v.z, v.w));
            } else {
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                for (int t = 0; t < words; ++t)
                    if (e0 + t < count) dst[e0 + t] = __uint_as_float(w[t]);
            }
        } else if (ln.j == 0) {
            report_flag_timeout(st, rank, ln.k);
        }
    }
    pdl_release();
}

template <int NR>
__global__ void __launch_bounds__(kThreads)
ll128_reduce_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out, size_t count, uint64_t step, int64_t spin_ns, DevStatus* st)
{
    pdl_acquire();
    const size_t L = (count + 29) / 30;
    const size_t warp = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
    for (size_t kb = warp * 4; kb < L; kb += nwarps * 4) {  // warp-uniform loop
        const Lane128 ln = lane128(kb);
        const bool active = ln.k < L;
        const size_t off = 8 * ln.k + ln.j;
        uint4 x[NR];
#pragma unroll
        for (int q = 0; q < NR; ++q)
            x[q] = active ? ld16(static_cast<const uint4*>(in.p[q]) + off) : make_uint4(0u, 0u, 0u, 0u);
        uint32_t bad = 0;  // bit q: rank q's copy lacks the flag
#pragma unroll
        for (int q = 0; q < NR; ++q) {
            const uint64_t f = group_flag(x[q], ln.leader);  // every lane shuffles
            if (active && f != step) bad |= 1u << q;
        }
        if (!__all_sync(kFull, bad == 0)) {
            const uint64_t t0 = globaltimer_ns(), cap = max_polls(spin_ns);
            for (uint64_t it = 0; it < cap; ++it) {
                __nanosleep(64);
                uint32_t now = 0;
#pragma unroll
                for (int q = 0; q < NR; ++q) {
                    if (bad & (1u << q)) x[q] = ld16_volatile(static_cast<const uint4*>(in.p[q]) + off);
                    const uint64_t f = group_flag(x[q], ln.leader);
                    if (active && f != step) now |= 1u << q;
                }
                bad = now;
                const bool late = (int64_t)(globaltimer_ns() - t0) > spin_ns;
                if (__all_sync(kFull, bad == 0) || __any_sync(kFull, late)) break;
            }
        }
        if (!active) continue;
        if (bad == 0) {
            float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int q = 0; q < NR; ++q) {
                a[0] = a[0] + __uint_as_float(x[q].x);
                a[1] = a[1] + __uint_as_float(x[q].y);
                a[2] = a[2] + __uint_as_float(x[q].z);
                a[3] = a[3] + __uint_as_float(x[q].w);
            }
            uint4 r = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                                 __float_as_uint(a[3]));
            if (ln.j == 7) {
                r.z = (uint32_t)step;
                r.w = (uint32_t)(step >> 32);
            }
#pragma unroll
            for (int q = 0; q < NR; ++q) st16(static_cast<uint4*>(out.p[q]) + off, r);
        } else if (ln.j == 0) {
            report_flag_timeout(st, __ffs(bad) - 1, ln.k);
        }
    }
    pdl_release();
}

}  // namespace

// Full CTAs for `work` thread-iterations in each of `rows` rows, or narrower
// ones when full CTAs would not give every SM one.  A row with less than one
// full CTA of work keeps its full CTA: measured on GB300 (n = 8 fp32
// payloads), the LL passes of 8-512 B ran up to 0.2 us slower narrowed, those
// of 4-256 KiB 0.1-0.4 us faster.
static Shape rows_shape(const Handle& h, size_t work, int rows)
{
    const unsigned g = grid_for_rows(h, work, rows);
    if (work < (size_t)kThreads || g * (unsigned)rows >= (unsigned)h.sm_count) return Shape{g, kThreads};
    return narrow_shape(h, work, rows);
}

// Tables of `nb` buffers (1 for the single-buffer calls, n for the batched ones).
static void tables(int nb, const void* const* src, void* const* dst, SrcTable& st, DstTable& dt)
{
    for (int i = 0; i < kMaxRanks; ++i) {
        st.p[i] = i < nb ? src[i] : nullptr;
        dt.p[i] = i < nb ? dst[i] : nullptr;
    }
}

int launch_ll_pack(Handle& h, int nb, const float* const* src, void* const* lines, size_t count, uint32_t step,
                   cudaStream_t s)
{
    SrcTable st;
    DstTable dt;
    tables(nb, reinterpret_cast<const void* const*>(src), lines, st, dt);
    const Shape sh = rows_shape(h, count / 4, nb);
    rec_begin(h, s);
    launch_kernel(h, ll_pack_kernel, dim3(sh.grid_x, nb), sh.block, 0, s, st, dt, count, step);
    rec_end(h, s, AR_K_LL_PACK, 12ull * count * nb);
    return launch_status();
}

int launch_ll_unpack(Handle& h, int nb, const void* const* lines, float* const* dst, size_t count, uint32_t step,
                     cudaStream_t s)
{
    SrcTable st;
    DstTable dt;
    tables(nb, lines, reinterpret_cast<void* const*>(dst), st, dt);
    const Shape sh = rows_shape(h, count / 4, nb);
    rec_begin(h, s);
    launch_kernel(h, ll_unpack_kernel, dim3(sh.grid_x, nb), sh.block, 0, s, st, dt, count, step, h.spin_ns,
                  h.status);
    rec_end(h, s, AR_K_LL_UNPACK, 12ull * count * nb);
    return launch_status();
}

int launch_ll_reduce(Handle& h, const void* const* in, void* const* out, size_t count, uint32_t step,
                     cudaStream_t s)
{
    return dispatch_ranks(h.n, [&](auto nrc) -> int {
        constexpr int NR = decltype(nrc)::value;
        CPtrs<NR> ip;
        MPtrs<NR> op;
        for (int q = 0; q < NR; ++q) {
            ip.p[q] = in[q];
            op.p[q] = out[q];
        }
        const Shape sh = rows_shape(h, (count + 1) / 2, 1);
        rec_begin(h, s);
        launch_kernel(h, ll_reduce_kernel<NR>, sh.grid_x, sh.block, 0, s, ip, op, count, step, h.spin_ns, h.status);
        rec_end(h, s, AR_K_LL_REDUCE, 16ull * NR * count);
        return launch_status();
    });
}

int launch_ll128_pack(Handle& h, int nb, const float* const* src, void* const* lines, size_t count, uint64_t step,
                      cudaStream_t s)
{
    SrcTable st;
    DstTable dt;
    tables(nb, reinterpret_cast<const void* const*>(src), lines, st, dt);
    const size_t L = (count + 29) / 30;
    const Shape sh = rows_shape(h, L * 8, nb);
    rec_begin(h, s);
    launch_kernel(h, ll128_pack_kernel, dim3(sh.grid_x, nb), sh.block, 0, s, st, dt, count, step);
    rec_end(h, s, AR_K_LL128_PACK, (4ull * count + 128ull * L) * nb);
    return launch_status();
}

int launch_ll128_unpack(Handle& h, int nb, const void* const* lines, float* const* dst, size_t count,
                        uint64_t step, cudaStream_t s)
{
    SrcTable st;
    DstTable dt;
    tables(nb, lines, reinterpret_cast<void* const*>(dst), st, dt);
    const size_t L = (count + 29) / 30;
    const Shape sh = rows_shape(h, L * 8, nb);
    rec_begin(h, s);
    launch_kernel(h, ll128_unpack_kernel, dim3(sh.grid_x, nb), sh.block, 0, s, st, dt, count, step, h.spin_ns,
                  h.status);
    rec_end(h, s, AR_K_LL128_UNPACK, (4ull * count + 128ull * L) * nb);
    return launch_status();
}

int launch_ll128_reduce(Handle& h, const void* const* in, void* const* out, size_t count, uint64_t step,
                        cudaStream_t s)
{
    return dispatch_ranks(h.n, [&](auto nrc) -> int {
        constexpr int NR = decltype(nrc)::value;
        CPtrs<NR> ip;
        MPtrs<NR> op;
        for (int q = 0; q < NR; ++q) {
            ip.p[q] = in[q];
            op.p[q] = out[q];
        }
        const size_t L = (count + 29) / 30;
        const Shape sh = rows_shape(h, L * 8, 1);
        rec_begin(h, s);
        launch_kernel(h, ll128_reduce_kernel<NR>, sh.grid_x, sh.block, 0, s, ip, op, count, step, h.spin_ns,
                      h.status);
        rec_end(h, s, AR_K_LL128_REDUCE, 256ull * NR * L);
        return launch_status();
    });
}

}  // namespace argb
