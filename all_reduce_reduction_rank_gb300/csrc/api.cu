// C-ABI entry points of libar_gb300.so (declared in include/ar.h): handle
// life cycle, argument checks, the traffic plan, the sticky status word and
// the calls that launch the kernels of one_shot.cu, two_shot.cu, ring.cu and
// ll.cu.  Host code only; nothing here allocates after ar_create.
#include <climits>
#include <cmath>
#include <cstring>
#include <new>

#include "common.cuh"

using namespace argb;

namespace {

constexpr uint32_t kMagic = 0x41524742u;  // "ARGB"

bool is_ll_op(int op) { return op == AR_OP_LL_REDUCE || op == AR_OP_LL128_REDUCE; }

size_t ll128_lines(size_t count) { return (count + 29u) / 30u; }

// Bytes of one rank's buffer that a call touches.
size_t buffer_bytes(int op, size_t count, int dt)
{
    switch (op) {
    case AR_OP_LL_PACK:
    case AR_OP_LL_UNPACK:
    case AR_OP_LL_REDUCE: return 8u * count;
    case AR_OP_LL128_PACK:
    case AR_OP_LL128_UNPACK:
    case AR_OP_LL128_REDUCE: return 128u * ll128_lines(count);
    default: return count * elem_bytes(dt);
    }
}

bool overlap(const void* a, const void* b, size_t bytes)
{
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return bytes && x < y + bytes && y < x + bytes;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// [a, a + an) and [b, b + bn) intersect.
bool overlap_sized(const void* a, size_t an, const void* b, size_t bn)
{
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return an && bn && x < y + bn && y < x + an;
}

int check_size(size_t count, int dt, size_t max_bytes)
{
    const size_t e = elem_bytes(dt);
    if (count > SIZE_MAX / 128u) return AR_ERR_TOO_LARGE;
    if (count * e > max_bytes) return AR_ERR_TOO_LARGE;
    return AR_OK;
}

// Checks shared by every multi-rank call, in this order: n and dtype,
// NULL pointers, size, alignment, overlap.
int check_multi(int op, int n, size_t max_bytes, const void* const* in, void* const* out, size_t count, int dt)
{
    if (n < 2 || n > kMaxRanks) return AR_ERR_INVALID;
    if (dt != AR_F32 && dt != AR_BF16 && dt != AR_F16) return AR_ERR_INVALID;
    if (is_ll_op(op) && dt != AR_F32) return AR_ERR_INVALID;
    if ((op == AR_OP_TREE || op == AR_OP_TREE_FUSED) && (n & (n - 1))) return AR_ERR_INVALID;
    if (!in || !out) return AR_ERR_INVALID;
    for (int r = 0; r < n; ++r)
        if (!in[r] || !out[r]) return AR_ERR_INVALID;
    if (int rc = check_size(count, dt, max_bytes)) return rc;
    for (int r = 0; r < n; ++r)
        if (!aligned16(in[r]) || !aligned16(out[r])) return AR_ERR_ALIGN;
    const size_t bytes = buffer_bytes(op, count, dt);
    for (int r = 0; r < n; ++r) {
        if (out[r] != in[r] && overlap(out[r], in[r], bytes)) return AR_ERR_INVALID;
        for (int q = 0; q < n; ++q) {
            if (q == r) continue;
            if (overlap(out[r], out[q], bytes) || overlap(out[r], in[q], bytes)) return AR_ERR_INVALID;
        }
    }
    return AR_OK;
}

// Checks of the single-buffer pack / unpack calls.
int check_single(int op, size_t max_bytes, const void* src, const void* dst, size_t count)
{
    if (!src || !dst) return AR_ERR_INVALID;
    if (int rc = check_size(count, AR_F32, max_bytes)) return rc;
    if (!aligned16(src) || !aligned16(dst)) return AR_ERR_ALIGN;
    const size_t lines = buffer_bytes(op, count, AR_F32), payload = 4u * count;
    const uintptr_t s = (uintptr_t)src, d = (uintptr_t)dst;
    const bool src_is_lines = (op == AR_OP_LL_UNPACK || op == AR_OP_LL128_UNPACK);
    const size_t sb = src_is_lines ? lines : payload, db = src_is_lines ? payload : lines;
    if (count && s < d + db && d < s + sb) return AR_ERR_INVALID;
    return AR_OK;
}

// Checks of the rank-batched pack / unpack calls: n sources and n
// destinations of different sizes (payload vs lines); sources may alias.
int check_batch(int op, int n, size_t max_bytes, const void* const* src, const void* const* dst, size_t count)
{
    if (!src || !dst) return AR_ERR_INVALID;
    for (int r = 0; r < n; ++r)
        if (!src[r] || !dst[r]) return AR_ERR_INVALID;
    if (int rc = check_size(count, AR_F32, max_bytes)) return rc;
    for (int r = 0; r < n; ++r)
        if (!aligned16(src[r]) || !aligned16(dst[r])) return AR_ERR_ALIGN;
    const size_t lines = buffer_bytes(op, count, AR_F32), payload = 4u * count;
    const bool src_is_lines = (op == AR_OP_LL_UNPACK || op == AR_OP_LL128_UNPACK);
    const size_t sb = src_is_lines ? lines : payload, db = src_is_lines ? payload : lines;
    if (!count) return AR_OK;
    for (int r = 0; r < n; ++r) {
        for (int q = 0; q < n; ++q) {
            const uintptr_t s = (uintptr_t)src[q], d = (uintptr_t)dst[r];
            if (s < d + db && d < s + sb) return AR_ERR_INVALID;
            if (q != r && overlap(dst[r], dst[q], db)) return AR_ERR_INVALID;
        }
    }
    return AR_OK;
}

void plan(int op, int n, size_t count, int dt, ar_traffic_t* t)
{
    std::memset(t, 0, sizeof(*t));
    t->op = op;
    t->n_ranks = n;
    t->count = count;
    const bool ll = op >= AR_OP_LL_PACK && op <= AR_OP_LL128_REDUCE;  // fp32 payload words
    t->elem_bytes = ll ? 4u : elem_bytes(dt);
    const uint64_t e = t->elem_bytes, N = count, S = N * e, nn = (uint64_t)n;
    const uint64_t L = ll128_lines(count);
    switch (op) {
    case AR_OP_ONE_SHOT:
        t->link_bytes_per_rank = (double)(nn - 1) * (double)S;
        t->steps = 1;
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = nn * S;
        t->hbm_write_bytes = nn * S;
        break;
    case AR_OP_TWO_SHOT:
        // rank r reads (n-1) |chunk r| in phase 1 and S - |chunk r| in phase 2;
        // summed over ranks that is 2 (n-1) S for any chunking.
        t->link_bytes_per_rank = 2.0 * (double)(nn - 1) * (double)S / (double)nn;
        t->steps = 2;
        t->launches = count ? (two_shot_one_launch(0) ? 1 : 2) : 0;  // the default form's launches
        t->hbm_read_bytes = (nn + 1) * S;
        t->hbm_write_bytes = nn * S;
        break;
    case AR_OP_RING:
        // every step moves each chunk once: (n-1) N e per phase over all ranks
        t->link_bytes_per_rank = 2.0 * (double)(nn - 1) * (double)S / (double)nn;
        t->steps = 2 * (n - 1);
        t->launches = count ? 2 * (n - 1) : 0;
        if (n == 2) {
            t->hbm_read_bytes = 3 * e * N;
            t->hbm_write_bytes = 2 * e * N;
        } else {
            t->hbm_read_bytes = 2 * e * N + (nn - 2) * (4 + e) * N + (nn - 1) * e * N;
            t->hbm_write_bytes = (nn - 2) * 4 * N + e * N + (nn - 1) * e * N;
        }
        break;
    case AR_OP_LL_PACK:
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = nn * 4 * N;
        t->hbm_write_bytes = nn * 8 * N;
        break;
    case AR_OP_LL_UNPACK:
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = nn * 8 * N;
        t->hbm_write_bytes = nn * 4 * N;
        break;
    case AR_OP_LL_REDUCE:
        t->steps = 1;
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = nn * 8 * N;
        t->hbm_write_bytes = nn * 8 * N;
        break;
    case AR_OP_LL128_PACK:
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = nn * 4 * N;
        t->hbm_write_bytes = nn * 128 * L;
        break;
    case AR_OP_LL128_UNPACK:
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = nn * 128 * L;
        t->hbm_write_bytes = nn * 4 * N;
        break;
    case AR_OP_RING_ROUNDED:
        t->link_bytes_per_rank = 2.0 * (double)(nn - 1) * (double)S / (double)nn;
        t->steps = 2 * (n - 1);
        t->launches = count ? 2 * (n - 1) : 0;
        t->hbm_read_bytes = 2 * e * N * (nn - 1) + e * N * (nn - 1);
        t->hbm_write_bytes = e * N * (nn - 1) + e * N * (nn - 1);
        break;
    case AR_OP_TREE: {
        int levels = 0;
        while ((1 << levels) < n) ++levels;
        t->link_bytes_per_rank = (double)levels * (double)S;   // the peer's buffer, once per level
        t->steps = levels;
        t->launches = count ? levels : 0;
        t->hbm_read_bytes = (uint64_t)levels * nn * S;
        t->hbm_write_bytes = (uint64_t)levels * nn * S;
        break;
    }
    case AR_OP_RING_PERSISTENT: {
        const uint64_t lines = persist_lines_per_step(n, count, dt);
        t->link_bytes_per_rank = 2.0 * (double)(nn - 1) * (double)S / (double)nn;
        t->steps = 2 * (n - 1);
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = nn * S + (2 * nn - 2) * 128 * lines;
        t->hbm_write_bytes = nn * S + (2 * nn - 2) * 128 * lines;
        break;
    }
    case AR_OP_TREE_FUSED: {
        int levels = 0;
        while ((1 << levels) < n) ++levels;
        t->link_bytes_per_rank = (double)levels * (double)S;
        t->steps = levels;
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = nn * S;
        t->hbm_write_bytes = nn * S;
        break;
    }
    case AR_OP_RING_CLUSTER:
    case AR_OP_RING_FUSED:
    case AR_OP_RING_ROUNDED_FUSED:
        t->link_bytes_per_rank = 2.0 * (double)(nn - 1) * (double)S / (double)nn;
        t->steps = 2 * (n - 1);
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = nn * S;
        t->hbm_write_bytes = nn * S;
        break;
    case AR_OP_ONE_SHOT_PUSH:
        t->link_bytes_per_rank = (double)(nn - 1) * (double)S;  // pushed to the peers
        t->steps = 1;
        t->launches = count ? 2 : 0;
        t->hbm_read_bytes = nn * S + nn * nn * S;
        t->hbm_write_bytes = nn * (nn - 1) * S + nn * S;
        break;
    case AR_OP_ONE_SHOT_COPYIN:
        t->link_bytes_per_rank = (double)(nn - 1) * (double)S;
        t->steps = 1;
        t->launches = count ? 2 : 0;
        t->hbm_read_bytes = 2 * nn * S;
        t->hbm_write_bytes = 2 * nn * S;
        break;
    case AR_OP_ALLREDUCE_RMSNORM:
        t->link_bytes_per_rank = (double)(nn - 1) * (double)S;
        t->steps = 1;
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = (nn + 1) * S;
        t->hbm_write_bytes = (nn + 1) * S;
        break;
    case AR_OP_LL128_REDUCE:
        t->steps = 1;
        t->launches = count ? 1 : 0;
        t->hbm_read_bytes = nn * 128 * L;
        t->hbm_write_bytes = nn * 128 * L;
        break;
    default: break;
    }
}

// Runs a launch on the handle's device, restoring the caller's device after.
template <typename F>
int on_device(const Handle& h, F&& f)
{
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return AR_ERR_CUDA;
    if (cur != h.device && cudaSetDevice(h.device) != cudaSuccess) return AR_ERR_CUDA;
    const int rc = f();
    if (cur != h.device) cudaSetDevice(cur);
    return rc;
}

void free_timing(Timing& t)
{
    for (cudaEvent_t e : t.start) cudaEventDestroy(e);
    for (cudaEvent_t e : t.stop) cudaEventDestroy(e);
    t.start.clear();
    t.stop.clear();
    t.rec.clear();
    t.capacity = 0;
    t.head = t.count = 0;
}

int make_timing(Timing& t, int capacity)
{
    free_timing(t);
    if (capacity == 0) return AR_OK;
    t.start.assign((size_t)capacity, nullptr);
    t.stop.assign((size_t)capacity, nullptr);
    t.rec.assign((size_t)capacity, ar_launch_time_t{});
    for (int i = 0; i < capacity; ++i) {
        if (cudaEventCreate(&t.start[i]) != cudaSuccess || cudaEventCreate(&t.stop[i]) != cudaSuccess) {
            cudaGetLastError();
            t.capacity = capacity;  // so free_timing destroys what was made
            free_timing(t);
            return AR_ERR_CUDA;
        }
    }
    t.capacity = capacity;
    return AR_OK;
}

}  // namespace

struct ar_ctx {
    uint32_t magic;
    Handle h;
};

static Handle* get(ar_handle hd)
{
    return (hd && hd->magic == kMagic) ? &hd->h : nullptr;
}

typedef int (*multi_launcher)(Handle&, const void* const*, void* const*, size_t, int, cudaStream_t, int*);

static int all_reduce_call(int op, multi_launcher fn, ar_handle hd, const void* const* in, void* const* out,
                           size_t count, ar_dtype dt, ar_stream_t stream)
{
    Handle* h = get(hd);
    if (!h) return AR_ERR_INVALID;
    if (int rc = check_multi(op, h->n, h->max_bytes, in, out, count, dt)) return rc;
    int launches = 0;
    int rc = AR_OK;
    h->timing.op = op;
    if (count) rc = on_device(*h, [&] { return fn(*h, in, out, count, dt, (cudaStream_t)stream, &launches); });
    if (rc != AR_OK) return rc;
    plan(op, h->n, count, dt, &h->last);
    h->last.launches = launches;
    h->last_stream = (cudaStream_t)stream;
    return AR_OK;
}

template <typename F>
static int single_call(int op, ar_handle hd, const void* src, const void* dst, size_t count, uint64_t step,
                       ar_stream_t stream, F&& launch)
{
    Handle* h = get(hd);
    if (!h) return AR_ERR_INVALID;
    if (step == 0) return AR_ERR_INVALID;
    if (int rc = check_single(op, h->max_bytes, src, dst, count)) return rc;
    int rc = AR_OK;
    h->timing.op = op;
    if (count) rc = on_device(*h, [&] { return launch(*h, (cudaStream_t)stream); });
    if (rc != AR_OK) return rc;
    plan(op, 1, count, AR_F32, &h->last);
    h->last_stream = (cudaStream_t)stream;
    return AR_OK;
}

template <typename F>
static int batch_call(int op, ar_handle hd, const void* const* src, const void* const* dst, size_t count,
                      uint64_t step, ar_stream_t stream, F&& launch)
{
    Handle* h = get(hd);
    if (!h) return AR_ERR_INVALID;
    if (step == 0) return AR_ERR_INVALID;
    if (int rc = check_batch(op, h->n, h->max_bytes, src, dst, count)) return rc;
    int rc = AR_OK;
    h->timing.op = op;
    if (count) rc = on_device(*h, [&] { return launch(*h, (cudaStream_t)stream); });
    if (rc != AR_OK) return rc;
    plan(op, h->n, count, AR_F32, &h->last);
    h->last_stream = (cudaStream_t)stream;
    return AR_OK;
}

template <typename F>
static int reduce_call(int op, ar_handle hd, const void* const* in, void* const* out, size_t count, uint64_t step,
                       ar_stream_t stream, F&& launch)
{
    Handle* h = get(hd);
    if (!h) return AR_ERR_INVALID;
    if (step == 0) return AR_ERR_INVALID;
    if (int rc = check_multi(op, h->n, h->max_bytes, in, out, count, AR_F32)) return rc;
    int rc = AR_OK;
    h->timing.op = op;
    if (count) rc = on_device(*h, [&] { return launch(*h, (cudaStream_t)stream); });
    if (rc != AR_OK) return rc;
    plan(op, h->n, count, AR_F32, &h->last);
    h->last_stream = (cudaStream_t)stream;
    return AR_OK;
}

extern "C" {

const char* ar_strerror(int code)
{
    switch (code) {
    case AR_OK: return "ok";
    case AR_ERR_INVALID: return "invalid argument";
    case AR_ERR_ALIGN: return "pointer not 16-byte aligned";
    case AR_ERR_TOO_LARGE: return "count x element size exceeds max_bytes";
    case AR_ERR_CUDA: return "CUDA runtime error";
    case AR_ERR_FLAG_TIMEOUT: return "LL/LL128 flag not seen within the spin limit";
    case AR_ERR_WAIT_TIMEOUT: return "a kernel's bounded wait (its bulk copies, or a peer freeing a slot) ran out";
    default: return "unknown error code";
    }
}

size_t ar_ll_bytes(size_t payload_bytes) { return 2u * ((payload_bytes + 3u) / 4u * 4u); }

size_t ar_ll128_bytes(size_t payload_bytes) { return 128u * ((payload_bytes + 119u) / 120u); }

int ar_plan(int op, int n_ranks, size_t count, ar_dtype dt, ar_traffic_t* t)
{
    if (!t || op < AR_OP_ONE_SHOT || op > AR_OP_RING_ROUNDED_FUSED) return AR_ERR_INVALID;
    const bool multi =
        op <= AR_OP_RING || op == AR_OP_LL_REDUCE || op == AR_OP_LL128_REDUCE || op >= AR_OP_ALLREDUCE_RMSNORM;
    if (multi && (n_ranks < 2 || n_ranks > kMaxRanks)) return AR_ERR_INVALID;
    if ((op == AR_OP_TREE || op == AR_OP_TREE_FUSED) && (n_ranks & (n_ranks - 1))) return AR_ERR_INVALID;
    if (!multi && (n_ranks < 1 || n_ranks > kMaxRanks)) return AR_ERR_INVALID;  // buffers packed
    if (dt != AR_F32 && dt != AR_BF16 && dt != AR_F16) return AR_ERR_INVALID;
    plan(op, n_ranks, count, dt, t);
    return AR_OK;
}

int ar_check_args(int op, int n_ranks, size_t max_bytes, const void* const* in, void* const* out, size_t count,
                  ar_dtype dt)
{
    if (op == AR_OP_LL_PACK || op == AR_OP_LL_UNPACK || op == AR_OP_LL128_PACK || op == AR_OP_LL128_UNPACK) {
        if (n_ranks < 1 || n_ranks > kMaxRanks || dt != AR_F32) return AR_ERR_INVALID;
        return check_batch(op, n_ranks, max_bytes, in, out, count);
    }
    if (op != AR_OP_ONE_SHOT && op != AR_OP_TWO_SHOT && op != AR_OP_RING && op != AR_OP_ONE_SHOT_PUSH &&
        op != AR_OP_ONE_SHOT_COPYIN && op != AR_OP_RING_ROUNDED && op != AR_OP_TREE &&
        op != AR_OP_RING_PERSISTENT && op != AR_OP_RING_CLUSTER && op != AR_OP_TREE_FUSED &&
        op != AR_OP_RING_FUSED && op != AR_OP_RING_ROUNDED_FUSED && !is_ll_op(op))
        return AR_ERR_INVALID;
    return check_multi(op, n_ranks, max_bytes, in, out, count, dt);
}

int ar_create(int n_ranks, size_t max_bytes, ar_handle* out)
{
    if (!out || n_ranks < 2 || n_ranks > kMaxRanks || max_bytes < 16) return AR_ERR_INVALID;
    ar_ctx* c = new (std::nothrow) ar_ctx();
    if (!c) return AR_ERR_INVALID;
    c->magic = kMagic;
    Handle& h = c->h;
    h.n = n_ranks;
    h.max_bytes = max_bytes;
    int rc = AR_OK;
    if (cudaGetDevice(&h.device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h.sm_count, cudaDevAttrMultiProcessorCount, h.device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h.l2_bytes, cudaDevAttrL2CacheSize, h.device) != cudaSuccess)
        rc = AR_ERR_CUDA;
    // ring scratch: the largest chunk over the payload types
    size_t cmax = 0;
    for (int dt = AR_F32; dt <= AR_F16; ++dt) {
        const size_t c_dt = chunk_elems(n_ranks, max_bytes / elem_bytes(dt), dt);
        if (c_dt > cmax) cmax = c_dt;
    }
    h.ring_chunk_max = cmax;
    h.stage_slot = (max_bytes + 255u) / 256u * 256u;
    if (rc == AR_OK && cudaMalloc(&h.ring_scratch, 2u * (size_t)n_ranks * cmax * sizeof(float)) != cudaSuccess)
        rc = AR_ERR_CUDA;
    if (rc == AR_OK && cudaMalloc(&h.status, sizeof(DevStatus)) != cudaSuccess) rc = AR_ERR_CUDA;
    if (rc == AR_OK && cudaMemset(h.status, 0, sizeof(DevStatus)) != cudaSuccess) rc = AR_ERR_CUDA;
    // the one-launch two-shot's counters and tile flags: zero, so no flag matches a call's epoch (>= 1)
    h.two_shot_sync_words = two_shot_sync_words(n_ranks, max_bytes);
    if (rc == AR_OK && cudaMalloc(&h.two_shot_sync, h.two_shot_sync_words * sizeof(unsigned)) != cudaSuccess)
        rc = AR_ERR_CUDA;
    if (rc == AR_OK && cudaMemset(h.two_shot_sync, 0, h.two_shot_sync_words * sizeof(unsigned)) != cudaSuccess)
        rc = AR_ERR_CUDA;
    if (rc == AR_OK && (cudaStreamCreateWithFlags(&h.side, cudaStreamNonBlocking) != cudaSuccess ||
                        cudaEventCreateWithFlags(&h.ev_fork, cudaEventDisableTiming) != cudaSuccess ||
                        cudaEventCreateWithFlags(&h.ev_join, cudaEventDisableTiming) != cudaSuccess))
        rc = AR_ERR_CUDA;
    if (rc == AR_OK && cudaDeviceSynchronize() != cudaSuccess) rc = AR_ERR_CUDA;
    if (rc != AR_OK) {
        if (h.ring_scratch) cudaFree(h.ring_scratch);
        if (h.status) cudaFree(h.status);
        if (h.two_shot_sync) cudaFree(h.two_shot_sync);
        if (h.side) cudaStreamDestroy(h.side);
        if (h.ev_fork) cudaEventDestroy(h.ev_fork);
        if (h.ev_join) cudaEventDestroy(h.ev_join);
        cudaGetLastError();
        c->magic = 0;
        delete c;
        return rc;
    }
    *out = c;
    return AR_OK;
}

int ar_destroy(ar_handle hd)
{
    Handle* h = get(hd);
    if (!h) return AR_ERR_INVALID;
    int rc = on_device(*h, [&] {
        int r = cudaDeviceSynchronize() == cudaSuccess ? AR_OK : AR_ERR_CUDA;
        if (cudaFree(h->ring_scratch) != cudaSuccess) r = AR_ERR_CUDA;
        if (cudaFree(h->status) != cudaSuccess) r = AR_ERR_CUDA;
        if (cudaFree(h->two_shot_sync) != cudaSuccess) r = AR_ERR_CUDA;
        if (h->push_stage && cudaFree(h->push_stage) != cudaSuccess) r = AR_ERR_CUDA;
        if (h->registered && cudaFree(h->registered) != cudaSuccess) r = AR_ERR_CUDA;
        if (h->persist && cudaFree(h->persist) != cudaSuccess) r = AR_ERR_CUDA;
        if (cudaStreamDestroy(h->side) != cudaSuccess) r = AR_ERR_CUDA;
        if (cudaEventDestroy(h->ev_fork) != cudaSuccess) r = AR_ERR_CUDA;
        if (cudaEventDestroy(h->ev_join) != cudaSuccess) r = AR_ERR_CUDA;
        free_timing(h->timing);
        return r;
    });
    hd->magic = 0;
    delete hd;
    return rc;
}

int ar_set_option(ar_handle hd, int option, int64_t value)
{
    Handle* h = get(hd);
    if (!h) return AR_ERR_INVALID;
    switch (option) {
    case AR_OPT_CTAS_PER_SM:
        if (value < 0 || value > 1024) return AR_ERR_INVALID;
        h->ctas_per_sm = (int)value;
        return AR_OK;
    case AR_OPT_SPIN_NS:
        if (value < 1 || value > 10000000000LL) return AR_ERR_INVALID;
        h->spin_ns = value;
        return AR_OK;
    case AR_OPT_ONE_SHOT_IMPL:
        if (value < 0 || value > 2) return AR_ERR_INVALID;
        h->one_shot_impl = (int)value;
        return AR_OK;
    case AR_OPT_TWO_SHOT_IMPL:
        if (value < 0 || value > 3) return AR_ERR_INVALID;
        h->two_shot_impl = (int)value;
        return AR_OK;
    case AR_OPT_AUTO_POLICY:
        if (value != AR_AUTO_MODEL && value != AR_AUTO_EMULATED) return AR_ERR_INVALID;
        h->auto_policy = (int)value;
        return AR_OK;
    case AR_OPT_AUTO_ALPHA_NS:
        if (value < 0 || value > 1000000000LL) return AR_ERR_INVALID;
        h->auto_alpha_ns = value;
        return AR_OK;
    case AR_OPT_AUTO_BETA_MBS:
        if (value < 1 || value > 1000000000LL) return AR_ERR_INVALID;
        h->auto_beta_mbs = value;
        return AR_OK;
    case AR_OPT_AUTO_HANDOFF:
        if (value < 0) return AR_ERR_INVALID;
        h->auto_handoff = value;
        return AR_OK;
    case AR_OPT_PUSH_STAGING:
    case AR_OPT_REGISTERED: {
        if (value != 0 && value != 1) return AR_ERR_INVALID;
        uint8_t** buf = option == AR_OPT_PUSH_STAGING ? &h->push_stage : &h->registered;
        const size_t bytes = (option == AR_OPT_PUSH_STAGING ? (size_t)h->n * h->n : (size_t)h->n) * h->stage_slot;
        return on_device(*h, [&] {
            if (cudaDeviceSynchronize() != cudaSuccess) return (int)AR_ERR_CUDA;
            if (*buf) {
                cudaFree(*buf);
                *buf = nullptr;
            }
            if (value == 1 && cudaMalloc(reinterpret_cast<void**>(buf), bytes) != cudaSuccess) {
                cudaGetLastError();
                *buf = nullptr;
                return (int)AR_ERR_CUDA;
            }
            return (int)AR_OK;
        });
    }
    case AR_OPT_PERSISTENT:
        if (value != 0 && value != 1) return AR_ERR_INVALID;
        return on_device(*h, [&] {
            if (cudaDeviceSynchronize() != cudaSuccess) return (int)AR_ERR_CUDA;
            if (h->persist) {
                cudaFree(h->persist);
                h->persist = nullptr;
            }
            if (value == 0) return (int)AR_OK;
            const size_t bytes = persist_bytes(h->n, h->max_bytes, h->sm_count);
            // zeroed: no flag, acknowledgement or abort word of a call matches 0
            if (cudaMalloc(reinterpret_cast<void**>(&h->persist), bytes) != cudaSuccess ||
                cudaMemset(h->persist, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
                cudaGetLastError();
                if (h->persist) cudaFree(h->persist);
                h->persist = nullptr;
                return (int)AR_ERR_CUDA;
            }
            return (int)AR_OK;
        });
    case AR_OPT_ABSENT_RANK:
        if (value < -1 || value >= h->n) return AR_ERR_INVALID;
        h->persist_absent = (int)value;
        return AR_OK;
    case AR_OPT_PDL:
        if (value < 0 || value > 1) return AR_ERR_INVALID;
        h->pdl = (int)value;
        return AR_OK;
    case AR_OPT_TIMING_PAUSE:
        if (value < 0 || value > 1 || h->timing.capacity == 0) return AR_ERR_INVALID;
        h->timing.paused = (int)value;
        return AR_OK;
    case AR_OPT_TIMING:
        if (value < 0 || value > (1 << 20)) return AR_ERR_INVALID;
        return on_device(*h, [&] {
            if (cudaDeviceSynchronize() != cudaSuccess) return (int)AR_ERR_CUDA;
            return make_timing(h->timing, (int)value);
        });
    default: return AR_ERR_INVALID;
    }
}

int ar_one_shot(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt, ar_stream_t s)
{
    return all_reduce_call(AR_OP_ONE_SHOT, launch_one_shot, h, in, out, count, dt, s);
}

int ar_tree_fused(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt, ar_stream_t s)
{
    return all_reduce_call(AR_OP_TREE_FUSED, launch_tree_fused, h, in, out, count, dt, s);
}

int ar_ring_cluster(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt, ar_stream_t s)
{
    return all_reduce_call(AR_OP_RING_CLUSTER, launch_ring_cluster, h, in, out, count, dt, s);
}

int ar_ring_fused(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt, ar_stream_t s)
{
    return all_reduce_call(AR_OP_RING_FUSED, launch_ring_fused, h, in, out, count, dt, s);
}

int ar_ring_rounded_fused(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                          ar_stream_t s)
{
    return all_reduce_call(AR_OP_RING_ROUNDED_FUSED, launch_ring_rounded_fused, h, in, out, count, dt, s);
}

int ar_one_shot_push(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                     ar_stream_t s)
{
    Handle* hh = get(h);
    if (!hh || !hh->push_stage) return AR_ERR_INVALID;
    return all_reduce_call(AR_OP_ONE_SHOT_PUSH, launch_one_shot_push, h, in, out, count, dt, s);
}

int ar_one_shot_copyin(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                       ar_stream_t s)
{
    Handle* hh = get(h);
    if (!hh || !hh->registered) return AR_ERR_INVALID;
    return all_reduce_call(AR_OP_ONE_SHOT_COPYIN, launch_one_shot_copyin, h, in, out, count, dt, s);
}

int ar_ring_rounded(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt, ar_stream_t s)
{
    return all_reduce_call(AR_OP_RING_ROUNDED, launch_ring_rounded, h, in, out, count, dt, s);
}

int ar_tree(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt, ar_stream_t s)
{
    return all_reduce_call(AR_OP_TREE, launch_tree, h, in, out, count, dt, s);
}

int ar_ring_persistent(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                       ar_stream_t s)
{
    Handle* hh = get(h);
    if (!hh || !hh->persist) return AR_ERR_INVALID;
    return all_reduce_call(AR_OP_RING_PERSISTENT, launch_ring_persistent, h, in, out, count, dt, s);
}

int ar_two_shot(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt, ar_stream_t s)
{
    return all_reduce_call(AR_OP_TWO_SHOT, launch_two_shot, h, in, out, count, dt, s);
}

int ar_ring(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt, ar_stream_t s)
{
    return all_reduce_call(AR_OP_RING, launch_ring, h, in, out, count, dt, s);
}

int ar_ll_pack(ar_handle h, const float* src, void* lines, size_t count, uint32_t step, ar_stream_t s)
{
    return single_call(AR_OP_LL_PACK, h, src, lines, count, step, s, [&](Handle& hh, cudaStream_t st) {
        return launch_ll_pack(hh, 1, &src, &lines, count, step, st);
    });
}

int ar_ll_unpack(ar_handle h, const void* lines, float* dst, size_t count, uint32_t step, ar_stream_t s)
{
    return single_call(AR_OP_LL_UNPACK, h, lines, dst, count, step, s, [&](Handle& hh, cudaStream_t st) {
        return launch_ll_unpack(hh, 1, &lines, &dst, count, step, st);
    });
}

int ar_ll128_pack(ar_handle h, const float* src, void* lines, size_t count, uint64_t step, ar_stream_t s)
{
    return single_call(AR_OP_LL128_PACK, h, src, lines, count, step, s, [&](Handle& hh, cudaStream_t st) {
        return launch_ll128_pack(hh, 1, &src, &lines, count, step, st);
    });
}

int ar_ll128_unpack(ar_handle h, const void* lines, float* dst, size_t count, uint64_t step, ar_stream_t s)
{
    return single_call(AR_OP_LL128_UNPACK, h, lines, dst, count, step, s, [&](Handle& hh, cudaStream_t st) {
        return launch_ll128_unpack(hh, 1, &lines, &dst, count, step, st);
    });
}

int ar_ll_pack_n(ar_handle h, const float* const* src, void* const* lines, size_t count, uint32_t step,
                 ar_stream_t s)
{
    return batch_call(AR_OP_LL_PACK, h, reinterpret_cast<const void* const*>(src), lines, count, step, s,
                      [&](Handle& hh, cudaStream_t st) { return launch_ll_pack(hh, hh.n, src, lines, count, step, st); });
}

int ar_ll_unpack_n(ar_handle h, const void* const* lines, float* const* dst, size_t count, uint32_t step,
                   ar_stream_t s)
{
    return batch_call(AR_OP_LL_UNPACK, h, lines, reinterpret_cast<const void* const*>(dst), count, step, s,
                      [&](Handle& hh, cudaStream_t st) { return launch_ll_unpack(hh, hh.n, lines, dst, count, step, st); });
}

int ar_ll128_pack_n(ar_handle h, const float* const* src, void* const* lines, size_t count, uint64_t step,
                    ar_stream_t s)
{
    return batch_call(AR_OP_LL128_PACK, h, reinterpret_cast<const void* const*>(src), lines, count, step, s,
                      [&](Handle& hh, cudaStream_t st) { return launch_ll128_pack(hh, hh.n, src, lines, count, step, st); });
}

int ar_ll128_unpack_n(ar_handle h, const void* const* lines, float* const* dst, size_t count, uint64_t step,
                      ar_stream_t s)
{
    return batch_call(AR_OP_LL128_UNPACK, h, lines, reinterpret_cast<const void* const*>(dst), count, step, s,
                      [&](Handle& hh, cudaStream_t st) {
                          return launch_ll128_unpack(hh, hh.n, lines, dst, count, step, st);
                      });
}

int ar_ll_reduce(ar_handle h, const void* const* in, void* const* out, size_t count, uint32_t step, ar_stream_t s)
{
    return reduce_call(AR_OP_LL_REDUCE, h, in, out, count, step, s, [&](Handle& hh, cudaStream_t st) {
        return launch_ll_reduce(hh, in, out, count, step, st);
    });
}

int ar_ll128_reduce(ar_handle h, const void* const* in, void* const* out, size_t count, uint64_t step,
                    ar_stream_t s)
{
    return reduce_call(AR_OP_LL128_REDUCE, h, in, out, count, step, s, [&](Handle& hh, cudaStream_t st) {
        return launch_ll128_reduce(hh, in, out, count, step, st);
    });
}

int ar_allreduce_rmsnorm(ar_handle hd, const void* const* in, const void* residual, const void* weight, float eps,
                         void* const* norm_out, void* residual_out, size_t tokens, size_t hidden, ar_dtype dt,
                         ar_stream_t stream)
{
    Handle* h = get(hd);
    if (!h) return AR_ERR_INVALID;
    if (dt != AR_F32 && dt != AR_BF16 && dt != AR_F16) return AR_ERR_INVALID;
    if (!(eps >= 0.0f) || eps == INFINITY) return AR_ERR_INVALID;
    const size_t e = elem_bytes(dt);
    if (hidden == 0 || hidden % (16u / e) != 0 || !rmsnorm_fits(hidden, dt)) return AR_ERR_INVALID;
    if (tokens > SIZE_MAX / hidden / 128u) return AR_ERR_TOO_LARGE;
    const size_t count = tokens * hidden;
    if (int rc = check_multi(AR_OP_ONE_SHOT, h->n, h->max_bytes, in, norm_out, count, dt)) return rc;
    if (!residual || !weight || !residual_out) return AR_ERR_INVALID;
    if (!aligned16(residual) || !aligned16(weight) || !aligned16(residual_out)) return AR_ERR_ALIGN;
    const size_t S = count * e, W = hidden * e;
    if (residual_out != residual && overlap(residual_out, residual, S)) return AR_ERR_INVALID;
    if (overlap_sized(residual_out, S, weight, W)) return AR_ERR_INVALID;
    for (int r = 0; r < h->n; ++r)
        if (overlap(residual_out, in[r], S) || overlap(residual_out, norm_out[r], S) ||
            overlap(norm_out[r], residual, S) || overlap_sized(norm_out[r], S, weight, W))
            return AR_ERR_INVALID;
    int rc = AR_OK;
    h->timing.op = AR_OP_ALLREDUCE_RMSNORM;
    if (count)
        rc = on_device(*h, [&] {
            return launch_allreduce_rmsnorm(*h, in, residual, weight, eps, norm_out, residual_out, tokens, hidden, dt,
                                            (cudaStream_t)stream);
        });
    if (rc != AR_OK) return rc;
    plan(AR_OP_ALLREDUCE_RMSNORM, h->n, count, dt, &h->last);
    if (count) h->last.hbm_read_bytes += W;
    h->last_stream = (cudaStream_t)stream;
    return AR_OK;
}

int ar_select(int policy, int n_ranks, size_t bytes_per_rank, double alpha_s, double beta, size_t handoff_bytes)
{
    if (n_ranks < 2 || n_ranks > kMaxRanks) return AR_ERR_INVALID;
    if (policy == AR_AUTO_EMULATED) return AR_OP_ONE_SHOT;
    if (policy != AR_AUTO_MODEL || !(alpha_s >= 0.0) || !(beta > 0.0)) return AR_ERR_INVALID;
    if (handoff_bytes && bytes_per_rank > handoff_bytes) return AR_OP_RING;
    // the alpha-beta model of the three algorithms (per-rank bytes S):
    //   one-shot 2a + (n-1) S / b;  two-shot 4a + 2 (n-1)/n S / b;  ring 2(n-1) a + 2 (n-1)/n S / b
    const double n = n_ranks, S = (double)bytes_per_rank;
    const double t1 = 2.0 * alpha_s + (n - 1.0) * S / beta;
    const double t2 = 4.0 * alpha_s + 2.0 * (n - 1.0) / n * S / beta;
    const double tr = 2.0 * (n - 1.0) * alpha_s + 2.0 * (n - 1.0) / n * S / beta;
    if (t1 <= t2 && t1 <= tr) return AR_OP_ONE_SHOT;  // ties keep the simpler call
    return t2 <= tr ? AR_OP_TWO_SHOT : AR_OP_RING;
}

int ar_auto(ar_handle hd, const void* const* in, void* const* out, size_t count, ar_dtype dt, ar_stream_t s)
{
    Handle* h = get(hd);
    if (!h) return AR_ERR_INVALID;
    if (dt != AR_F32 && dt != AR_BF16 && dt != AR_F16) return AR_ERR_INVALID;
    const int op = ar_select(h->auto_policy, h->n, count * elem_bytes(dt), (double)h->auto_alpha_ns * 1e-9,
                             (double)h->auto_beta_mbs * 1e6, (size_t)h->auto_handoff);
    switch (op) {
    case AR_OP_ONE_SHOT: return ar_one_shot(hd, in, out, count, dt, s);
    case AR_OP_TWO_SHOT: return ar_two_shot(hd, in, out, count, dt, s);
    case AR_OP_RING: return ar_ring(hd, in, out, count, dt, s);
    default: return op < 0 ? op : AR_ERR_INVALID;
    }
}

int ar_status_info(ar_handle hd, ar_status_info_t* info)
{
    Handle* h = get(hd);
    if (!h) return AR_ERR_INVALID;
    DevStatus st{};
    int rc = on_device(*h, [&] {
        if (cudaDeviceSynchronize() != cudaSuccess) return AR_ERR_CUDA;
        if (cudaMemcpy(&st, h->status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return AR_ERR_CUDA;
        if ((st.code != 0 || st.skipped != 0) && cudaMemset(h->status, 0, sizeof(DevStatus)) != cudaSuccess)
            return AR_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return AR_ERR_CUDA;
        return AR_OK;
    });
    if (info) {
        info->code = rc != AR_OK ? rc : st.code;
        info->rank = st.code ? st.rank : -1;
        info->line = st.line;
        info->lines_skipped = st.skipped;
    }
    return rc != AR_OK ? rc : st.code;
}

int ar_status(ar_handle h) { return ar_status_info(h, nullptr); }

int ar_timing(ar_handle hd, ar_launch_time_t* out, int max, int* n_out)
{
    Handle* h = get(hd);
    if (!h || !n_out || max < 0 || (max > 0 && !out) || h->timing.capacity == 0) return AR_ERR_INVALID;
    Timing& t = h->timing;
    *n_out = 0;
    return on_device(*h, [&] {
        const size_t cap = (size_t)t.capacity;
        const size_t first = (t.head + cap - t.count) % cap;
        int rc = AR_OK;
        if (t.count) {
            const size_t lastslot = (t.head + cap - 1) % cap;
            if (cudaEventSynchronize(t.stop[lastslot]) != cudaSuccess) rc = AR_ERR_CUDA;
        }
        int copied = 0;
        for (size_t i = 0; i < t.count && rc == AR_OK && copied < max; ++i) {
            const size_t k = (first + i) % cap;
            ar_launch_time_t r = t.rec[k];
            if (cudaEventElapsedTime(&r.ms, t.start[k], t.stop[k]) != cudaSuccess) {
                rc = AR_ERR_CUDA;
                break;
            }
            out[copied++] = r;
        }
        *n_out = copied;
        t.count = 0;
        if (rc != AR_OK) cudaGetLastError();
        return rc;
    });
}

int ar_traffic(ar_handle hd, ar_traffic_t* t)
{
    Handle* h = get(hd);
    if (!h || !t) return AR_ERR_INVALID;
    *t = h->last;
    return AR_OK;
}

}  // extern "C"
