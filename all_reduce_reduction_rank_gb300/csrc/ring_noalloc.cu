// ar_ring_noalloc: the step-by-step ring all-reduce without a handle and
// without any allocation, for callers that cannot allocate device memory:
// code that runs where cudaMalloc is not allowed or not wanted (inside a
// framework that owns the device heap, a memory-capped serving process, a
// plugin handed only its input and output buffers).  Such a caller cannot
// use ar_ring, because ar_create allocates the partial-sum scratch.
//
// Here the scratch is one file-scope __device__ array of kNoAllocScratchBytes
// (32 MiB).  Every GPU that loads this library holds it until the process
// exits.  Host code never uses the array's name as an address: the first call
// on a device, with that device current, asks the runtime for the array's
// device address (cudaGetSymbolAddress) and the SM count, checks the result,
// and keeps both for later calls on that device.  Only a successful lookup is
// kept: a call whose lookup fails returns AR_ERR_CUDA and the next call on
// that device tries again.  Make that first call before any stream capture
// (the lookup may have to load the library's device code, which a capture
// does not allow).
//
// All calls share the one array, which keeps whatever the last call left in
// it.  Nothing in it has to start at zero: each call writes every partial
// before it reads it.  Two calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on the array; issue them in order.
//
// The kernels are variants of the ring step kernels of ring.cu (same chunks,
// same rotation, same fp32 partials, same single rounding, the same L2 hints:
// write-back stores for what the next step reads, streaming last-use loads),
// reading and writing their partials in the static array.
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace argb {
namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_ring_scratch[kNoAllocScratchBytes / sizeof(float)];

struct DeviceSetup {
    std::mutex mu;
    std::atomic<bool> ready{false};
    float* scratch = nullptr;  // device address of g_ring_scratch on this device
    int sm_count = 0;
};

DeviceSetup g_setup[kMaxDevices];

// The device address of the array and the SM count, looked up on the first
// call made with that device current and kept once the lookup succeeds.  A
// failed lookup keeps nothing, so a later call retries it; it clears the
// runtime's last-error state only if no error was pending before it.
int device_setup(int dev, DeviceSetup** out)
{
    if (dev < 0 || dev >= kMaxDevices) return AR_ERR_CUDA;
    DeviceSetup& d = g_setup[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(d.mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            const bool pending = cudaPeekAtLastError() != cudaSuccess;
            void* p = nullptr;
            int sms = 0;
            if (cudaGetSymbolAddress(&p, g_ring_scratch) != cudaSuccess || p == nullptr ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
                if (!pending) cudaGetLastError();
                return AR_ERR_CUDA;
            }
            d.scratch = static_cast<float*>(p);
            d.sm_count = sms;
            d.ready.store(true, std::memory_order_release);
        }
    }
    *out = &d;
    return AR_OK;
}

// Grid cap: the library's default launch policy (at most 64 CTAs per SM per
// launch, shared by the n rank rows, the CTAs grid-striding past that), the
// same cap ar_ring's step launches use when no AR_OPT_CTAS_PER_SM is set.
// Many short-lived CTAs let the block scheduler balance the SMs; measured on
// GB300 they beat one resident wave of grid-striding CTAs by 5-14%.
constexpr int kCtasPerSm = 64;

// Reduce-scatter step s: rank r sends chunk (r - s) mod n to rank r + 1, which
// adds its own chunk; fp32 partials in `scratch` ([2][n][C], by step parity).
template <int NR, int DT>
__global__ void __launch_bounds__(kThreads)
noalloc_ring_rs_kernel(const __grid_constant__ CPtrs<NR> in, const __grid_constant__ MPtrs<NR> out,
                       float* __restrict__ scratch, size_t C, size_t count, int s)
{
    constexpr int VE = kVecElems<DT>;
    constexpr int PW = VE / 4;
    using T = typename Payload<DT>::scalar_t;
    const int r = blockIdx.y;
    const int d = (r + 1) % NR;
    const int c = (r - s + NR) % NR;
    const bool first = (s == 0), last = (s == NR - 2);
    const size_t e_lo = (size_t)c * C;
    if (e_lo >= count) return;
    const size_t len = count - e_lo < C ? count - e_lo : C;
    const size_t nv = len / VE;
    const T* const xr = static_cast<const T*>(in.p[r]) + e_lo;
    const T* const xd = static_cast<const T*>(in.p[d]) + e_lo;
    T* const od = static_cast<T*>(out.p[d]) + e_lo;
    const float* const pr = scratch + (size_t)((s + 1) & 1) * NR * C + (size_t)r * C;
    float* const pw = scratch + (size_t)(s & 1) * NR * C + (size_t)d * C;
    for (size_t k = (size_t)blockIdx.x * kThreads + threadIdx.x; k < nv; k += (size_t)gridDim.x * kThreads) {
        float a[VE];
        if (first) {
            const uint4 x = ld16_last(xr + k * VE);
#pragma unroll
            for (int j = 0; j < 4; ++j) Payload<DT>::widen(word(x, j), a + j * Payload<DT>::kPerWord);
        } else {
#pragma unroll
            for (int j = 0; j < PW; ++j) {
                const uint4 t = ld16_last(pr + k * VE + 4 * j);
                a[4 * j] = __uint_as_float(t.x);
                a[4 * j + 1] = __uint_as_float(t.y);
                a[4 * j + 2] = __uint_as_float(t.z);
                a[4 * j + 3] = __uint_as_float(t.w);
            }
        }
        accumulate<DT>(a, ld16_last(xd + k * VE));
        if (last) {
            st16_next(od + k * VE, round_vec<DT>(a));
        } else {
#pragma unroll
            for (int j = 0; j < PW; ++j)
                st16_next(pw + k * VE + 4 * j, make_uint4(__float_as_uint(a[4 * j]), __float_as_uint(a[4 * j + 1]),
                                                          __float_as_uint(a[4 * j + 2]), __float_as_uint(a[4 * j + 3])));
        }
    }
    if (blockIdx.x == gridDim.x - 1) {  // the ragged end of the last chunk
        const size_t j = nv * VE + threadIdx.x;
        if (j < len) {
            const float up = first ? Payload<DT>::widen1(xr[j]) : pr[j];
            const float sum = up + Payload<DT>::widen1(xd[j]);
            if (last) od[j] = Payload<DT>::narrow1(sum);
            else pw[j] = sum;
        }
    }
}

// All-gather step s: rank r + 1 copies chunk (r + 1 - s) mod n from rank r.
template <int NR, int DT>
__global__ void __launch_bounds__(kThreads)
noalloc_ring_ag_kernel(const __grid_constant__ MPtrs<NR> out, size_t C, size_t count, int s)
{
    constexpr int VE = kVecElems<DT>;
    using T = typename Payload<DT>::scalar_t;
    const int r = blockIdx.y;
    const int d = (r + 1) % NR;
    const int c = (r + 1 - s + NR) % NR;
    const size_t e_lo = (size_t)c * C;
    if (e_lo >= count) return;
    const size_t len = count - e_lo < C ? count - e_lo : C;
    const size_t nv = len / VE;
    const T* const src = static_cast<const T*>(out.p[r]) + e_lo;
    T* const dst = static_cast<T*>(out.p[d]) + e_lo;
    for (size_t k = (size_t)blockIdx.x * kThreads + threadIdx.x; k < nv; k += (size_t)gridDim.x * kThreads)
        st16_next(dst + k * VE, ld16(src + k * VE));
    if (blockIdx.x == gridDim.x - 1) {
        const size_t j = nv * VE + threadIdx.x;
        if (j < len) dst[j] = src[j];
    }
}

}  // namespace
}  // namespace argb

using namespace argb;

extern "C" int ar_ring_noalloc(int n_ranks, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                               ar_stream_t stream)
{
    // the same argument checks as ar_ring, with no handle and no size cap here ...
    int rc = ar_check_args(AR_OP_RING, n_ranks, SIZE_MAX, in, out, count, dt);
    if (rc != AR_OK) return rc;
    if (count == 0) return AR_OK;
    // ... and the cap of the static scratch: 2 x n x C fp32 partials
    const size_t C = chunk_elems(n_ranks, count, dt);
    if (C > kNoAllocScratchBytes / sizeof(float) / 2 / (size_t)n_ranks) return AR_ERR_TOO_LARGE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
    DeviceSetup* d = nullptr;
    if ((rc = device_setup(dev, &d)) != AR_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return dispatch_dtype(dt, [&](auto dtc) -> int {
        constexpr int DT = decltype(dtc)::value;
        return dispatch_ranks(n_ranks, [&](auto nrc) -> int {
            constexpr int NR = decltype(nrc)::value;
            CPtrs<NR> ip;
            MPtrs<NR> op;
            for (int q = 0; q < NR; ++q) {
                ip.p[q] = in[q];
                op.p[q] = out[q];
            }
            const size_t cvec = C / kVecElems<DT>;
            size_t gx = (cvec + kThreads - 1) / kThreads;
            const size_t cap = (size_t)d->sm_count * kCtasPerSm / NR;
            if (gx > cap) gx = cap;
            if (gx == 0) gx = 1;
            const dim3 grid((unsigned)gx, NR);
            for (int step = 0; step < NR - 1; ++step) {
                noalloc_ring_rs_kernel<NR, DT><<<grid, kThreads, 0, s>>>(ip, op, d->scratch, C, count, step);
                if (cudaGetLastError() != cudaSuccess) return AR_ERR_CUDA;
            }
            for (int step = 0; step < NR - 1; ++step) {
                noalloc_ring_ag_kernel<NR, DT><<<grid, kThreads, 0, s>>>(op, C, count, step);
                if (cudaGetLastError() != cudaSuccess) return AR_ERR_CUDA;
            }
            return AR_OK;
        });
    });
}
