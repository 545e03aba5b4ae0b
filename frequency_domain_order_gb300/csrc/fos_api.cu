// fos_api.cu -- the C ABI of libfir_os.so (include/fir_os.h): plans, argument checks,
// launches, the plan-time kernels and the pipelined host-buffer path.
//
// Method: "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法" (zl.czvv.com/42398539.html),
// 主权项 steps 1-6.  Step 1 (frequency response) runs here at plan time; steps 3-5 run in the
// fused block kernels (fos_block.cuh, fos_resident.cu, fos_pair.cu); steps 2 and 6 (moving chunks between
// host and device and repeating) are fir_os_execute_host.
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "fir_os.h"  // include/ is on the include path (build.py)
#include "fos_chan.h"
#include "fos_fft.cuh"
#include "fos_kernels.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(FIR_OS_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define FOS_CUDA(call, what)                          \
    do {                                              \
        cudaError_t e_ = (call);                      \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

// Every allocation the library makes -- its plan objects and its device buffers -- goes
// through alloc_take / dev_alloc and is returned through alloc_give / dev_free, which keep
// the number of live allocations (fir_os_debug_live_allocs) and can be told to fail the k-th
// next allocation as if memory had run out (fir_os_debug_fail_alloc): a host-side way to
// reach every allocation-failure path without exhausting a device.
std::atomic<long long> g_live_allocs{0};
std::atomic<int> g_fail_countdown{0};

// True when this allocation is the one chosen to fail.
bool injected_failure() {
    int k = g_fail_countdown.load();
    while (k > 0 && !g_fail_countdown.compare_exchange_weak(k, k - 1)) {
    }
    return k == 1;
}

cudaError_t dev_alloc_raw(void **ptr, size_t bytes) {
    *ptr = nullptr;
    if (injected_failure()) return cudaErrorMemoryAllocation;
    const cudaError_t e = cudaMalloc(ptr, bytes);
    if (e == cudaSuccess) ++g_live_allocs;
    return e;
}
template <class T>
cudaError_t dev_alloc(T **ptr, size_t bytes) {
    void *v = nullptr;
    const cudaError_t e = dev_alloc_raw(&v, bytes);
    *ptr = static_cast<T *>(v);
    return e;
}
void dev_free(void *ptr) {
    if (!ptr) return;
    cudaFree(ptr);
    --g_live_allocs;
}
template <class T>
T *alloc_take() {
    if (injected_failure()) return nullptr;
    T *p = new (std::nothrow) T;
    if (p) ++g_live_allocs;
    return p;
}
template <class T>
void alloc_give(T *p) {
    if (!p) return;
    delete p;
    --g_live_allocs;
}

// status of a failed device allocation: FIR_OS_E_NOMEM when memory ran out, else the CUDA error
int alloc_fail(cudaError_t e, const char *what) {
    cudaGetLastError();  // an allocation failure leaves no sticky error; clear the last-error slot
    if (e == cudaErrorMemoryAllocation) return fail(FIR_OS_E_NOMEM, "%s: out of device memory", what);
    return cuda_fail(e, what);
}

// ------------------------------------------------------------------ plan-time kernels

// A[t] = h[t] (t < M), 0 (M <= t < N), in float64.
__global__ void fos_fill_h64(double2 *A, const void *h, int M, int N, int h_complex) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= N) return;
    double2 v = make_double2(0.0, 0.0);
    if (t < M) {
        if (h_complex) {
            const float2 z = static_cast<const float2 *>(h)[t];
            v = make_double2((double)z.x, (double)z.y);
        } else {
            v = make_double2((double)static_cast<const float *>(h)[t], 0.0);
        }
    }
    A[t] = v;
}

// One radix-2 Stockham pass of the forward float64 FFT: group j = 0..N/2-1 reads z[j] and
// z[j + N/2], multiplies the second by e^{-2 pi i m / (2 Ns)} (m = j mod Ns) and writes the
// sum and difference to (j / Ns) 2 Ns + m and that + Ns.
__global__ void fos_radix2_pass64(const double2 *src, double2 *dst, int N, int Ns) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N / 2) return;
    const int m = j & (Ns - 1);
    double s, c;
    sincospi(-(double)m / (double)Ns, &s, &c);
    const double2 a = src[j], b0 = src[j + N / 2];
    const double2 b = make_double2(b0.x * c - b0.y * s, b0.x * s + b0.y * c);
    const int o = (j / Ns) * 2 * Ns + m;
    dst[o] = make_double2(a.x + b.x, a.y + b.y);
    dst[o + Ns] = make_double2(a.x - b.x, a.y - b.y);
}

// H[t] = A[t] / N rounded to float32 (the inverse transform's 1/N folded into H).
__global__ void fos_finish_h(const double2 *A, float2 *H, int N) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < N) H[t] = make_float2((float)(A[t].x / N), (float)(A[t].y / N));
}

// H[t] = Hin[t] / N (N a power of two: exact).
__global__ void fos_scale_h(const float2 *Hin, float2 *H, int N) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < N) {
        const float s = 1.0f / (float)N;
        H[t] = make_float2(Hin[t].x * s, Hin[t].y * s);
    }
}

// Hk[c (N / C) + d] = H[c + C d]: the c-major order of the resident kernel.
__global__ void fos_permute_h(const float2 *H, float2 *Hk, int N, int C) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < N) {
        const int P = N / C;
        Hk[t] = H[(t % P) * C + t / P];
    }
}

// S0' = last `hist` samples of concat(S0, x), in place, for channels blockIdx.y, blockIdx.y +
// gridDim.y, ... (channel c's x and state start at c * x_stride and c * s_stride).  Used when
// the kernel that read S0 cannot write the state itself.  n >= hist: a copy of x's tail spread
// over the CTAs of a row (blockIdx.x).  n < hist: the kept part of S0 moves towards the front,
// by CTA 0 of the row alone; chunks are read completely before they are written and every
// later chunk reads only indices beyond what earlier chunks wrote.  Launched with programmatic
// serialization: it waits for the kernel before it (which reads S0) before touching anything.
template <typename T>
__global__ void fos_state_kernel(const T *x, int64_t n, T *state, int hist, int64_t x_stride, int64_t s_stride,
                                 int channels) {
    fos::griddep_launch_dependents();
    fos::griddep_wait();
    for (int c = blockIdx.y; c < channels; c += gridDim.y) {
        const T *xc = x + c * x_stride;
        T *sc = state + c * s_stride;
        if (n >= hist) {
            const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
            if (t < hist) sc[t] = xc[n - hist + t];
            continue;
        }
        if (blockIdx.x != 0) continue;
        const int keep = hist - (int)n;  // samples of S0 that stay
        for (int c0 = 0; c0 < hist; c0 += blockDim.x) {
            const int t = c0 + threadIdx.x;
            T v{};
            if (t < hist) v = t < keep ? sc[n + t] : xc[t - keep];
            __syncthreads();
            if (t < hist) sc[t] = v;
            __syncthreads();
        }
    }
}

// Enqueue fos_state_kernel for `channels` channels after the kernel just launched on `stream`.
template <typename T>
cudaError_t launch_state(const void *x, int64_t n, void *state, int hist, int64_t xs, int64_t ss, int channels,
                         cudaStream_t stream) {
    const bool copy = n >= hist;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(copy ? 256 : 1024);
    cfg.gridDim = dim3(copy ? (unsigned)((hist + 255) / 256) : 1u, (unsigned)(channels < 65535 ? channels : 65535));
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fos_state_kernel<T>, static_cast<const T *>(x), n, static_cast<T *>(state), hist,
                              xs, ss, channels);
}

// Measurement aid for the FP32 roofline: eight independent multiply-add chains per thread, so
// that every SM's FP32 lanes stay busy.  The sum is stored only if it equals -1, which the
// chains never reach (every value stays positive); the compiler cannot drop them.
__global__ void __launch_bounds__(1024) fos_fp32_probe_kernel(float *sink, int iters) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 1.0f + 1e-3f * (float)(threadIdx.x + i);
    const float b = 0.9999f, c = 1e-4f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = fmaf(a[i], b, c);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += a[i];
    if (s == -1.0f) sink[blockIdx.x] = s;
}

// ------------------------------------------------------------------ allocation-free response
// fir_os_frequency_response_noalloc runs the float64 step-1 transform above with its two
// ping-pong buffers taken from this fixed device array instead of cudaMalloc.  Every device
// that loads the library holds these 2 MiB until the process exits; all calls share them.
constexpr int kNoallocMaxN = 65536;
static __device__ __align__(256) double2 g_noalloc_scratch[2 * kNoallocMaxN];

// H[t] = A[t] rounded to complex64 (unscaled, as a given response is passed to a plan).
__global__ void fos_store_h(const double2 *A, float2 *H, int N) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < N) H[t] = make_float2((float)A[t].x, (float)A[t].y);
}

std::mutex g_noalloc_mu;
double2 *g_noalloc_ptr[128] = {};

// Device address of the scratch array for the current device, looked up once per device
// with that device current (the array's name is only a host-side stand-in in host code).
int noalloc_scratch(double2 **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 128) return fail(FIR_OS_E_UNSUPPORTED, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        // the first lookup on a device may load the library's device code there, which is when
        // the array itself is allocated: running out of memory then is FIR_OS_E_NOMEM
        if (e != cudaSuccess) return alloc_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_noalloc_ptr[dev] = static_cast<double2 *>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return FIR_OS_OK;
}

// ------------------------------------------------------------------ plan

bool ranges_overlap(uintptr_t a, size_t na, uintptr_t b, size_t nb) {
    if (na == 0 || nb == 0) return false;
    return a < b + nb && b < a + na;
}

}  // namespace

struct fir_os_plan {
    int M = 0, N = 0, L = 0;
    int data_kind = FIR_OS_COMPLEX;
    int device = 0;
    int sms = 0;
    fos::KernelEntry kernel;
    int max_units_in_flight = 0;  // CTAs, or clusters for a cluster kernel
    float2 *d_H = nullptr;
    float2 *d_Hk = nullptr;  // H in the kernel's order, when that is not the natural one
    float2 *d_tw = nullptr;
    float2 *d_twa = nullptr;
    int *d_err = nullptr;
    uint64_t wait_ns = fos::kWaitLimitNs;  // limit of a kernel's wait for one bulk copy
    int dft_engine = FIR_OS_DFT_FP32;      // FIR_OS_DFT_TENSOR: the tensor-core kernel variant
    float2 *d_btc = nullptr;               // its split 16-point DFT matrices (fos_tc.cuh)
    // host-buffer path (lazily created)
    int64_t host_chunk = 0;
    void *hx[2] = {nullptr, nullptr};
    void *hy[2] = {nullptr, nullptr};
    void *hstate = nullptr;
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    cudaEvent_t ev_in[2] = {nullptr, nullptr}, ev_comp[2] = {nullptr, nullptr}, ev_out[2] = {nullptr, nullptr};
    cudaEvent_t ev_start = nullptr;
};

namespace {

int sample_bytes(const fir_os_plan *p) { return p->data_kind == FIR_OS_REAL ? 4 : 8; }

// Makes `dev` the current device for the lifetime of the object and then restores the
// caller's current device (plans are destroyed on the device that holds their memory).
struct DeviceScope {
    int prev = -1;
    explicit DeviceScope(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            cudaGetLastError();
            prev = -1;
        } else if (prev != dev) {
            cudaSetDevice(dev);
        }
    }
    ~DeviceScope() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

// The host-buffer path's device buffers, events and streams (created on its first call).
void release_host_path(fir_os_plan *p) {
    for (int k = 0; k < 2; ++k) {
        dev_free(p->hx[k]);
        dev_free(p->hy[k]);
        p->hx[k] = p->hy[k] = nullptr;
        if (p->ev_in[k]) cudaEventDestroy(p->ev_in[k]);
        if (p->ev_comp[k]) cudaEventDestroy(p->ev_comp[k]);
        if (p->ev_out[k]) cudaEventDestroy(p->ev_out[k]);
        p->ev_in[k] = p->ev_comp[k] = p->ev_out[k] = nullptr;
    }
    dev_free(p->hstate);
    p->hstate = nullptr;
    if (p->ev_start) cudaEventDestroy(p->ev_start);
    if (p->s_in) cudaStreamDestroy(p->s_in);
    if (p->s_comp) cudaStreamDestroy(p->s_comp);
    if (p->s_out) cudaStreamDestroy(p->s_out);
    p->ev_start = nullptr;
    p->s_in = p->s_comp = p->s_out = nullptr;
    p->host_chunk = 0;
}

void free_plan(fir_os_plan *p) {
    if (!p) return;
    dev_free(p->d_H);
    dev_free(p->d_Hk);
    dev_free(p->d_tw);
    dev_free(p->d_twa);
    dev_free(p->d_err);
    dev_free(p->d_btc);
    release_host_path(p);
    alloc_give(p);
}

// Stockham pass twiddles of a 2^logn-point per-CTA transform (layout in fos_fft.cuh),
// computed in float64 and rounded.
template <int LOGN>
void fill_pass_twiddles(std::vector<float2> &tw) {
    using S = fos::FftShape<LOGN>;
    tw.assign(S::TW_ENTRIES > 0 ? S::TW_ENTRIES : 1, make_float2(0.f, 0.f));
    for (int p = 1; p < S::NPASS; ++p) {
        const int Ns = S::ns(p);
        const long long period = 16LL * Ns;
        for (int r = 1; r < 16; ++r)
            for (int m = 0; m < Ns; ++m) {
                const long long e = ((long long)m * r) % period;
                const double ang = -2.0 * M_PI * (double)e / (double)period;
                tw[S::twoff(p) + (r - 1) * Ns + m] = make_float2((float)std::cos(ang), (float)std::sin(ang));
            }
    }
}

bool pass_twiddles(int logn, std::vector<float2> &tw) {
    switch (logn) {
        case 6: fill_pass_twiddles<6>(tw); return true;
        case 7: fill_pass_twiddles<7>(tw); return true;
        case 8: fill_pass_twiddles<8>(tw); return true;
        case 9: fill_pass_twiddles<9>(tw); return true;
        case 10: fill_pass_twiddles<10>(tw); return true;
        case 11: fill_pass_twiddles<11>(tw); return true;
        case 12: fill_pass_twiddles<12>(tw); return true;
        case 13: fill_pass_twiddles<13>(tw); return true;
        default: return false;
    }
}

int ilog2i(int v) {
    int r = 0;
    while ((1 << r) < v) ++r;
    return r;
}

int64_t units_for(const fir_os_plan *p, int64_t n) {
    const int64_t blocks = (n + p->L - 1) / p->L;
    const int64_t per = p->data_kind == FIR_OS_REAL ? (blocks + 1) / 2 : blocks;  // transforms
    return (per + p->kernel.units_per_cta - 1) / p->kernel.units_per_cta;
}

// The block kernel writes S0' itself when only its first work unit reads S0 (the next unit
// starts at or after sample 0); the cluster and resident kernels additionally need n >= M-1,
// because they write S0' from x (they keep no staged copy of S0).
bool fuse_state(const fir_os_plan *p, int64_t n) {
    if (p->M == 1) return true;
    const int64_t span = (int64_t)p->kernel.units_per_cta * p->L * (p->data_kind == FIR_OS_REAL ? 2 : 1);
    if (p->kernel.cluster == 1 && !p->kernel.state_from_x) return span >= p->M - 1;
    return span >= p->M - 1 && n >= p->M - 1;
}

// One call over `channels` streams of n samples each; channel c's x, y and state start at
// c * xs, c * ys and c * ss samples.
int launch_blocks(fir_os_plan *p, const void *x, int64_t n, void *y, void *state, cudaStream_t stream,
                  bool host_resident = false, int channels = 1, int64_t xs = 0, int64_t ys = 0,
                  int64_t ss = 0) {
    const bool real = p->data_kind == FIR_OS_REAL;
    fos::BlockParams bp{};
    bp.x = x;
    bp.y = y;
    bp.state = state;
    bp.H = p->d_Hk ? p->d_Hk : p->d_H;
    bp.tw = p->d_tw;
    bp.twa = p->d_twa;
    bp.err = p->d_err;
    bp.wait_ns = p->wait_ns;
    bp.btc = p->d_btc;
    bp.n = n;
    bp.upc = units_for(p, n);
    bp.nunits = bp.upc * channels;
    bp.x_stride = xs;
    bp.y_stride = ys;
    bp.s_stride = ss;
    bp.M = p->M;
    bp.L = p->L;
    bp.fuse_state = fuse_state(p, n);
    bp.no_bulk = host_resident ? 1 : 0;
    // CTAs (or clusters) to launch: one per unit, at most what is resident, so that a call of
    // few units runs on as many SMs as it can (the block kernel deals units across CTAs first)
    const int64_t groups = bp.nunits < p->max_units_in_flight ? bp.nunits : p->max_units_in_flight;
    void *args[] = {&bp};
    // programmatic serialization: the kernel's set-up (Tensor Memory, plan constants) overlaps
    // the end of the kernel before it in the stream; it waits for that kernel before it touches
    // x, y or the state
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(groups * p->kernel.cluster));
    cfg.blockDim = dim3(p->kernel.threads);
    cfg.dynamicSmemBytes = (size_t)p->kernel.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p->kernel.cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = p->kernel.cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    const void *func = channels > 1 && p->kernel.func_multi ? p->kernel.func_multi : p->kernel.func;
    // less than one wave: each group filters one unit at most, so the per-thread Tensor Memory
    // set-up of the plan constants would sit on the call's critical path; the variant that keeps
    // them in shared memory avoids it
    if (p->dft_engine == FIR_OS_DFT_TENSOR) {
        func = channels > 1 && p->kernel.func_multi_tc ? p->kernel.func_multi_tc : p->kernel.func_tc;
        cfg.dynamicSmemBytes = (size_t)p->kernel.smem_tc;
    } else if (p->kernel.func_short && bp.nunits < (int64_t)p->max_units_in_flight * p->kernel.groups) {
        func = p->kernel.func_short;
        cfg.dynamicSmemBytes = (size_t)p->kernel.smem_short;
    }
    FOS_CUDA(cudaLaunchKernelExC(&cfg, func, args), "block kernel launch");
    if (!bp.fuse_state && p->M > 1)
        FOS_CUDA(real ? launch_state<float>(x, n, state, p->M - 1, xs, ss, channels, stream)
                      : launch_state<float2>(x, n, state, p->M - 1, xs, ss, channels, stream),
                 "state kernel launch");
    return FIR_OS_OK;
}

// Page-locked host memory that kernels can address directly (its device address in *dev).
bool host_mapped(const void *p, void **dev) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // pageable memory is not an error here
        return false;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return false;
    *dev = a.devicePointer;
    return true;
}

int check_device(const fir_os_plan *p) {
    int dev = -1;
    FOS_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev != p->device)
        return fail(FIR_OS_E_INVAL, "plan was created on device %d but device %d is current", p->device, dev);
    return FIR_OS_OK;
}

// Device time of one block (real data: one block of a packed pair) in SM-microseconds, measured
// on a GB300 (152 SMs, 2070 MHz) by timing one call of at least 2048 blocks (about 64 M samples)
// per N with M - 1 = N/4, N/2 and 3N/4, i.e. L/N = 3/4, 1/2, 1/4 (stored in increasing L/N).
struct BlockCost {
    int N;
    int real;
    double sm_us[3];  // at L/N = 1/4, 1/2, 3/4
};
const BlockCost kBlockCost[] = {
    {64, 0, {0.0309, 0.0330, 0.0357}},
    {128, 0, {0.0460, 0.0484, 0.0513}},
    {256, 0, {0.0858, 0.0893, 0.0931}},
    {512, 0, {0.2290, 0.2354, 0.2434}},
    {1024, 0, {0.4600, 0.4732, 0.4841}},
    {2048, 0, {1.0472, 1.0486, 1.0733}},
    {4096, 0, {2.3304, 2.3415, 2.4525}},
    {8192, 0, {6.4839, 6.7751, 7.1168}},
    {16384, 0, {12.2143, 12.7163, 13.1371}},
    {32768, 0, {23.9522, 24.8781, 26.2362}},
    {65536, 0, {61.0155, 63.3709, 65.2650}},
    {64, 1, {0.0206, 0.0229, 0.0259}},
    {128, 1, {0.0278, 0.0301, 0.0327}},
    {256, 1, {0.0472, 0.0502, 0.0534}},
    {512, 1, {0.1212, 0.1277, 0.1344}},
    {1024, 1, {0.2384, 0.2499, 0.2649}},
    {2048, 1, {0.5367, 0.5664, 0.5943}},
    {4096, 1, {1.2849, 1.2285, 1.3766}},
    {8192, 1, {3.3923, 3.5429, 3.7589}},
    {16384, 1, {6.4027, 6.7892, 7.1268}},
    {32768, 1, {12.8559, 14.3569, 15.0027}},
    {65536, 1, {31.5299, 34.3959, 35.3792}},
};

// Predicted throughput (output samples per second, 1e9) of an (M, N) plan on `sms` SMs: L
// samples per block, the block's SM time interpolated linearly in L/N between the measured
// points (extrapolated linearly beyond them).
double predict_gsps(int M, int N, bool real, int sms) {
    for (const BlockCost &b : kBlockCost) {
        if (b.N != N || b.real != (real ? 1 : 0)) continue;
        const int L = N - M + 1;
        const double f = (double)L / N;
        const double x0 = f <= 0.5 ? 0.25 : 0.5;
        const double y0 = f <= 0.5 ? b.sm_us[0] : b.sm_us[1];
        const double y1 = f <= 0.5 ? b.sm_us[1] : b.sm_us[2];
        double t = y0 + (y1 - y0) * (f - x0) / 0.25;
        if (t < 0.5 * b.sm_us[0]) t = 0.5 * b.sm_us[0];
        return (double)L * sms / t * 1e-3;
    }
    return 0.0;
}

}  // namespace

extern "C" {

int fir_os_predict_gsps(int M, int N, int data_kind, int sms, double *gsps) {
    if (!gsps) return fail(FIR_OS_E_INVAL, "gsps is NULL");
    if (data_kind != FIR_OS_REAL && data_kind != FIR_OS_COMPLEX)
        return fail(FIR_OS_E_INVAL, "data_kind %d is neither FIR_OS_REAL nor FIR_OS_COMPLEX", data_kind);
    if (sms < 0) return fail(FIR_OS_E_INVAL, "sms < 0");
    if (N < 64 || N > 65536 || (N & (N - 1)) != 0)
        return fail(FIR_OS_E_UNSUPPORTED, "N = %d is not a power of two in [64, 65536]", N);
    if (M < 1 || M > N) return fail(FIR_OS_E_UNSUPPORTED, "M = %d must be in [1, N = %d]", M, N);
    *gsps = predict_gsps(M, N, data_kind == FIR_OS_REAL, sms ? sms : 152);
    return FIR_OS_OK;
}

int fir_os_choose_n(int M, int data_kind, int sms, int *N, double *gsps) {
    if (!N) return fail(FIR_OS_E_INVAL, "N is NULL");
    if (data_kind != FIR_OS_REAL && data_kind != FIR_OS_COMPLEX)
        return fail(FIR_OS_E_INVAL, "data_kind %d is neither FIR_OS_REAL nor FIR_OS_COMPLEX", data_kind);
    if (sms < 0) return fail(FIR_OS_E_INVAL, "sms < 0");
    if (M < 1) return fail(FIR_OS_E_INVAL, "M = %d < 1", M);
    if (M > 65536) return fail(FIR_OS_E_UNSUPPORTED, "M = %d > 65536", M);
    int best = 0;
    double best_g = -1.0;
    for (int n = 64; n <= 65536; n *= 2) {
        if (n < M) continue;
        const double g = predict_gsps(M, n, data_kind == FIR_OS_REAL, sms ? sms : 152);
        if (g > best_g) {
            best_g = g;
            best = n;
        }
    }
    *N = best;
    if (gsps) *gsps = best_g;
    return FIR_OS_OK;
}


const char *fir_os_status_string(int status) {
    switch (status) {
        case FIR_OS_OK: return "ok";
        case FIR_OS_E_INVAL: return "invalid argument";
        case FIR_OS_E_UNSUPPORTED: return "unsupported configuration";
        case FIR_OS_E_ALIGN: return "misaligned buffer";
        case FIR_OS_E_NOMEM: return "out of memory";
        case FIR_OS_E_CUDA: return "CUDA error";
        case FIR_OS_E_DEVICE: return "device-side wait ran out";
        default: return "unknown status";
    }
}

const char *fir_os_last_error(void) { return g_last_error; }

int fir_os_plan_create(fir_os_plan_t *out, int M, int N, int data_kind, int coef_kind, int coef_complex,
                       const void *coef_dev, void *stream_) {
    g_last_error[0] = 0;
    if (!out) return fail(FIR_OS_E_INVAL, "out is NULL");
    *out = nullptr;
    if (N < 64 || N > 65536 || (N & (N - 1)) != 0)
        return fail(FIR_OS_E_UNSUPPORTED, "N = %d is not a power of two in [64, 65536]", N);
    if (M < 1 || M > N) return fail(FIR_OS_E_UNSUPPORTED, "M = %d must be in [1, N = %d]", M, N);
    if (data_kind != FIR_OS_REAL && data_kind != FIR_OS_COMPLEX)
        return fail(FIR_OS_E_INVAL, "data_kind %d is neither FIR_OS_REAL nor FIR_OS_COMPLEX", data_kind);
    if (coef_kind != FIR_OS_COEF_TIME && coef_kind != FIR_OS_COEF_FREQ)
        return fail(FIR_OS_E_INVAL, "coef_kind %d is neither FIR_OS_COEF_TIME nor FIR_OS_COEF_FREQ", coef_kind);
    if (coef_kind == FIR_OS_COEF_TIME && coef_complex != 0 && coef_complex != 1)
        return fail(FIR_OS_E_INVAL, "coef_complex must be 0 or 1");
    if (!coef_dev) return fail(FIR_OS_E_INVAL, "coef_dev is NULL");
    if (coef_kind == FIR_OS_COEF_TIME && data_kind == FIR_OS_REAL && coef_complex)
        return fail(FIR_OS_E_UNSUPPORTED, "real data needs a real h");
    if (coef_kind == FIR_OS_COEF_FREQ && (reinterpret_cast<uintptr_t>(coef_dev) & 15))
        return fail(FIR_OS_E_ALIGN, "a given H must be 16-byte aligned");
    if (coef_kind == FIR_OS_COEF_TIME && (reinterpret_cast<uintptr_t>(coef_dev) & (coef_complex ? 7 : 3)))
        return fail(FIR_OS_E_ALIGN, "h must be naturally aligned");

    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    fir_os_plan *p = alloc_take<fir_os_plan>();
    if (!p) return fail(FIR_OS_E_NOMEM, "plan allocation failed");
    int rc = FIR_OS_OK;
    auto bail = [&](int status) {
        free_plan(p);
        return status;
    };
    p->M = M;
    p->N = N;
    p->L = N - M + 1;
    p->data_kind = data_kind;
    {
        cudaError_t e = cudaGetDevice(&p->device);
        if (e != cudaSuccess) return bail(cuda_fail(e, "cudaGetDevice"));
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, p->device);
        if (e != cudaSuccess) return bail(cuda_fail(e, "cudaGetDeviceProperties"));
        if (!(prop.major == 10 && prop.minor == 3))
            return bail(fail(FIR_OS_E_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                             p->device, prop.major, prop.minor));
        p->sms = prop.multiProcessorCount;
    }

    const int logn = ilog2i(N);
    const bool real = data_kind == FIR_OS_REAL;
    if (logn <= 9) p->kernel = fos::block_kernel_small(logn, real);
    else if (logn <= 13) p->kernel = fos::block_kernel_large(logn, real);
    else if (logn <= 15) p->kernel = fos::resident_kernel(logn, real);
    else p->kernel = fos::pair_kernel(logn, real);
    if (!p->kernel.func) return bail(fail(FIR_OS_E_UNSUPPORTED, "no kernel for N = %d", N));

    // launch shape
    {
        cudaError_t e = cudaFuncSetAttribute(p->kernel.func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             p->kernel.smem);
        if (e != cudaSuccess) return bail(cuda_fail(e, "cudaFuncSetAttribute(smem)"));
        if (p->kernel.func_multi) {
            e = cudaFuncSetAttribute(p->kernel.func_multi, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     p->kernel.smem);
            if (e != cudaSuccess) return bail(cuda_fail(e, "cudaFuncSetAttribute(smem)"));
        }
        if (p->kernel.func_short) {
            e = cudaFuncSetAttribute(p->kernel.func_short, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     p->kernel.smem_short);
            if (e != cudaSuccess) return bail(cuda_fail(e, "cudaFuncSetAttribute(smem)"));
        }
        if (p->kernel.cluster == 1) {
            int per_sm = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, p->kernel.func, p->kernel.threads,
                                                              (size_t)p->kernel.smem);
            if (e != cudaSuccess) return bail(cuda_fail(e, "occupancy query"));
            if (per_sm < 1) return bail(fail(FIR_OS_E_UNSUPPORTED, "block kernel does not fit an SM"));
            p->max_units_in_flight = per_sm * p->sms;
        } else {

            cudaLaunchConfig_t cfg{};
            cfg.gridDim = dim3(p->kernel.cluster * 64);
            cfg.blockDim = dim3(p->kernel.threads);
            cfg.dynamicSmemBytes = (size_t)p->kernel.smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = p->kernel.cluster;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            e = cudaOccupancyMaxActiveClusters(&clusters, p->kernel.func, &cfg);
            if (e != cudaSuccess) return bail(cuda_fail(e, "cluster occupancy query"));
            if (clusters < 1)
                return bail(fail(FIR_OS_E_UNSUPPORTED, "a cluster of %d CTAs cannot be resident", p->kernel.cluster));
            p->max_units_in_flight = clusters;
        }
    }

    // device memory
    {
        cudaError_t e;
        if ((e = dev_alloc(&p->d_H, sizeof(float2) * N)) != cudaSuccess ||
            (e = dev_alloc(&p->d_err, sizeof(int))) != cudaSuccess)
            return bail(alloc_fail(e, "cudaMalloc(H, error word)"));
        std::vector<float2> tw;
        if (!pass_twiddles(p->kernel.fft_logn, tw)) return bail(fail(FIR_OS_E_UNSUPPORTED, "twiddles"));
        if ((e = dev_alloc(&p->d_tw, sizeof(float2) * tw.size())) != cudaSuccess)
            return bail(alloc_fail(e, "cudaMalloc(twiddles)"));
        if ((e = cudaMemcpyAsync(p->d_tw, tw.data(), sizeof(float2) * tw.size(), cudaMemcpyHostToDevice,
                                 stream)) != cudaSuccess)
            return bail(cuda_fail(e, "twiddle upload"));
        if (p->kernel.split_c > 0) {
            // W_N^b for b = r + 128 m, as its factors: W_N^r (r < 128), then W_N^{128 m} (m < 32);
            // float64, then rounded
            std::vector<float2> twa((size_t)(128 + 32));
            for (int r = 0; r < 128; ++r) {
                const double ang = -2.0 * M_PI * (double)r / (double)N;
                twa[(size_t)r] = make_float2((float)std::cos(ang), (float)std::sin(ang));
            }
            for (int m = 0; m < 32; ++m) {
                const double ang = -2.0 * M_PI * (double)(128 * m) / (double)N;
                twa[(size_t)128 + m] = make_float2((float)std::cos(ang), (float)std::sin(ang));
            }
            if ((e = dev_alloc(&p->d_twa, sizeof(float2) * twa.size())) != cudaSuccess)
                return bail(alloc_fail(e, "cudaMalloc(split twiddles)"));
            if ((e = cudaMemcpyAsync(p->d_twa, twa.data(), sizeof(float2) * twa.size(), cudaMemcpyHostToDevice,
                                     stream)) != cudaSuccess)
                return bail(cuda_fail(e, "split twiddle upload"));
            if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return bail(cuda_fail(e, "sync"));
        }
        if ((e = cudaMemsetAsync(p->d_err, 0, sizeof(int), stream)) != cudaSuccess)
            return bail(cuda_fail(e, "cudaMemsetAsync"));
        if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return bail(cuda_fail(e, "sync"));
    }

    // step 1: the frequency response
    const int tpb = 256;
    if (coef_kind == FIR_OS_COEF_TIME) {
        double2 *A = nullptr, *B = nullptr;
        cudaError_t e;
        if ((e = dev_alloc(&A, sizeof(double2) * N)) != cudaSuccess ||
            (e = dev_alloc(&B, sizeof(double2) * N)) != cudaSuccess) {
            dev_free(A);
            return bail(alloc_fail(e, "cudaMalloc(plan scratch)"));
        }
        fos_fill_h64<<<(N + tpb - 1) / tpb, tpb, 0, stream>>>(A, coef_dev, M, N, coef_complex);
        for (int Ns = 1; Ns < N; Ns *= 2) {
            fos_radix2_pass64<<<(N / 2 + tpb - 1) / tpb, tpb, 0, stream>>>(A, B, N, Ns);
            double2 *t = A;
            A = B;
            B = t;
        }
        fos_finish_h<<<(N + tpb - 1) / tpb, tpb, 0, stream>>>(A, p->d_H, N);
        e = cudaGetLastError();
        cudaError_t e2 = cudaStreamSynchronize(stream);
        dev_free(A);
        dev_free(B);
        if (e != cudaSuccess) return bail(cuda_fail(e, "frequency-response kernels"));
        if (e2 != cudaSuccess) return bail(cuda_fail(e2, "frequency-response sync"));
    } else {
        fos_scale_h<<<(N + tpb - 1) / tpb, tpb, 0, stream>>>(static_cast<const float2 *>(coef_dev), p->d_H, N);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return bail(cuda_fail(e, "H copy kernel"));
        if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return bail(cuda_fail(e, "H copy sync"));
        if (real) {
            // real data packs two blocks per transform, which needs a real impulse response:
            // H[k] == conj(H[N-k]) within 1e-6 of the largest bin
            std::vector<float2> H((size_t)N);
            if ((e = cudaMemcpy(H.data(), p->d_H, sizeof(float2) * N, cudaMemcpyDeviceToHost)) != cudaSuccess)
                return bail(cuda_fail(e, "H readback"));
            double hmax = 0.0, dev = 0.0;
            for (int k = 0; k < N; ++k) hmax = std::fmax(hmax, std::hypot((double)H[k].x, (double)H[k].y));
            for (int k = 0; k < N; ++k) {
                const float2 a = H[k], b = H[(N - k) % N];
                dev = std::fmax(dev, std::hypot((double)a.x - b.x, (double)a.y + b.y));
            }
            if (dev > 1e-6 * hmax)
                return bail(fail(FIR_OS_E_UNSUPPORTED, "real data needs a Hermitian H (deviation %.3g of max %.3g)",
                                 dev, hmax));
        }
    }
    if (p->kernel.split_c > 0) {
        // the resident kernel reads H[c + C d] for one c at a time: store it c-major
        cudaError_t e = dev_alloc(&p->d_Hk, sizeof(float2) * N);
        if (e != cudaSuccess) return bail(alloc_fail(e, "cudaMalloc(H, c-major)"));
        fos_permute_h<<<(N + tpb - 1) / tpb, tpb, 0, stream>>>(p->d_H, p->d_Hk, N, p->kernel.split_c);
        if ((e = cudaGetLastError()) != cudaSuccess) return bail(cuda_fail(e, "H permute kernel"));
        if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return bail(cuda_fail(e, "H permute sync"));
    }
    (void)rc;
    *out = p;
    return FIR_OS_OK;
}

int fir_os_plan_destroy(fir_os_plan_t plan) {
    if (!plan) return FIR_OS_OK;
    DeviceScope on(plan->device);
    cudaDeviceSynchronize();
    free_plan(plan);
    return FIR_OS_OK;
}

int fir_os_plan_set_wait_limit(fir_os_plan_t plan, int64_t limit_ns) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    if (limit_ns < 0 || limit_ns > 60LL * 1000000000LL)
        return fail(FIR_OS_E_INVAL, "wait limit %lld ns is outside [0, 60 s]", (long long)limit_ns);
    plan->wait_ns = (uint64_t)limit_ns;
    return FIR_OS_OK;
}

int fir_os_plan_set_dft_engine(fir_os_plan_t plan, int engine) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    if (engine != FIR_OS_DFT_FP32 && engine != FIR_OS_DFT_TENSOR)
        return fail(FIR_OS_E_INVAL, "engine %d is neither FIR_OS_DFT_FP32 nor FIR_OS_DFT_TENSOR", engine);
    if (engine == FIR_OS_DFT_TENSOR && !plan->kernel.func_tc)
        return fail(FIR_OS_E_UNSUPPORTED,
                    "the tensor-core DFT engine exists for N = 4096, 16384, 32768 and 65536 (N = %d)", plan->N);
    if (engine == FIR_OS_DFT_TENSOR && !plan->d_btc) {
        int rc = check_device(plan);
        if (rc) return rc;
        // B[c][k], c = 2m + output component, k = 2e + input component, of the 16-point DFT
        // sum_e v[e] W^{em} with W = e^{dir 2 pi i / 16}, split into a TF32 part (low 13 mantissa
        // bits cleared) and the float32 rest, from float64 values; laid out as the tensor cores
        // read a K-major tile (fos_tc.cuh): forward hi, forward lo, inverse hi, inverse lo
        const int per = (int)(fos::kTcBTileBytes / 4);
        std::vector<float> tab((size_t)4 * per, 0.f);
        for (int d = 0; d < 2; ++d) {
            const double dir = d == 0 ? -1.0 : 1.0;
            for (int c = 0; c < 32; ++c)
                for (int k = 0; k < 32; ++k) {
                    const int m = c >> 1, e = k >> 1;
                    const double ang = 2.0 * M_PI * (double)((e * m) % 16) / 16.0;
                    const double cs = std::cos(ang), sn = dir * std::sin(ang);
                    const double val = (c & 1) == 0 ? ((k & 1) == 0 ? cs : -sn) : ((k & 1) == 0 ? sn : cs);
                    float hi = (float)val;
                    uint32_t bits;
                    std::memcpy(&bits, &hi, 4);
                    bits &= 0xFFFFE000u;
                    std::memcpy(&hi, &bits, 4);
                    const float lo = (float)(val - (double)hi);
                    const uint32_t off = fos::tc_offset(c, k) / 4;
                    tab[(size_t)(2 * d) * per + off] = hi;
                    tab[(size_t)(2 * d + 1) * per + off] = lo;
                }
        }
        DeviceScope on(plan->device);
        cudaError_t e = dev_alloc(&plan->d_btc, sizeof(float) * tab.size());
        if (e != cudaSuccess) return alloc_fail(e, "cudaMalloc(tensor-core DFT matrices)");
        if ((e = cudaMemcpy(plan->d_btc, tab.data(), sizeof(float) * tab.size(), cudaMemcpyHostToDevice)) !=
            cudaSuccess) {
            dev_free(plan->d_btc);
            plan->d_btc = nullptr;
            return cuda_fail(e, "tensor-core DFT matrix upload");
        }
        for (const void *f : {plan->kernel.func_tc, plan->kernel.func_multi_tc})
            if (f && (e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               plan->kernel.smem_tc)) != cudaSuccess)
                return cuda_fail(e, "cudaFuncSetAttribute(smem, tensor-core variant)");
    }
    plan->dft_engine = engine;
    return FIR_OS_OK;
}

int fir_os_debug_fail_alloc(int k) {
    if (k < 0) return fail(FIR_OS_E_INVAL, "k = %d < 0", k);
    g_fail_countdown.store(k);
    return FIR_OS_OK;
}

int64_t fir_os_debug_live_allocs(void) { return (int64_t)g_live_allocs.load(); }

int fir_os_plan_info(fir_os_plan_t plan, int *M, int *N, int *L) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    if (M) *M = plan->M;
    if (N) *N = plan->N;
    if (L) *L = plan->L;
    return FIR_OS_OK;
}

int fir_os_plan_kernel(fir_os_plan_t plan, int *kind, int *cluster_size, int *grid, int *smem_bytes) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    if (kind) *kind = plan->kernel.cluster > 1 ? 1 : plan->kernel.split_c > 0 ? 2 : 0;
    if (cluster_size) *cluster_size = plan->kernel.cluster;
    if (grid) *grid = plan->max_units_in_flight * plan->kernel.cluster;
    if (smem_bytes) *smem_bytes = plan->kernel.smem;
    return FIR_OS_OK;
}

int fir_os_execute(fir_os_plan_t plan, const void *x, int64_t n, void *y, void *state, void *stream_) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    if (n < 0) return fail(FIR_OS_E_INVAL, "n_samples < 0");
    if (n == 0) return FIR_OS_OK;
    const int sb = sample_bytes(plan);
    if (!x || !y) return fail(FIR_OS_E_INVAL, "x or y is NULL");
    if (plan->M > 1 && !state) return fail(FIR_OS_E_INVAL, "state is NULL but M > 1");
    const uintptr_t ux = reinterpret_cast<uintptr_t>(x), uy = reinterpret_cast<uintptr_t>(y),
                    us = reinterpret_cast<uintptr_t>(state);
    if ((ux | uy) & (uintptr_t)(sb - 1) || (plan->M > 1 && (us & (uintptr_t)(sb - 1))))
        return fail(FIR_OS_E_ALIGN, "x, y and state must be %d-byte aligned", sb);
    const size_t bytes = (size_t)n * sb, sbytes = (size_t)(plan->M - 1) * sb;
    if (ranges_overlap(ux, bytes, uy, bytes)) return fail(FIR_OS_E_INVAL, "x and y overlap");
    if (ranges_overlap(us, sbytes, ux, bytes) || ranges_overlap(us, sbytes, uy, bytes))
        return fail(FIR_OS_E_INVAL, "state overlaps x or y");
    int rc = check_device(plan);
    if (rc) return rc;
    return launch_blocks(plan, x, n, y, state, static_cast<cudaStream_t>(stream_));
}

int fir_os_execute_batched(fir_os_plan_t plan, const void *x, int64_t x_stride, void *y, int64_t y_stride,
                           void *state, int64_t state_stride, int64_t n, int channels, void *stream_) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    if (n < 0) return fail(FIR_OS_E_INVAL, "n_samples < 0");
    if (channels < 1) return fail(FIR_OS_E_INVAL, "channels must be >= 1");
    if (n == 0) return FIR_OS_OK;
    const int sb = sample_bytes(plan);
    const int hist = plan->M - 1;
    if (!x || !y) return fail(FIR_OS_E_INVAL, "x or y is NULL");
    if (hist > 0 && !state) return fail(FIR_OS_E_INVAL, "state is NULL but M > 1");
    if (channels > 1 && (x_stride < n || y_stride < n || (hist > 0 && state_stride < hist)))
        return fail(FIR_OS_E_INVAL, "strides must be at least n_samples (x, y) and M-1 (state)");
    if (x_stride < 0 || y_stride < 0 || state_stride < 0) return fail(FIR_OS_E_INVAL, "negative stride");
    const uintptr_t ux = reinterpret_cast<uintptr_t>(x), uy = reinterpret_cast<uintptr_t>(y),
                    us = reinterpret_cast<uintptr_t>(state);
    if ((ux | uy) & (uintptr_t)(sb - 1) || (hist > 0 && (us & (uintptr_t)(sb - 1))))
        return fail(FIR_OS_E_ALIGN, "x, y and state must be %d-byte aligned", sb);
    // the whole extents (first to last channel) of x, y and the state must be disjoint
    const size_t xe = ((size_t)(channels - 1) * x_stride + n) * sb, ye = ((size_t)(channels - 1) * y_stride + n) * sb;
    const size_t se = hist > 0 ? ((size_t)(channels - 1) * state_stride + hist) * sb : 0;
    if (ranges_overlap(ux, xe, uy, ye)) return fail(FIR_OS_E_INVAL, "x and y overlap");
    if (ranges_overlap(us, se, ux, xe) || ranges_overlap(us, se, uy, ye))
        return fail(FIR_OS_E_INVAL, "state overlaps x or y");
    int rc = check_device(plan);
    if (rc) return rc;
    return launch_blocks(plan, x, n, y, state, static_cast<cudaStream_t>(stream_), false, channels,
                         channels > 1 ? x_stride : 0, channels > 1 ? y_stride : 0, channels > 1 ? state_stride : 0);
}

int fir_os_launches(fir_os_plan_t plan, int64_t n) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    if (n < 0) return fail(FIR_OS_E_INVAL, "n_samples < 0");
    if (n == 0) return 0;
    return fuse_state(plan, n) ? 1 : 2;
}

int fir_os_device_status(fir_os_plan_t plan, void *stream_) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    int rc = check_device(plan);
    if (rc) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    int flag = 0;
    FOS_CUDA(cudaMemcpyAsync(&flag, plan->d_err, sizeof(int), cudaMemcpyDeviceToHost, stream), "status read");
    FOS_CUDA(cudaMemsetAsync(plan->d_err, 0, sizeof(int), stream), "status clear");
    FOS_CUDA(cudaStreamSynchronize(stream), "status sync");
    if (flag) return fail(FIR_OS_E_DEVICE, "a kernel's bounded wait for a bulk copy ran out");
    return FIR_OS_OK;
}

int fir_os_execute_host(fir_os_plan_t plan, const void *x_host, int64_t n, void *y_host, void *state_host,
                        void *stream_) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    if (n < 0) return fail(FIR_OS_E_INVAL, "n_samples < 0");
    if (plan->M > 1 && !state_host) return fail(FIR_OS_E_INVAL, "state is NULL but M > 1");
    if (n > 0 && (!x_host || !y_host)) return fail(FIR_OS_E_INVAL, "x or y is NULL");
    int rc = check_device(plan);
    if (rc) return rc;
    const int sb = sample_bytes(plan);
    const size_t sbytes = (size_t)(plan->M - 1) * sb;
    if (n > 0 && ranges_overlap(reinterpret_cast<uintptr_t>(x_host), (size_t)n * sb,
                                reinterpret_cast<uintptr_t>(y_host), (size_t)n * sb))
        return fail(FIR_OS_E_INVAL, "x and y overlap");
    cudaStream_t caller = static_cast<cudaStream_t>(stream_);

    // With the block kernel, page-locked buffers are read and written in place over the host link:
    // no staging copies and no pipeline to fill and drain (measured faster than the copy-engine
    // pipeline below, and than copying x in by the copy engine while the kernel writes y in
    // place).  The resident and pair kernels go through the copy-engine pipeline: their gather
    // is point by point, and the pair kernel reads every window twice (once per CTA).
    void *xd = nullptr, *yd = nullptr, *sd = nullptr;
    if (n > 0 && plan->kernel.split_c == 0 && host_mapped(x_host, &xd) && host_mapped(y_host, &yd) &&
        (plan->M == 1 || host_mapped(state_host, &sd))) {
        if ((reinterpret_cast<uintptr_t>(xd) | reinterpret_cast<uintptr_t>(yd)) & (uintptr_t)(sb - 1) ||
            (plan->M > 1 && (reinterpret_cast<uintptr_t>(sd) & (uintptr_t)(sb - 1))))
            return fail(FIR_OS_E_ALIGN, "x, y and state must be %d-byte aligned", sb);
        if (ranges_overlap(reinterpret_cast<uintptr_t>(sd), sbytes, reinterpret_cast<uintptr_t>(xd), (size_t)n * sb) ||
            ranges_overlap(reinterpret_cast<uintptr_t>(sd), sbytes, reinterpret_cast<uintptr_t>(yd), (size_t)n * sb))
            return fail(FIR_OS_E_INVAL, "state overlaps x or y");
        rc = launch_blocks(plan, xd, n, yd, sd, caller, true);
        if (rc) return rc;
        FOS_CUDA(cudaStreamSynchronize(caller), "sync");
        return FIR_OS_OK;
    }

    if (!plan->s_comp) {
        // chunks of about 2^21 samples, a whole number of transforms (blocks, or block pairs for
        // real data), so that chunking changes nothing in what any transform computes
        const int64_t span = (int64_t)plan->L * (plan->data_kind == FIR_OS_REAL ? 2 : 1);
        int64_t chunk = ((int64_t)1 << 21) / span * span;
        if (chunk < span) chunk = span;
        plan->host_chunk = chunk;
        // on any failure everything made so far is released, so a later call starts afresh
        const int st = [&]() -> int {
            cudaError_t e;
            for (int k = 0; k < 2; ++k) {
                if ((e = dev_alloc(&plan->hx[k], (size_t)chunk * sb)) != cudaSuccess ||
                    (e = dev_alloc(&plan->hy[k], (size_t)chunk * sb)) != cudaSuccess)
                    return alloc_fail(e, "cudaMalloc(host path buffers)");
                FOS_CUDA(cudaEventCreateWithFlags(&plan->ev_in[k], cudaEventDisableTiming), "event");
                FOS_CUDA(cudaEventCreateWithFlags(&plan->ev_comp[k], cudaEventDisableTiming), "event");
                FOS_CUDA(cudaEventCreateWithFlags(&plan->ev_out[k], cudaEventDisableTiming), "event");
            }
            if (plan->M > 1 && (e = dev_alloc(&plan->hstate, sbytes)) != cudaSuccess)
                return alloc_fail(e, "cudaMalloc(host path state)");
            FOS_CUDA(cudaEventCreateWithFlags(&plan->ev_start, cudaEventDisableTiming), "event");
            FOS_CUDA(cudaStreamCreateWithFlags(&plan->s_in, cudaStreamNonBlocking), "stream");
            FOS_CUDA(cudaStreamCreateWithFlags(&plan->s_out, cudaStreamNonBlocking), "stream");
            FOS_CUDA(cudaStreamCreateWithFlags(&plan->s_comp, cudaStreamNonBlocking), "stream");
            return FIR_OS_OK;
        }();
        if (st != FIR_OS_OK) {
            release_host_path(plan);
            return st;
        }
        plan->host_chunk = chunk;
    }
    const int64_t chunk = plan->host_chunk;
    FOS_CUDA(cudaEventRecord(plan->ev_start, caller), "event record");
    FOS_CUDA(cudaStreamWaitEvent(plan->s_in, plan->ev_start, 0), "wait");
    FOS_CUDA(cudaStreamWaitEvent(plan->s_comp, plan->ev_start, 0), "wait");
    FOS_CUDA(cudaStreamWaitEvent(plan->s_out, plan->ev_start, 0), "wait");
    if (plan->M > 1)
        FOS_CUDA(cudaMemcpyAsync(plan->hstate, state_host, sbytes, cudaMemcpyHostToDevice, plan->s_comp), "state in");
    const char *xs = static_cast<const char *>(x_host);
    char *ys = static_cast<char *>(y_host);
    int64_t c = 0;
    for (int64_t off = 0; off < n; off += chunk, ++c) {
        const int k = (int)(c & 1);
        const int64_t len = (n - off) < chunk ? (n - off) : chunk;
        if (c >= 2) FOS_CUDA(cudaStreamWaitEvent(plan->s_in, plan->ev_comp[k], 0), "wait");
        FOS_CUDA(cudaMemcpyAsync(plan->hx[k], xs + off * sb, (size_t)len * sb, cudaMemcpyHostToDevice, plan->s_in),
                 "chunk in");
        FOS_CUDA(cudaEventRecord(plan->ev_in[k], plan->s_in), "event record");
        FOS_CUDA(cudaStreamWaitEvent(plan->s_comp, plan->ev_in[k], 0), "wait");
        if (c >= 2) FOS_CUDA(cudaStreamWaitEvent(plan->s_comp, plan->ev_out[k], 0), "wait");
        rc = launch_blocks(plan, plan->hx[k], len, plan->hy[k], plan->hstate, plan->s_comp);
        if (rc) return rc;
        FOS_CUDA(cudaEventRecord(plan->ev_comp[k], plan->s_comp), "event record");
        FOS_CUDA(cudaStreamWaitEvent(plan->s_out, plan->ev_comp[k], 0), "wait");
        FOS_CUDA(cudaMemcpyAsync(ys + off * sb, plan->hy[k], (size_t)len * sb, cudaMemcpyDeviceToHost, plan->s_out),
                 "chunk out");
        FOS_CUDA(cudaEventRecord(plan->ev_out[k], plan->s_out), "event record");
    }
    if (plan->M > 1)
        FOS_CUDA(cudaMemcpyAsync(state_host, plan->hstate, sbytes, cudaMemcpyDeviceToHost, plan->s_comp), "state out");
    FOS_CUDA(cudaStreamSynchronize(plan->s_in), "sync");
    FOS_CUDA(cudaStreamSynchronize(plan->s_comp), "sync");
    FOS_CUDA(cudaStreamSynchronize(plan->s_out), "sync");
    return FIR_OS_OK;
}

int fir_os_fp32_probe(int iters, void *stream_, double *flops) {
    if (iters < 1 || !flops) return fail(FIR_OS_E_INVAL, "iters must be >= 1 and flops non-NULL");
    int dev = 0, sms = 0, per_sm = 0;
    FOS_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    FOS_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "device attribute");
    FOS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fos_fp32_probe_kernel, 1024, 0),
             "occupancy query");
    if (per_sm < 1) per_sm = 1;
    const int grid = sms * per_sm;
    fos_fp32_probe_kernel<<<grid, 1024, 0, static_cast<cudaStream_t>(stream_)>>>(nullptr, iters);
    FOS_CUDA(cudaGetLastError(), "probe launch");
    *flops = 2.0 * 8.0 * 1024.0 * (double)grid * (double)iters;
    return FIR_OS_OK;
}

int fir_os_frequency_response_noalloc(const void *h_dev, int M, int N, int h_complex, void *H_dev,
                                      void *stream_) {
    if (!h_dev || !H_dev) return fail(FIR_OS_E_INVAL, "h or H is NULL");
    if (N > kNoallocMaxN)
        return fail(FIR_OS_E_UNSUPPORTED, "N = %d exceeds the %d points the static scratch holds", N, kNoallocMaxN);
    if (N < 64 || (N & (N - 1)) != 0)
        return fail(FIR_OS_E_UNSUPPORTED, "N = %d is not a power of two in [64, %d]", N, kNoallocMaxN);
    if (M < 1 || M > N) return fail(FIR_OS_E_UNSUPPORTED, "M = %d must be in [1, N = %d]", M, N);
    if (h_complex != 0 && h_complex != 1) return fail(FIR_OS_E_INVAL, "h_complex must be 0 or 1");
    if (reinterpret_cast<uintptr_t>(h_dev) & (h_complex ? 7 : 3))
        return fail(FIR_OS_E_ALIGN, "h must be naturally aligned");
    if (reinterpret_cast<uintptr_t>(H_dev) & 7) return fail(FIR_OS_E_ALIGN, "H must be 8-byte aligned");
    double2 *scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    double2 *A = scratch, *B = scratch + kNoallocMaxN;
    const int tpb = 256;
    // every entry of A[0..N) is written here, so nothing left by an earlier call is read
    fos_fill_h64<<<(N + tpb - 1) / tpb, tpb, 0, stream>>>(A, h_dev, M, N, h_complex);
    for (int Ns = 1; Ns < N; Ns *= 2) {
        fos_radix2_pass64<<<(N / 2 + tpb - 1) / tpb, tpb, 0, stream>>>(A, B, N, Ns);
        double2 *t = A;
        A = B;
        B = t;
    }
    fos_store_h<<<(N + tpb - 1) / tpb, tpb, 0, stream>>>(A, static_cast<float2 *>(H_dev), N);
    FOS_CUDA(cudaGetLastError(), "frequency-response kernels");
    return FIR_OS_OK;
}

// ------------------------------------------------------------------ channelizer

struct fir_chan_plan {
    int K = 0, D = 0, Nh = 0, P = 0;
    int data_kind = FIR_OS_REAL;
    int device = 0;
    int smem = 0;
    int max_ctas = 0;
    fos::ChanEntry kernel;
    float *d_h = nullptr;
    float2 *d_tw = nullptr;
};

int fir_chan_plan_destroy(fir_chan_plan_t plan) {
    if (!plan) return FIR_OS_OK;
    DeviceScope on(plan->device);
    cudaDeviceSynchronize();
    dev_free(plan->d_h);
    dev_free(plan->d_tw);
    alloc_give(plan);
    return FIR_OS_OK;
}

int fir_chan_plan_create(fir_chan_plan_t *out, int K, int D, int Nh, int data_kind, const float *h_dev,
                         void *stream_) {
    g_last_error[0] = 0;
    if (!out) return fail(FIR_OS_E_INVAL, "out is NULL");
    *out = nullptr;
    if (K < 64 || K > 4096 || (K & (K - 1)) != 0)
        return fail(FIR_OS_E_UNSUPPORTED, "K = %d is not a power of two in [64, 4096]", K);
    if (D < 1 || D > K) return fail(FIR_OS_E_INVAL, "D = %d must be in [1, K = %d]", D, K);
    if (Nh < 1) return fail(FIR_OS_E_INVAL, "Nh = %d < 1", Nh);
    if (data_kind != FIR_OS_REAL && data_kind != FIR_OS_COMPLEX)
        return fail(FIR_OS_E_INVAL, "data_kind %d is neither FIR_OS_REAL nor FIR_OS_COMPLEX", data_kind);
    if (!h_dev) return fail(FIR_OS_E_INVAL, "h is NULL");
    if (reinterpret_cast<uintptr_t>(h_dev) & 3) return fail(FIR_OS_E_ALIGN, "h must be 4-byte aligned");
    const int logk = ilog2i(K);
    fos::ChanEntry k = fos::chan_kernel(logk, data_kind == FIR_OS_REAL);
    if (!k.func) return fail(FIR_OS_E_UNSUPPORTED, "no channelizer kernel for K = %d", K);
    const int P = (Nh + K - 1) / K;
    const int smem = k.smem_fixed + 4 * P * K;
    int dev = 0;
    FOS_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    cudaDeviceProp prop;
    FOS_CUDA(cudaGetDeviceProperties(&prop, dev), "cudaGetDeviceProperties");
    if (!(prop.major == 10 && prop.minor == 3))
        return fail(FIR_OS_E_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev, prop.major,
                    prop.minor);
    if (smem > (int)prop.sharedMemPerBlockOptin)
        return fail(FIR_OS_E_UNSUPPORTED, "a prototype of %d taps (%d per branch) does not fit shared memory "
                                          "with K = %d (at most %d taps)",
                    Nh, P, K, (int)((prop.sharedMemPerBlockOptin - k.smem_fixed) / (4 * K)) * K);
    fir_chan_plan *p = alloc_take<fir_chan_plan>();
    if (!p) return fail(FIR_OS_E_NOMEM, "plan allocation failed");
    auto bail = [&](int status) {
        fir_chan_plan_destroy(p);
        return status;
    };
    p->K = K;
    p->D = D;
    p->Nh = Nh;
    p->P = P;
    p->data_kind = data_kind;
    p->device = dev;
    p->smem = smem;
    p->kernel = k;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    cudaError_t e = cudaFuncSetAttribute(k.func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaFuncSetAttribute(smem)"));
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.func, k.threads, (size_t)smem);
    if (e != cudaSuccess) return bail(cuda_fail(e, "occupancy query"));
    if (per_sm < 1) return bail(fail(FIR_OS_E_UNSUPPORTED, "channelizer kernel does not fit an SM"));
    p->max_ctas = per_sm * prop.multiProcessorCount;
    std::vector<float2> tw;
    if (!pass_twiddles(logk, tw)) return bail(fail(FIR_OS_E_UNSUPPORTED, "twiddles"));
    if ((e = dev_alloc(&p->d_tw, sizeof(float2) * tw.size())) != cudaSuccess ||
        (e = dev_alloc(&p->d_h, sizeof(float) * (size_t)P * K)) != cudaSuccess)
        return bail(alloc_fail(e, "cudaMalloc(channelizer tables)"));
    // the prototype zero-padded to P K taps, so that the kernel reads it in whole 16-byte pieces
    if ((e = cudaMemcpyAsync(p->d_tw, tw.data(), sizeof(float2) * tw.size(), cudaMemcpyHostToDevice, stream)) !=
            cudaSuccess ||
        (e = cudaMemsetAsync(p->d_h, 0, sizeof(float) * (size_t)P * K, stream)) != cudaSuccess ||
        (e = cudaMemcpyAsync(p->d_h, h_dev, sizeof(float) * Nh, cudaMemcpyDeviceToDevice, stream)) != cudaSuccess)
        return bail(cuda_fail(e, "plan upload"));
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return bail(cuda_fail(e, "sync"));
    *out = p;
    return FIR_OS_OK;
}

int fir_chan_plan_info(fir_chan_plan_t plan, int *K, int *D, int *Nh) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    if (K) *K = plan->K;
    if (D) *D = plan->D;
    if (Nh) *Nh = plan->Nh;
    return FIR_OS_OK;
}

int fir_chan_execute(fir_chan_plan_t plan, const void *x, int64_t n, void *y, void *state, void *stream_) {
    if (!plan) return fail(FIR_OS_E_INVAL, "plan is NULL");
    if (n < 0) return fail(FIR_OS_E_INVAL, "n_samples < 0");
    if (n % plan->D) return fail(FIR_OS_E_INVAL, "n_samples = %lld is not a multiple of D = %d", (long long)n, plan->D);
    if (n == 0) return FIR_OS_OK;
    const int sb = plan->data_kind == FIR_OS_REAL ? 4 : 8;
    const int hist = plan->Nh - 1;
    if (!x || !y) return fail(FIR_OS_E_INVAL, "x or y is NULL");
    if (hist > 0 && !state) return fail(FIR_OS_E_INVAL, "state is NULL but Nh > 1");
    const uintptr_t ux = reinterpret_cast<uintptr_t>(x), uy = reinterpret_cast<uintptr_t>(y),
                    us = reinterpret_cast<uintptr_t>(state);
    if ((ux & (uintptr_t)(sb - 1)) || (uy & 7) || (hist > 0 && (us & (uintptr_t)(sb - 1))))
        return fail(FIR_OS_E_ALIGN, "x and the state must be %d-byte aligned, y 8-byte aligned", sb);
    const int64_t nout = n / plan->D;
    const size_t xb = (size_t)n * sb, yb = (size_t)nout * plan->K * 8, stb = (size_t)hist * sb;
    if (ranges_overlap(ux, xb, uy, yb)) return fail(FIR_OS_E_INVAL, "x and y overlap");
    if (ranges_overlap(us, stb, ux, xb) || ranges_overlap(us, stb, uy, yb))
        return fail(FIR_OS_E_INVAL, "state overlaps x or y");
    int dev = -1;
    FOS_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev != plan->device)
        return fail(FIR_OS_E_INVAL, "plan was created on device %d but device %d is current", plan->device, dev);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    fos::ChanParams cp{};
    cp.x = x;
    cp.y = static_cast<float2 *>(y);
    cp.state = state;
    cp.h = plan->d_h;
    cp.tw = plan->d_tw;
    cp.nout = nout;
    // Real input shares a transform between two output vectors (2i, 2i + 1 of the call) when
    // the call fills every transform slot of the device at least twice over without that, and
    // with K = 2D a slot takes four vectors (two transforms) when it fills them four times over;
    // shorter calls are latency-bound and keep one vector per transform.  All three give the
    // same pairs, so only the unpacked choice changes rounding.
    const int64_t per_wave = (int64_t)plan->max_ctas * plan->kernel.groups * plan->kernel.per_unit;
    cp.pack = 0;
    if (plan->data_kind == FIR_OS_REAL && nout >= 2 * per_wave)
        cp.pack = plan->K == 2 * plan->D && nout >= 4 * per_wave ? 2 : 1;
    const int64_t per_unit = (int64_t)plan->kernel.per_unit * (cp.pack == 2 ? 4 : cp.pack == 1 ? 2 : 1);
    cp.nunits = (nout + per_unit - 1) / per_unit;
    cp.K = plan->K;
    cp.D = plan->D;
    cp.Nh = plan->Nh;
    cp.P = plan->P;
    // one CTA per unit up to one per SM: the kernel deals units across CTAs first
    const int64_t grid = cp.nunits < plan->max_ctas ? cp.nunits : plan->max_ctas;
    void *args[] = {&cp};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(plan->kernel.threads);
    cfg.dynamicSmemBytes = (size_t)plan->smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    FOS_CUDA(cudaLaunchKernelExC(&cfg, plan->kernel.func, args), "channelizer launch");
    if (hist > 0) {
        // S0' = the last Nh - 1 samples of concat(S0, x), after the filter bank has read S0
        FOS_CUDA(plan->data_kind == FIR_OS_REAL ? launch_state<float>(x, n, state, hist, 0, 0, 1, stream)
                                                : launch_state<float2>(x, n, state, hist, 0, 0, 1, stream),
                 "state kernel launch");
    }
    return FIR_OS_OK;
}

}  // extern "C"
