/*
 * fir_os.h -- C ABI of libfir_os.so: high-order FIR filtering by the frequency-domain
 * overlap-save method on one GB300 (sm_103a).
 *
 * The method is the one claimed in "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法"
 * (zl.czvv.com/42398539.html), 主权项 steps 1-6:
 *   step 1  an M-tap impulse response h is zero-padded to N and transformed, H = FFT_N(h),
 *           or the N-point response H is given directly;
 *   step 2  the input is cut into blocks B_i of L = N - M + 1 samples;
 *   step 3  each block is extended by the M-1 samples before it, E_0 = {S0, B_0},
 *           E_i = {D_{i-1}, B_i}, and the newest M-1 samples are carried as the next S0;
 *   step 4  R_i = IFFT(FFT(E_i) * H);
 *   step 5  the first M-1 samples of each R_i are dropped, Y_i = R_i[M-1 .. M-1+L);
 *   step 6  the caller repeats with the next chunk of input.
 * Together these compute, for every output j of a call,
 *       y[j] = sum_{m=0}^{M-1} h[m] * xt[j-m],   xt[t] = x[t] (t >= 0), S0[M-1+t] (t < 0),
 * a linear convolution continued seamlessly across calls.
 *
 * Conventions: the forward transform is e^{-2 pi i nk/N} unscaled and the inverse is
 * e^{+2 pi i nk/N} scaled by 1/N; a given H is therefore the unscaled FFT of the taps.
 * Samples are float32 (real data) or interleaved float32 (re, im) pairs (complex64).
 * All arithmetic on the device is float32.
 *
 * Errors: every entry point returns FIR_OS_OK (0) or a negative status; no call throws,
 * traps on the device or aborts.  Arguments are validated on the host before anything is
 * enqueued.  fir_os_last_error() gives a one-line description of the last failure on the
 * calling thread.
 *
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 * Device work is enqueued asynchronously on it unless stated otherwise.
 */
#ifndef FIR_OS_H
#define FIR_OS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define FIR_OS_OK 0
#define FIR_OS_E_INVAL (-1)       /* null pointer, bad size, overlapping buffers, bad kind */
#define FIR_OS_E_UNSUPPORTED (-2) /* N not a power of two in [64, 65536], M > N, real data
                                     with a complex or non-Hermitian response, no device */
#define FIR_OS_E_ALIGN (-3)       /* a buffer without the alignment stated below */
#define FIR_OS_E_NOMEM (-4)       /* device or host allocation failed */
#define FIR_OS_E_CUDA (-5)        /* a CUDA runtime call or a launch failed */
#define FIR_OS_E_DEVICE (-6)      /* a kernel reported a bounded wait that ran out */

/* data kinds */
#define FIR_OS_REAL 0    /* x, y, state: float32 */
#define FIR_OS_COMPLEX 1 /* x, y, state: complex64 (float32 re, im interleaved) */

/* coefficient kinds */
#define FIR_OS_COEF_TIME 0 /* coef = h, M taps (step 1, first case) */
#define FIR_OS_COEF_FREQ 1 /* coef = H, N bins of complex64 (step 1, second case) */

typedef struct fir_os_plan *fir_os_plan_t;
typedef struct fir_chan_plan *fir_chan_plan_t;

/*
 * fir_os_plan_create -- step 1: build the frequency response and everything the block
 * kernels need for one (M, N, data kind) combination.
 *
 *   out          receives the plan handle (set to NULL on failure)
 *   M            taps, 1 <= M <= N
 *   N            FFT size, a power of two in [64, 65536]; the block length is L = N - M + 1
 *   data_kind    FIR_OS_REAL or FIR_OS_COMPLEX (the x / y / state sample type)
 *   coef_kind    FIR_OS_COEF_TIME: coef_dev holds h[0..M-1]; H = FFT_N(h zero-padded to N)
 *                is computed on the device in float64 and rounded to complex64.
 *                FIR_OS_COEF_FREQ: coef_dev holds H[0..N-1] (complex64) and must be
 *                16-byte aligned (the claim stores H at an address that is a multiple of
 *                the memory width); it is copied.
 *   coef_complex for COEF_TIME: 0 = h is float32, 1 = h is complex64.  Ignored for FREQ.
 *                Real data needs a real h, or (FREQ) an H that is Hermitian within 1e-6 of
 *                its largest bin; otherwise FIR_OS_E_UNSUPPORTED.
 *   coef_dev     device pointer, owned by the caller; it may be freed once this returns
 *   stream       the plan-time kernels run on it; the call synchronises it before returning
 *
 * The plan owns its device memory (H scaled by 1/N, twiddle tables, an error word) and
 * keeps the device that was current at creation; later calls must be made with that
 * device current.
 */
int fir_os_plan_create(fir_os_plan_t *out, int M, int N, int data_kind, int coef_kind,
                       int coef_complex, const void *coef_dev, void *stream);

/*
 * fir_os_execute -- steps 2-5 for one chunk of n_samples input samples, asynchronously on
 * `stream`.
 *
 *   x_dev      n_samples input samples (device), naturally aligned (4 B real, 8 B complex)
 *   n_samples  >= 0; 0 is a no-op.  Need not be a multiple of L: the last block is
 *              zero-padded past the input and only n_samples outputs are written.
 *   y_dev      n_samples output samples (device), same type and alignment as x; must not
 *              overlap x or the state
 *   state_dev  M-1 samples (device, oldest first) holding S0 on entry and, in stream order
 *              after the call, the newest M-1 samples of concat(S0, x): the next call's S0.
 *              Zero it before the first call of a stream.  May be NULL only when M == 1.
 *
 * Returns after enqueueing; y and the state are valid in stream order.  Concurrent calls
 * that share a state buffer must be serialised by the caller.  A device-side wait that
 * ran out is reported later by fir_os_device_status().
 */
int fir_os_execute(fir_os_plan_t plan, const void *x_dev, int64_t n_samples, void *y_dev,
                   void *state_dev, void *stream);

/*
 * fir_os_execute_batched -- fir_os_execute over `channels` independent streams that share the
 * plan's filter, in one launch (a bank of identical filters: the channels of an array, a
 * multi-channel recording).  The method's page filters one stream; each channel here is
 * filtered exactly as fir_os_execute filters it (steps 3-5 and the state carry of the claim in
 * "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法", 主权项).
 *
 *   x, y           device memory; channel c's n_samples samples start at x + c * x_stride and
 *                  y + c * y_stride (strides in samples, >= n_samples when channels > 1)
 *   state          device memory; channel c's M-1 samples (in/out, oldest first) start at
 *                  state + c * state_stride (stride >= M-1 when channels > 1); NULL only if M == 1
 *   n_samples      per channel, >= 0 (0 is a no-op)
 *   channels       >= 1
 *   stream         as for fir_os_execute
 *
 * Returns FIR_OS_E_INVAL for channels < 1, short or negative strides, or when the extents of x,
 * y and the state (first to last channel) overlap; FIR_OS_E_ALIGN as fir_os_execute.  Every
 * channel's output and state equal those of fir_os_execute on that channel alone, bit for bit.
 */
int fir_os_execute_batched(fir_os_plan_t plan, const void *x, int64_t x_stride, void *y,
                           int64_t y_stride, void *state, int64_t state_stride, int64_t n_samples,
                           int channels, void *stream);

/*
 * fir_os_execute_host -- the same filtering for input and output in HOST memory: step 2
 * and step 6 of the claim (move a chunk to the GPU, filter it, move the result back, repeat
 * while data remains).  Synchronous: returns when y_host and state_host hold the results.
 *
 *   x_host, y_host   n_samples samples each, host memory
 *   state_host       M-1 samples in/out (host), as for fir_os_execute; NULL only if M == 1
 *   stream           the caller's stream; work is ordered after it and it is synchronised
 *
 * When x, y and the state are all page-locked (cudaHostAlloc / cudaHostRegister, e.g. torch
 * pin_memory) and N <= 8192, the kernel reads x and writes y and the state in place over the
 * host link: no staging copies.  Otherwise the call copies chunks of about 2^21 samples (a whole number of
 * transforms -- blocks, or block pairs for real data -- so the chunks cut the stream where one
 * fir_os_execute call's transforms begin) through two device buffer sets, pipelined over three
 * streams so that the copies of one chunk overlap the filtering of the next; the plan allocates
 * those buffers on first use and keeps them until fir_os_plan_destroy.  Either way the results
 * equal fir_os_execute's, bit for bit.
 */
int fir_os_execute_host(fir_os_plan_t plan, const void *x_host, int64_t n_samples,
                        void *y_host, void *state_host, void *stream);

/* fir_os_fp32_probe -- a measurement aid, not a step of the method: enqueues on `stream` one
 * kernel of independent float32 multiply-add chains (eight per thread, 1024 threads per CTA, as
 * many CTAs as are resident on every SM at once) running `iters` iterations, for measuring the
 * FP32 peak that the filter's arithmetic roofline is taken against.  The caller times it (for
 * example with events on `stream`).  *flops receives the floating-point operations the kernel
 * performs (two per multiply-add).  FIR_OS_E_INVAL for iters < 1 or flops NULL. */
int fir_os_fp32_probe(int iters, void *stream, double *flops);

/* fir_os_plan_destroy -- synchronises the plan's device (made current for the call; the
 * caller's current device is restored) and frees the plan.  NULL is a no-op. */
int fir_os_plan_destroy(fir_os_plan_t plan);

/* fir_os_plan_info -- M, N and L = N - M + 1 of a plan (any output pointer may be NULL). */
int fir_os_plan_info(fir_os_plan_t plan, int *M, int *N, int *L);

/* fir_os_plan_kernel -- which block kernel a plan launches: 0 = one CTA per block group
 * (N <= 8192), 1 = a two-CTA cluster per block, half of it in each SM's Tensor Memory
 * (N = 65536), 2 = one block resident in one SM's Tensor Memory (N = 16384, 32768).
 * *cluster_size is 1 or
 * the cluster's CTA count; *grid the CTAs one launch uses; *smem_bytes the dynamic shared
 * memory per CTA.  Any output pointer may be NULL. */
int fir_os_plan_kernel(fir_os_plan_t plan, int *kind, int *cluster_size, int *grid,
                       int *smem_bytes);

/* fir_os_launches -- how many kernels one fir_os_execute call of n_samples launches: 0 for
 * n_samples == 0, else 1 (the fused block kernel, which also writes the new state) or 2 (the
 * block kernel and a one-CTA state kernel, when more than one work unit reads S0).
 * Returns a negative status for a bad plan or n_samples < 0. */
int fir_os_launches(fir_os_plan_t plan, int64_t n_samples);

/* fir_os_device_status -- synchronises `stream`, then reads and clears the plan's device
 * error word: FIR_OS_OK, or FIR_OS_E_DEVICE if a kernel's bounded wait ran out since the
 * last check. */
int fir_os_device_status(fir_os_plan_t plan, void *stream);

/* fir_os_plan_set_wait_limit -- the longest a kernel of this plan waits for one bulk copy of
 * its input window (step 3 of the claim, the overlap gather, which the N <= 8192 kernels stage
 * into shared memory by bulk copies) before it gives up on that copy: 1 s by default.  A wait
 * that runs out sets the plan's error word (fir_os_device_status then returns FIR_OS_E_DEVICE);
 * the kernel lets that copy land (a second wait of at most 1 s) and gathers the window, and
 * every later one of the same launch, with plain loads instead, so the outputs are still
 * correct.  limit_ns = 0 makes every such wait run out at once -- a way to run the fallback
 * on a healthy device; the N >= 16384 kernels have no such waits.  Applies to launches
 * enqueued after the call.  FIR_OS_E_INVAL for a NULL plan or a limit outside [0, 60 s]. */
int fir_os_plan_set_wait_limit(fir_os_plan_t plan, int64_t limit_ns);

/* fir_os_plan_set_dft_engine -- how the 16-point DFTs of the plan's radix-16 transform passes
 * (step 4 of the claim: the FFT and IFFT of every block) are computed:
 *   FIR_OS_DFT_FP32    (default) as butterflies in float32 registers;
 *   FIR_OS_DFT_TENSOR  as matrix products on the tensor cores: 128 vectors per tcgen05.mma tile,
 *                      TF32 operands split into a TF32 part and the float32 rest (three products,
 *                      float32 accumulation in Tensor Memory), the twiddles still in float32.
 * The tensor engine exists for N = 4096 (every pass of the block transform) and for N = 16384,
 * 32768 and 65536 (every pass of their 4096-point sub-transforms; FIR_OS_E_UNSUPPORTED for the
 * other sizes); it is an option, off by default.  Its outputs meet the same parity bar but are not bitwise equal to
 * the default's.  The first
 * FIR_OS_DFT_TENSOR call allocates and uploads the 16 KB of split DFT matrices (synchronous;
 * FIR_OS_E_NOMEM if that allocation fails).  Applies to launches enqueued after the call.
 * FIR_OS_E_INVAL for a NULL plan or an unknown engine. */
#define FIR_OS_DFT_FP32 0
#define FIR_OS_DFT_TENSOR 1
int fir_os_plan_set_dft_engine(fir_os_plan_t plan, int engine);

/* fir_os_debug_fail_alloc -- make the k-th next allocation of the library (its plan objects
 * and the device buffers of fir_os_plan_create, fir_chan_plan_create and the first
 * fir_os_execute_host call) fail as if memory had run out, without asking CUDA; k = 0
 * disarms.  The failing call returns FIR_OS_E_NOMEM and releases everything it had allocated.
 * A process-wide host-side test hook (not for concurrent use) for the library's own error
 * paths; the claim has no counterpart.  FIR_OS_E_INVAL for k < 0. */
int fir_os_debug_fail_alloc(int k);

/* fir_os_debug_live_allocs -- the number of the library's allocations (plan objects and device
 * buffers) alive now, process-wide; with fir_os_debug_fail_alloc it shows that a failed call
 * left nothing behind.  A test aid; the claim has no counterpart. */
int64_t fir_os_debug_live_allocs(void);

/*
 * fir_os_frequency_response_noalloc -- H = FFT_N(h zero-padded to N), the unscaled
 * complex64 response that fir_os_plan_create accepts as FIR_OS_COEF_FREQ, computed on the
 * device in float64 without allocating any memory.  The paper has no counterpart of this
 * entry point; it exists for callers that must not allocate device memory at the point where
 * they build a response: code whose device memory is handed out entirely by its own pool,
 * real-time threads that cannot afford an allocation's unbounded latency, or a process that
 * is at its memory limit.  fir_os_plan_create needs float64 working buffers for the same
 * transform and allocates them; this call uses a fixed 2 MiB array in the library's device
 * image instead.  CUDA allocates that array on a device when the library's device code is
 * loaded there (with lazy module loading, the default: at the library's first kernel launch or
 * symbol lookup on that device, which may be this call's), and holds it until the process
 * exits; so make one call (or create a plan) early, outside stream capture and away from the
 * device's memory limit.  If loading runs out of memory the call returns FIR_OS_E_NOMEM.
 *
 *   h_dev      M taps (device): float32 if h_complex == 0, complex64 if 1, naturally aligned
 *   M          1 <= M <= N
 *   N          a power of two in [64, 65536]; larger N is rejected (FIR_OS_E_UNSUPPORTED)
 *              because the fixed array holds two 65536-point float64 buffers and no more
 *   H_dev      N complex64 bins (device, 8-byte aligned; 16-byte aligned if it is to be
 *              passed to fir_os_plan_create), written in stream order
 *   stream     the kernels are enqueued on it asynchronously
 *
 * Calls no cudaMalloc, cudaFree or other allocating routine.  The first call on a device
 * looks up the device address of the fixed array (once per device, with that device
 * current); make that first call before any stream capture.  All calls share the one array
 * and leave their intermediate values in it; each call rewrites every entry it reads, but
 * calls whose kernels overlap on the GPU (different streams, or different host threads
 * without ordering) race on the array and must be serialised by the caller.
 */
int fir_os_frequency_response_noalloc(const void *h_dev, int M, int N, int h_complex,
                                      void *H_dev, void *stream);

/* fir_os_choose_n -- the FFT size for an M-tap filter: the power of two N in [max(64, M), 65536]
 * with the highest predicted throughput, and that throughput (output samples per second / 1e9)
 * in *gsps (may be NULL).  The claim of "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法"
 * (主权项, 步骤二) leaves N free beyond N = L + M - 1; a longer N spends more transform work per
 * block on more outputs per block.  The prediction is L x sms / t(N, L/N): t is the device time
 * of one block in SM-microseconds, measured on a GB300 for every N at L/N = 1/4, 1/2, 3/4 in
 * large calls and interpolated linearly in L/N.  sms = 0 means the GB300's 152.  Host-only: no
 * device call.  FIR_OS_E_INVAL for M < 1, a bad data_kind or sms < 0; FIR_OS_E_UNSUPPORTED for
 * M > 65536. */
int fir_os_choose_n(int M, int data_kind, int sms, int *N, double *gsps);

/* fir_os_predict_gsps -- the prediction fir_os_choose_n maximises, for one (M, N).  Errors as
 * fir_os_plan_create's for N and M. */
int fir_os_predict_gsps(int M, int N, int data_kind, int sms, double *gsps);

/* ---------------------------------------------------------------------------------------
 * Polyphase DFT channelizer ("GPU加速短波信道化：多相滤波器组的并行重构与CUDA实现", sections 2-3):
 * K channels of a real lowpass prototype h (Nh taps) modulated to the K frequencies q / K and
 * decimated by D (D = K/2 for the page's 50%-overlapping channels),
 *
 *   y[m][q] = sum_{l < Nh} h[l] e^{-2 pi i q l / K} xt[m D + D - 1 - l],
 *
 * computed by the page's three steps: input dealt into K branches, each branch filtered by its
 * polyphase component h[r K + k], a K-point DFT across the branches.  xt is x preceded by the
 * state (Nh - 1 samples, oldest first, carried from call to call like fir_os_execute's).
 */

/* fir_chan_plan_create -- K a power of two in [64, 4096]; 1 <= D <= K; Nh >= 1 with
 * ceil(Nh / K) K taps fitting shared memory (FIR_OS_E_UNSUPPORTED otherwise; the message gives
 * the limit, 20 K taps at K = 1024); data_kind FIR_OS_REAL (float32 x) or FIR_OS_COMPLEX
 * (complex64 x); h_dev: Nh float32 taps in device memory, 4-byte aligned, copied into the plan
 * (the call synchronises `stream`, so h_dev may be freed afterwards).  Errors as
 * fir_os_plan_create's. */
int fir_chan_plan_create(fir_chan_plan_t *out, int K, int D, int Nh, int data_kind, const float *h_dev,
                         void *stream);

/* fir_chan_execute -- one call over n_samples input samples, asynchronous on `stream`.
 *   x       device memory, n_samples samples (float32 or complex64), naturally aligned
 *   y       device memory, (n_samples / D) x K complex64 outputs, y[m K + q], 8-byte aligned
 *   state   device memory, Nh - 1 samples in/out (NULL only if Nh == 1); zero it before the
 *           first call of a stream
 * n_samples must be a multiple of D (FIR_OS_E_INVAL otherwise); 0 is a no-op.  x, y and the
 * state must not overlap (FIR_OS_E_INVAL).  Launches the channelizer kernel and, when Nh > 1,
 * a one-CTA kernel that writes the new state.  Real input: a call of at least
 * 2 x SMs x 8192 / K output vectors (2432 at K = 1024 on 152 SMs) shares one complex
 * transform between its output vectors 2i and 2i + 1 (with K = 2D and twice that many vectors,
 * one thread computes the branch sums of two such transforms, with the same results); shorter
 * calls transform each vector alone.  A stream split into calls gives one call's output bit
 * for bit when every call makes the same choice between shared and single transforms and,
 * for shared ones, starts on an even vector; otherwise the results differ in rounding only. */
int fir_chan_execute(fir_chan_plan_t plan, const void *x, int64_t n_samples, void *y, void *state,
                     void *stream);

/* fir_chan_plan_info -- K, D and Nh of a channelizer plan (any output may be NULL). */
int fir_chan_plan_info(fir_chan_plan_t plan, int *K, int *D, int *Nh);

/* fir_chan_plan_destroy -- synchronises the plan's device (made current for the call; the
 * caller's current device is restored) and frees the plan.  NULL is a no-op. */
int fir_chan_plan_destroy(fir_chan_plan_t plan);

/* fir_os_status_string -- a static description of a status code. */
const char *fir_os_status_string(int status);

/* fir_os_last_error -- the calling thread's description of its last failed call (static
 * storage, overwritten by the next failure; "" if none). */
const char *fir_os_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FIR_OS_H */
