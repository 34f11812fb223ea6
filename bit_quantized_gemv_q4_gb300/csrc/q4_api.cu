// C ABI entry points for the GEMV calls, the thread-local error text and the
// per-device state (BaseRT: optimal LLM inference on Apple Silicon with native
// Metal, §3 "BaseRT runtime design": a C API over the runtime; §3.2
// "Zero-allocation decode loop": error handling through static thread-local
// buffers, nothing allocated on a hot call).
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "q4_internal.h"

// Device error word: bits latched by kernels (timeouts, failed device-side
// checks), read and cleared by q4_device_status.  One per device that loads
// the library; its address is taken once per device.
__device__ int q4_device_error_word;

namespace q4i {

namespace {
thread_local char t_error[512];

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices];
}  // namespace

void clear_error() { t_error[0] = '\0'; }

q4_status fail(q4_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_error, sizeof(t_error), fmt, ap);
    va_end(ap);
    return s;
}

q4_status cuda_fail(cudaError_t e, const char* what) {
    return fail(Q4_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

q4_status current_device(const DeviceInfo** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0) return fail(Q4_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    if (dev >= kMaxDevices) return fail(Q4_ERR_NO_DEVICE, "device ordinal %d too large", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ready[dev]) {
        DeviceInfo d;
        d.device = dev;
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (d.cc_major != 10 || d.cc_minor != 3)
            return fail(Q4_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                        d.cc_major, d.cc_minor);
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, q4_device_error_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(q4_device_error_word)");
        d.err_word = static_cast<int*>(p);
        g_dev[dev] = d;
        g_dev_ready[dev] = true;
    }
    *out = &g_dev[dev];
    return Q4_OK;
}

}  // namespace q4i

using namespace q4i;

extern "C" {

const char* q4_last_error(void) { return t_error; }

const char* q4_status_string(q4_status s) {
    switch (s) {
        case Q4_OK: return "ok";
        case Q4_ERR_INVALID_ARG: return "invalid argument";
        case Q4_ERR_UNSUPPORTED: return "unsupported";
        case Q4_ERR_MISALIGNED: return "misaligned pointer or leading dimension";
        case Q4_ERR_CUDA: return "CUDA error";
        case Q4_ERR_TIMEOUT: return "device-side wait timed out";
        case Q4_ERR_NO_DEVICE: return "no usable device";
        case Q4_ERR_DEVICE_CHECK: return "device-side check failed";
    }
    return "unknown status";
}

int q4_version(void) { return 100; }

q4_status q4_device_status(q4_stream_t stream) {
    clear_error();
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int word = 0, zero = 0;
    e = cudaMemcpy(&word, dev->err_word, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word == 0) return Q4_OK;
    e = cudaMemcpy(dev->err_word, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    if (word & 1) return fail(Q4_ERR_TIMEOUT, "a device-side wait ran out (error word 0x%x)", word);
    return fail(Q4_ERR_DEVICE_CHECK, "device-side validation failed (error word 0x%x)", word);
}

q4_status q4_gemv(const uint32_t* Wq, const uint16_t* scales, const uint16_t* biases, const uint16_t* x,
                  float* y, int M, int N, int K, q4_stream_t stream) {
    clear_error();
    q4_gemv_desc d = {};
    d.M = M;
    d.K = K;
    d.x = x;
    d.ldx = K;
    d.n_segments = 1;
    d.seg[0].Wq = Wq;
    d.seg[0].scales = scales;
    d.seg[0].biases = biases;
    d.seg[0].N = N;
    d.seg[0].y = y;
    d.out_dtype = Q4_F32;
    d.mode = Q4_GEMV_PLAIN;
    q4_status st = validate_gemv(d);
    if (st != Q4_OK) return st;
    return launch_gemv(d, reinterpret_cast<cudaStream_t>(stream), false, false);
}

q4_status q4_gemv8(const uint32_t* Wq, const uint16_t* scales, const uint16_t* biases, const uint16_t* x,
                   float* y, int M, int N, int K, q4_stream_t stream) {
    clear_error();
    q4_gemv_desc d = {};
    d.M = M;
    d.K = K;
    d.x = x;
    d.ldx = K;
    d.n_segments = 1;
    d.seg[0].Wq = Wq;
    d.seg[0].scales = scales;
    d.seg[0].biases = biases;
    d.seg[0].N = N;
    d.seg[0].y = y;
    d.out_dtype = Q4_F32;
    d.mode = Q4_GEMV_PLAIN;
    q4_status st = validate_gemv(d);
    if (st != Q4_OK) return st;
    return launch_gemv(d, reinterpret_cast<cudaStream_t>(stream), false, false, nullptr, 8);
}

q4_status q4_gemv_bits(const uint32_t* Wq, const uint16_t* scales, const uint16_t* biases, const uint16_t* x,
                       float* y, int M, int N, int K, int bits, q4_stream_t stream) {
    clear_error();
    if (bits < 2 || bits > 8 || bits == 7) return fail(Q4_ERR_INVALID_ARG, "bits=%d (2, 3, 4, 5, 6 or 8)", bits);
    q4_gemv_desc d = {};
    d.M = M;
    d.K = K;
    d.x = x;
    d.ldx = K;
    d.n_segments = 1;
    d.seg[0].Wq = Wq;
    d.seg[0].scales = scales;
    d.seg[0].biases = biases;
    d.seg[0].N = N;
    d.seg[0].y = y;
    d.out_dtype = Q4_F32;
    d.mode = Q4_GEMV_PLAIN;
    q4_status st = validate_gemv(d);
    if (st != Q4_OK) return st;
    if (bits != 4 && bits != 8 && M != 1) return fail(Q4_ERR_UNSUPPORTED, "%d-bit codes need M = 1", bits);
    return launch_gemv(d, reinterpret_cast<cudaStream_t>(stream), false, false, nullptr, bits);
}

q4_status q4_gemv_ex(const q4_gemv_desc* desc, q4_stream_t stream) {
    clear_error();
    if (!desc) return fail(Q4_ERR_INVALID_ARG, "desc is NULL");
    q4_status st = validate_gemv(*desc);
    if (st != Q4_OK) return st;
    const bool early = (desc->flags & Q4_GEMV_EARLY_WEIGHTS) != 0;
    return launch_gemv(*desc, reinterpret_cast<cudaStream_t>(stream), early, early);
}

}  // extern "C"
