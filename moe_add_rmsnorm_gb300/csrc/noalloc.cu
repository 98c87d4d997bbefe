// q8_gemv_noalloc: the Q8_0 projection for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point they need a projection: code running inside an allocator's own
// callbacks, real-time loops that forbid allocation after start-up, or hosts whose device memory is all handed out up
// front by another runtime.  q8_gemv needs a workspace (q8_workspace_create allocates it); this entry point instead
// uses scratch that the library itself holds in a fixed-size device array, so it allocates nothing at all.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "q8moe.h"

namespace q8 {
int model_fail(int code, const char* fmt, ...);
void gemv_call_scratch(const q8_mat* W, q8_mode mode, const float* x, const q8_act* xq, int64_t rows,
                       size_t* bytes, size_t* counters);
int gemv_over_scratch(const q8_mat* W, q8_mode mode, const float* x, const q8_act* xq, int64_t rows, float* y,
                      char* scratch, size_t bytes, int* counters, size_t n_counters, size_t zero_counters,
                      cudaStream_t st, const char* who);
}  // namespace q8

using namespace q8;

// The library's own scratch: every device that loads the library holds both arrays until the process exits.  They
// start zeroed; every projection leaves its arrival counters at zero again.
static __device__ __align__(256) unsigned char g_noalloc_scratch[Q8_NOALLOC_SCRATCH_BYTES];
static __device__ __align__(256) int g_noalloc_counters[Q8_NOALLOC_COUNTERS];

namespace {

struct DeviceScratch {
    char* scratch = nullptr;
    int* counters = nullptr;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices];

// The device addresses of the two arrays on the current device, looked up once per device.  In host code the arrays'
// names are only host-side stand-ins; a kernel must be given these addresses.
int device_scratch(DeviceScratch* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return model_fail(Q8_ECUDA, "q8_gemv_noalloc: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return model_fail(Q8_EUNSUPPORTED, "q8_gemv_noalloc: device %d", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceScratch& d = g_dev[dev];
    if (!d.scratch) {
        void* s = nullptr;
        void* c = nullptr;
        e = cudaGetSymbolAddress(&s, g_noalloc_scratch);
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&c, g_noalloc_counters);
        if (e != cudaSuccess || !s || !c)
            return model_fail(Q8_ECUDA, "q8_gemv_noalloc: scratch address lookup: %s", cudaGetErrorString(e));
        d.scratch = (char*)s;
        d.counters = (int*)c;
    }
    *out = d;
    return Q8_OK;
}

}  // namespace

extern "C" {

int q8_gemv_noalloc(const q8_mat* W, q8_mode mode, const float* x, const q8_act* xq, int64_t rows, float* y,
                    q8_stream stream) {
    if (!W || !W->q || !W->s || W->rows < 1 || W->cols < 1 || W->cols % 32 || rows < 0 || rows > 65536 ||
        (mode != Q8_F32ACT_F64SUM && mode != Q8_INT8ACT && mode != Q8_INT8ACT2))
        return gemv_over_scratch(W, mode, x, xq, rows, y, nullptr, 0, nullptr, 0, 0, (cudaStream_t)stream,
                                 "q8_gemv_noalloc");  // the projection's own argument checks name the problem
    size_t bytes = 0, counters = 0;
    gemv_call_scratch(W, mode, x, xq, rows, &bytes, &counters);
    if (bytes > Q8_NOALLOC_SCRATCH_BYTES || counters > Q8_NOALLOC_COUNTERS)
        return model_fail(Q8_ENOSPACE,
                          "q8_gemv_noalloc: this call needs %zu bytes and %zu counters of scratch; the library holds "
                          "%u bytes and %u counters (use q8_gemv with a workspace)",
                          bytes, counters, (unsigned)Q8_NOALLOC_SCRATCH_BYTES, (unsigned)Q8_NOALLOC_COUNTERS);
    DeviceScratch d;
    if (int r = device_scratch(&d)) return r;
    // the counters the call uses are cleared after its arguments pass their checks and before its launches
    return gemv_over_scratch(W, mode, x, xq, rows, y, d.scratch, Q8_NOALLOC_SCRATCH_BYTES, d.counters,
                             Q8_NOALLOC_COUNTERS, counters, (cudaStream_t)stream, "q8_gemv_noalloc");
}

}  // extern "C"
