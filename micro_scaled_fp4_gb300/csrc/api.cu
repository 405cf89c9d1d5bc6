// Status codes, per-thread error detail, device checks and the device status
// word of the fp4q library.
#include <atomic>
#include <mutex>
#include <stdarg.h>
#include <stdio.h>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "ring.cuh"
#include "tc.cuh"

namespace fp4q {

// One status word per device: kernels OR a bit into it when a bounded
// device-side wait gives up (they then skip their remaining work and return).
__device__ uint32_t g_status_word;

static thread_local char t_last_error[512] = "";

fp4q_status fail(fp4q_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return st;
}

fp4q_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return FP4Q_OK;
}

namespace {
constexpr int kMaxDevices = 64;
struct DeviceInfo {
    std::atomic<bool> ready{false};    // set (release) once the fields below are filled in
    bool supported = false;
    int sms = 0;
    uint32_t* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;
}  // namespace

fp4q_status current_device(int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(FP4Q_ERR_UNSUPPORTED_DEVICE, "device index %d", dev);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int major = 0, minor = 0, count = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return fail(FP4Q_ERR_CUDA, "cudaDeviceGetAttribute failed on device %d", dev);
            d.supported = (major == 10 && minor == 3);
            d.sms = count;
            if (d.supported) {
                void* p = nullptr;
                e = cudaGetSymbolAddress(&p, g_status_word);
                if (e != cudaSuccess)
                    return fail(FP4Q_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
                d.status = static_cast<uint32_t*>(p);
            }
            d.ready.store(true, std::memory_order_release);
        }
    }
    if (!d.supported)
        return fail(FP4Q_ERR_UNSUPPORTED_DEVICE, "device %d is not compute capability 10.3 (sm_103a)", dev);
    if (sms) *sms = d.sms;
    return FP4Q_OK;
}

uint32_t* status_word() {
    int dev = 0;
    cudaGetDevice(&dev);
    return g_dev[dev].status;
}

namespace {
// One thread waits, with the library's bounded wait, on an mbarrier that
// nothing will ever complete; when the limit runs out it records the
// self-check bit in the status word and returns.
__global__ void wait_timeout_kernel(uint64_t limit_ns, uint32_t* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    tc::mbar_init(tc::smem_u32(&bar), 1);
    tc::fence_barrier_init();
    if (!tc::mbar_wait(tc::smem_u32(&bar), 0, &abort_flag, limit_ns)) atomicOr(status, kStatusSelfCheck);
}
}  // namespace

}  // namespace fp4q

using namespace fp4q;

extern "C" fp4q_status fp4q_check_wait_timeout(uint64_t limit_ns, fp4q_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 2000000000ull)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "check_wait_timeout: limit must be in (0, 2 s]");
    fp4q_status st = current_device(nullptr);
    if (st != FP4Q_OK) return st;
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, status_word());
    return check_launch("check_wait_timeout");
}

extern "C" const char* fp4q_status_string(fp4q_status s) {
    switch (s) {
        case FP4Q_OK: return "FP4Q_OK";
        case FP4Q_ERR_INVALID_ARGUMENT: return "FP4Q_ERR_INVALID_ARGUMENT";
        case FP4Q_ERR_UNSUPPORTED_SHAPE: return "FP4Q_ERR_UNSUPPORTED_SHAPE";
        case FP4Q_ERR_MISALIGNED: return "FP4Q_ERR_MISALIGNED";
        case FP4Q_ERR_UNSUPPORTED_DEVICE: return "FP4Q_ERR_UNSUPPORTED_DEVICE";
        case FP4Q_ERR_CUDA: return "FP4Q_ERR_CUDA";
        case FP4Q_ERR_TIMEOUT: return "FP4Q_ERR_TIMEOUT";
    }
    return "FP4Q_UNKNOWN_STATUS";
}

extern "C" const char* fp4q_last_error(void) { return t_last_error; }

// 0 when the size does not fit a size_t (sizes no allocation could hold)
extern "C" size_t fp4q_scales_bytes(int64_t rows, int64_t scale_cols, fp4q_scale_layout layout) {
    if (rows < 0 || scale_cols < 0 || rows > (int64_t(1) << 60) || scale_cols > (int64_t(1) << 60)) return 0;
    size_t n = 0;
    if (layout == FP4Q_SCALES_MMA) {
        if (__builtin_mul_overflow(size_t((rows + 127) / 128), size_t((scale_cols + 3) / 4), &n) ||
            __builtin_mul_overflow(n, size_t(512), &n))
            return 0;
        return n;
    }
    return __builtin_mul_overflow(size_t(rows), size_t(scale_cols), &n) ? 0 : n;
}

extern "C" fp4q_status fp4q_device_status(uint32_t* status_out, int reset) {
    if (!status_out) return fail(FP4Q_ERR_INVALID_ARGUMENT, "status_out is NULL");
    fp4q_status st = current_device(nullptr);
    if (st != FP4Q_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
    uint32_t v = 0;
    e = cudaMemcpy(&v, status_word(), sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "read status word: %s", cudaGetErrorString(e));
    if (reset) {
        uint32_t z = 0;
        e = cudaMemcpy(status_word(), &z, sizeof z, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "reset status word: %s", cudaGetErrorString(e));
    }
    *status_out = v;
    return v ? FP4Q_ERR_TIMEOUT : FP4Q_OK;
}

extern "C" fp4q_status fp4q_stream_status(uint32_t* status_out, int reset, fp4q_stream_t stream) {
    fp4q_status st = current_device(nullptr);
    if (st != FP4Q_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, status_word(), sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && reset) e = cudaMemsetAsync(status_word(), 0, sizeof v, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "stream_status: %s", cudaGetErrorString(e));
    if (status_out) *status_out = v;
    return v ? FP4Q_ERR_TIMEOUT : FP4Q_OK;
}

namespace fp4q {
namespace ring {

fp4q_status encode_bf16_tile_map(CUtensorMap* map, const void* x, int64_t rows, int64_t cols, int64_t ld,
                                 uint32_t box_cols, uint32_t box_rows) {
    // looked up on first use; concurrent first calls store the same pointer
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> encode_fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn.load(std::memory_order_acquire);
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return fail(FP4Q_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        encode_fn.store(encode, std::memory_order_release);
    }
    cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(ld * 2)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FP4Q_ERR_CUDA, "cuTensorMapEncodeTiled (BF16 tile) failed (%d)", int(r));
    return FP4Q_OK;
}

}  // namespace ring
}  // namespace fp4q
