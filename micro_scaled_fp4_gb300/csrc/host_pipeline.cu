// Host-buffer form of the FP8 activation path: E4M3 activations and their
// 1x128 tile scales in host memory are quantized straight to MXFP4
// ("Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// abstract and section 1) and re-expanded to FP8 for an FP8 consumer (same
// page, section 2.B); the MXFP4 codes and scales and the FP8 copy come back to
// host memory.
//
// The rows are cut into chunks (the first a quarter of the others) that move
// through a ring of three device slots in the caller's workspace.  Three
// streams overlap the transfers with the conversion: a copy-in stream
// (host -> slot), the caller's stream (the two conversion kernels on the slot)
// and a copy-out stream (slot -> host), in order per chunk through events:
//   copy-in c   waits  copy-out c - 3   (the slot is free again)
//   convert c   waits  copy-in c
//   copy-out c  waits  convert c
// The call starts after the work already queued on the caller's stream and
// that stream waits, at the end, for both copy streams (also when an enqueue
// failed midway): the results are in host memory once the caller's stream has
// reached that point.
#include <algorithm>

#include "common.cuh"

namespace fp4q {
namespace {

constexpr int kSlots = 3;
constexpr int64_t kDefaultChunkRows = 2048;
constexpr int kMaxDevices = 64;

inline uint64_t align256(uint64_t v) { return (v + 255u) & ~uint64_t(255); }

// Byte offsets of one slot's buffers (every one 256-byte aligned).
struct SlotLayout {
    uint64_t x, ts, q, s, y, yt, bytes;
};

SlotLayout slot_layout(int64_t cols, int64_t chunk) {
    SlotLayout L;
    const uint64_t n = uint64_t(chunk), c = uint64_t(cols);
    uint64_t o = 0;
    L.x = o;  o += align256(n * c);               // E4M3 in
    L.ts = o; o += align256(n * (c / 128) * 4);   // FP32 tile scales in
    L.q = o;  o += align256(n * (c / 2));         // MXFP4 codes
    L.s = o;  o += align256(n * (c / 32));        // E8M0 scales
    L.y = o;  o += align256(n * c);               // E4M3 out
    L.yt = o; o += align256(n * (c / 128) * 4);   // FP32 tile scales out
    L.bytes = o;
    return L;
}

int64_t chunk_for(int64_t rows, int64_t chunk_rows) {
    const int64_t c = chunk_rows > 0 ? chunk_rows : kDefaultChunkRows;
    return rows > 0 ? std::min(c, rows) : c;
}

// The copy streams and the ring's events, one set per host thread and device
// (created on first use, kept until fp4q_fp8_pipeline_host_release or the end
// of the process).
struct Engine {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, in_done = nullptr, out_done = nullptr;
    cudaEvent_t loaded[kSlots] = {}, converted[kSlots] = {}, stored[kSlots] = {};
};
thread_local Engine t_engines[kMaxDevices];

fp4q_status engine(Engine** e_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(FP4Q_ERR_CUDA, "fp8_pipeline_host: no current device");
    Engine& g = t_engines[dev];
    if (!g.ready) {
        const unsigned ev = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&g.in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&g.out, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&g.start, ev)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&g.in_done, ev)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&g.out_done, ev)) != cudaSuccess)
            return fail(FP4Q_ERR_CUDA, "fp8_pipeline_host: stream setup: %s", cudaGetErrorString(e));
        for (int k = 0; k < kSlots; ++k)
            if ((e = cudaEventCreateWithFlags(&g.loaded[k], ev)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&g.converted[k], ev)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&g.stored[k], ev)) != cudaSuccess)
                return fail(FP4Q_ERR_CUDA, "fp8_pipeline_host: event setup: %s", cudaGetErrorString(e));
        g.ready = true;
    }
    *e_out = &g;
    return FP4Q_OK;
}

// Queues the chunks (copy-in, the two conversions on `s`, copy-out) through
// the ring of slots.
fp4q_status enqueue_chunks(Engine* g, const uint8_t* x, const float* tile_scale, int64_t rows, int64_t cols,
                           uint8_t* q, uint8_t* scales, uint8_t* y, float* y_tile_scale, int64_t chunk,
                           const SlotLayout& L, uint8_t* ws, cudaStream_t s, fp4q_stream_t stream) {
    const uint64_t c = uint64_t(cols), tpr = c / 128;
    cudaError_t e;
    fp4q_status st;
#define FP4Q_CUDA(call)                                                                         \
    do {                                                                                        \
        if ((e = (call)) != cudaSuccess)                                                        \
            return fail(FP4Q_ERR_CUDA, "fp8_pipeline_host: %s: %s", #call, cudaGetErrorString(e)); \
    } while (0)
    // The first chunk is a quarter chunk: the device-to-host stream, the
    // slower direction, starts after a quarter of the fill time.
    const int64_t first = std::max<int64_t>(1, std::min(chunk / 4, rows));
    int64_t ci = 0;
    for (int64_t r = 0; r < rows; ++ci) {
        const int k = int(ci % kSlots);
        const uint64_t r0 = uint64_t(r), n = uint64_t(std::min(ci == 0 ? first : chunk, rows - r));
        r += int64_t(n);
        uint8_t* slot = ws + uint64_t(k) * L.bytes;
        if (ci >= kSlots) FP4Q_CUDA(cudaStreamWaitEvent(g->in, g->stored[k], 0));
        FP4Q_CUDA(cudaMemcpyAsync(slot + L.x, x + r0 * c, n * c, cudaMemcpyHostToDevice, g->in));
        FP4Q_CUDA(cudaMemcpyAsync(slot + L.ts, tile_scale + r0 * tpr, n * tpr * 4, cudaMemcpyHostToDevice, g->in));
        FP4Q_CUDA(cudaEventRecord(g->loaded[k], g->in));

        FP4Q_CUDA(cudaStreamWaitEvent(s, g->loaded[k], 0));
        if ((st = fp4q_mx_quantize(slot + L.x, FP4Q_E4M3, reinterpret_cast<const float*>(slot + L.ts), int64_t(n),
                                   cols, cols, 1, slot + L.q, slot + L.s, FP4Q_SCALES_ROWMAJOR, stream)) != FP4Q_OK)
            return st;
        if ((st = fp4q_fp4_to_fp8(slot + L.q, slot + L.s, int64_t(n), cols, 1, slot + L.y,
                                  reinterpret_cast<float*>(slot + L.yt), stream)) != FP4Q_OK)
            return st;
        FP4Q_CUDA(cudaEventRecord(g->converted[k], s));

        FP4Q_CUDA(cudaStreamWaitEvent(g->out, g->converted[k], 0));
        FP4Q_CUDA(cudaMemcpyAsync(q + r0 * (c / 2), slot + L.q, n * (c / 2), cudaMemcpyDeviceToHost, g->out));
        FP4Q_CUDA(cudaMemcpyAsync(scales + r0 * (c / 32), slot + L.s, n * (c / 32), cudaMemcpyDeviceToHost, g->out));
        FP4Q_CUDA(cudaMemcpyAsync(y + r0 * c, slot + L.y, n * c, cudaMemcpyDeviceToHost, g->out));
        FP4Q_CUDA(cudaMemcpyAsync(y_tile_scale + r0 * tpr, slot + L.yt, n * tpr * 4, cudaMemcpyDeviceToHost, g->out));
        FP4Q_CUDA(cudaEventRecord(g->stored[k], g->out));
    }
#undef FP4Q_CUDA
    return FP4Q_OK;
}

}  // namespace
}  // namespace fp4q

using namespace fp4q;

// A slot of chunk x cols elements must stay far inside 64-bit sizes.
static bool slot_too_large(int64_t cols, int64_t chunk) {
    return cols > (int64_t(1) << 31) || chunk > (int64_t(1) << 40) / std::max<int64_t>(cols, 1);
}

extern "C" size_t fp4q_fp8_pipeline_host_workspace_bytes(int64_t cols, int64_t chunk_rows) {
    if (cols <= 0 || chunk_rows < 0) return 0;
    const int64_t chunk = chunk_for(0, chunk_rows);
    if (slot_too_large(cols, chunk)) return 0;
    return size_t(kSlots) * size_t(slot_layout(cols, chunk).bytes);
}

extern "C" fp4q_status fp4q_fp8_pipeline_host(const uint8_t* x, const float* tile_scale, int64_t rows,
                                              int64_t cols, uint8_t* q, uint8_t* scales, uint8_t* y,
                                              float* y_tile_scale, int64_t chunk_rows, void* workspace,
                                              size_t workspace_bytes, fp4q_stream_t stream) {
    if (rows < 0 || cols < 0 || chunk_rows < 0)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp8_pipeline_host: negative size");
    if (cols % 128) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "fp8_pipeline_host: cols %% 128 != 0");
    if (rows == 0 || cols == 0) return FP4Q_OK;
    if (!x || !tile_scale || !q || !scales || !y || !y_tile_scale || !workspace)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp8_pipeline_host: null pointer");
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(FP4Q_ERR_MISALIGNED, "fp8_pipeline_host: workspace must be 256-byte aligned");
    const int64_t chunk = chunk_for(rows, chunk_rows);
    if (slot_too_large(cols, chunk))
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "fp8_pipeline_host: chunk of %lld x %lld elements too large",
                    static_cast<long long>(chunk), static_cast<long long>(cols));
    const SlotLayout L = slot_layout(cols, chunk);
    if (workspace_bytes < size_t(kSlots) * L.bytes)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp8_pipeline_host: workspace too small (%zu < %zu)",
                    workspace_bytes, size_t(kSlots) * size_t(L.bytes));
    int sms = 0;
    fp4q_status st = current_device(&sms);
    if (st != FP4Q_OK) return st;
    Engine* g = nullptr;
    if ((st = engine(&g)) != FP4Q_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    // everything queued on the caller's stream before this call comes first
    cudaError_t e = cudaEventRecord(g->start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(g->in, g->start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(g->out, g->start, 0);
    if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "fp8_pipeline_host: stream ordering: %s", cudaGetErrorString(e));
    st = enqueue_chunks(g, x, tile_scale, rows, cols, q, scales, y, y_tile_scale, chunk, L, ws, s, stream);
    // The caller's stream continues once both copy streams are done with this
    // call -- also after a failed enqueue, so that no copy the call issued is
    // still running when the caller reuses its buffers.
    cudaError_t j = cudaEventRecord(g->in_done, g->in);
    if (j == cudaSuccess) j = cudaEventRecord(g->out_done, g->out);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(s, g->in_done, 0);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(s, g->out_done, 0);
    if (st == FP4Q_OK && j != cudaSuccess)
        st = fail(FP4Q_ERR_CUDA, "fp8_pipeline_host: stream ordering: %s", cudaGetErrorString(j));
    return st;
}

extern "C" fp4q_status fp4q_fp8_pipeline_host_release(void) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(FP4Q_ERR_CUDA, "fp8_pipeline_host_release: no current device");
    Engine& g = t_engines[dev];
    if (!g.ready) return FP4Q_OK;
    // no copy of an earlier call may still be running on the streams
    if ((e = cudaStreamSynchronize(g.in)) != cudaSuccess || (e = cudaStreamSynchronize(g.out)) != cudaSuccess)
        return fail(FP4Q_ERR_CUDA, "fp8_pipeline_host_release: %s", cudaGetErrorString(e));
    cudaStreamDestroy(g.in);
    cudaStreamDestroy(g.out);
    for (cudaEvent_t ev : {g.start, g.in_done, g.out_done}) cudaEventDestroy(ev);
    for (int k = 0; k < kSlots; ++k) {
        cudaEventDestroy(g.loaded[k]);
        cudaEventDestroy(g.converted[k]);
        cudaEventDestroy(g.stored[k]);
    }
    g = Engine();
    return FP4Q_OK;
}
