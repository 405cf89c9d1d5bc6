// Shared device and host helpers of the fp4q CUDA library (sm_103a).
//
// Number formats (OCP MX / OCP FP8):
//   E2M1  4-bit float, codes 0..7 = {0, .5, 1, 1.5, 2, 3, 4, 6}, bit 3 = sign.
//   E8M0  unsigned power-of-two exponent byte, value 2^(byte - 127).
//   E4M3  "FN" 8-bit float, bias 7, max 448, smallest subnormal 2^-9.
#pragma once

#include <algorithm>
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "../../include/fp4q.h"

namespace fp4q {

// ---------------------------------------------------------------------------
// Host side: status plumbing (api.cu)
// ---------------------------------------------------------------------------
fp4q_status fail(fp4q_status st, const char* fmt, ...);
fp4q_status check_launch(const char* what);
// Validates the current device (compute capability 10.3) and caches its
// properties; returns the SM count through *sms.
fp4q_status current_device(int* sms);
// Device address of the library's status word on the current device.
uint32_t* status_word();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 32-bit shared-memory address of a __shared__ object (for ld/st.shared).
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Status-word bits (which kernel gave up a bounded wait).
enum : uint32_t {
    kStatusGemmTimeout = 1u << 0,
    kStatusGroupedTimeout = 1u << 1,
    kStatusStreamTimeout = 1u << 2,
    kStatusBadTileScale = 1u << 3,
    kStatusSelfCheck = 1u << 31
};

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

// 2^e as an FP32 (exact), e in [-127, 127]; 2^-127 is the subnormal 0x00400000.
__device__ __forceinline__ float exp2i(int e) {
    return e >= -126 ? u2f(uint32_t(e + 127) << 23) : u2f(0x00400000u);
}

// floor(log2 |f|) of a positive finite FP32 bit pattern (subnormals included).
__device__ __forceinline__ int floor_log2_bits(uint32_t bits) {
    uint32_t ex = (bits >> 23) & 0xffu;
    if (ex != 0) return int(ex) - 127;
    uint32_t m = bits & 0x7fffffu;
    return -149 + (31 - __clz(m));
}

// MX shared exponent of a block from the FP32 bits of its amax:
// floor(log2 amax) - 2, clamped to [-127, 127]; amax == 0 -> -127.
__device__ __forceinline__ int mx_exponent_from_amax_bits(uint32_t amax_bits) {
    if (amax_bits == 0) return -127;
    int e = floor_log2_bits(amax_bits) - 2;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Two FP32 -> one byte of two E2M1 codes, round-to-nearest-even, saturating
// at +-6: `lo` goes to the low nibble, `hi` to the high nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u16.u8 %0, t;\n}"
        : "=h"(r) : "f"(hi), "f"(lo));
    return r & 0xffu;
}

// Packed FP32 pairs (Blackwell mul.rn.f32x2): two IEEE round-to-nearest-even
// multiplies per instruction, identical results to the scalar ones.
__device__ __forceinline__ uint64_t f32x2_splat(float s) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(s));
    return r;
}
__device__ __forceinline__ void mul_f32x2(float& a, float& b, uint64_t s2) {
    asm("{\n .reg .b64 x;\n mov.b64 x, {%0, %1};\n mul.rn.f32x2 x, x, %2;\n mov.b64 {%0, %1}, x;\n}"
        : "+f"(a), "+f"(b) : "l"(s2));
}
// FP16 pair (one 32-bit word) -> two FP32, each times the scale pair s2.
__device__ __forceinline__ void f16x2_mul_f32x2(uint32_t h, uint64_t s2, float& o0, float& o1) {
    asm("{\n .reg .b16 lo, hi;\n .reg .f32 a, b;\n .reg .b64 x;\n mov.b32 {lo, hi}, %2;\n"
        " cvt.f32.f16 a, lo;\n cvt.f32.f16 b, hi;\n mov.b64 x, {a, b};\n mul.rn.f32x2 x, x, %3;\n"
        " mov.b64 {%0, %1}, x;\n}" : "=f"(o0), "=f"(o1) : "r"(h), "l"(s2));
}

// Eight FP32 -> one 32-bit word of eight E2M1 codes (element j in nibble j),
// round-to-nearest-even, saturating at +-6.
__device__ __forceinline__ uint32_t cvt_e2m1x8(float v0, float v1, float v2, float v3, float v4, float v5,
                                               float v6, float v7) {
    uint32_t out;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        " mov.b32 %0, {b0, b1, b2, b3};\n}"
        : "=r"(out) : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
    return out;
}

// Four E4M3 bytes of a 32-bit word (byte j = element j) -> four FP32 (exact).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float (&f)[4]) {
    asm("{\n .reg .b16 lo, hi, x0, x1, x2, x3;\n .reg .b32 h01, h23;\n"
        " mov.b32 {lo, hi}, %4;\n"
        " cvt.rn.f16x2.e4m3x2 h01, lo;\n cvt.rn.f16x2.e4m3x2 h23, hi;\n"
        " mov.b32 {x0, x1}, h01;\n mov.b32 {x2, x3}, h23;\n"
        " cvt.f32.f16 %0, x0;\n cvt.f32.f16 %1, x1;\n cvt.f32.f16 %2, x2;\n cvt.f32.f16 %3, x3;\n}"
        : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]) : "r"(w));
}

// FP32 -> E4M3 byte, round-to-nearest-even, saturating at +-448.
__device__ __forceinline__ uint32_t cvt_e4m3(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xffu;
}

// Two E4M3 bytes (low byte = element 0) -> two FP32 (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_bytes) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_bytes));
    float2 f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f.x) : "h"((uint16_t)(h2 & 0xffffu)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(f.y) : "h"((uint16_t)(h2 >> 16)));
    return f;
}

// One byte of two E2M1 codes (low nibble = element 0) -> two FP32 (exact).
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
    uint32_t h2;
    asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(h2) : "r"(byte));
    float2 f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f.x) : "h"((uint16_t)(h2 & 0xffffu)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(f.y) : "h"((uint16_t)(h2 >> 16)));
    return f;
}

// Byte offset of scale (r, c) in the tcgen05 scale-factor layout of an
// R x S scale matrix: 128 x 4 tiles of 512 bytes, tile-row-major, and inside
// a tile (r % 32) * 16 + (r / 32 % 4) * 4 + c % 4.
__device__ __forceinline__ uint64_t mma_scale_offset(uint64_t r, uint32_t c, uint32_t S) {
    uint32_t s4 = (S + 3) >> 2;
    return ((r >> 7) * s4 + (c >> 2)) * 512ull + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (c & 3);
}

// 256-bit global load (read-only path, no L1 allocation) and store.
struct u32x8 { uint32_t v[8]; };
__device__ __forceinline__ u32x8 ldg256(const void* p) {
    u32x8 r;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]),
                   "=r"(r.v[4]), "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7]) : "l"(p));
    return r;
}
__device__ __forceinline__ void stg256(void* p, const u32x8& r) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" :: "l"(p),
                 "r"(r.v[0]), "r"(r.v[1]), "r"(r.v[2]), "r"(r.v[3]),
                 "r"(r.v[4]), "r"(r.v[5]), "r"(r.v[6]), "r"(r.v[7]) : "memory");
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 multiplies whose halves are xored with the other counter words
// and the key; the key advances by the two Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// Launch shape for row-wise block kernels: one thread per block of a row,
// `bpr` blocks per row; returns threads per CTA and CTAs along the row.
inline void row_launch_shape(int64_t bpr, int* tpb, int* nx, int64_t max_threads = 256) {
    int64_t n = (bpr + max_threads - 1) / max_threads;
    int64_t per = (bpr + n - 1) / n;
    per = (per + 31) / 32 * 32;
    *tpb = int(per);
    *nx = int(n);
}

// Like row_launch_shape, but when `units` (threads of work per row) does not
// fill whole warps, a CTA takes *rpc rows side by side (rpc * units threads, a
// multiple of 32, at most max_threads) so that no lane idles.
inline void packed_row_shape(int64_t units, int* tpb, int* nx, int* rpc, int64_t max_threads = 512) {
    int64_t g = 32;
    while (units % g) g >>= 1;
    const int64_t r = 32 / g;
    if (r > 1 && r * units <= max_threads) {
        *tpb = int(r * units);
        *nx = 1;
        *rpc = int(r);
    } else {
        row_launch_shape(units, tpb, nx, max_threads < 256 ? max_threads : 256);
        *rpc = 1;
    }
}

// CTAs along the rows for a row-wise kernel: one full wave of resident CTAs
// (`per_sm` per SM), each then looping over its share of rows.
inline unsigned row_grid_y(int64_t rows, int nx, int sms, int per_sm = 8) {
    int64_t want = (int64_t(sms > 0 ? sms : 148) * (per_sm > 0 ? per_sm : 1)) / nx;
    if (want < 1) want = 1;
    int64_t gy = rows < want ? rows : want;
    if (gy > 65535) gy = 65535;
    return unsigned(gy > 0 ? gy : 1);
}

// Programmatic dependent launch.  A kernel launched with launch_overlapped()
// may start while the previous kernel on its stream is still draining: its
// CTAs run whatever needs no global memory, then grid_dependency_wait()
// blocks until every prior grid on the stream has completed and its memory
// is visible.  allow_dependent_launch() lets the next such kernel be launched
// (it takes effect once every CTA of this grid has run it or exited, so all
// of this grid's CTAs have started by then).  Without the launch attribute
// both instructions do nothing.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Resident CTAs per SM of `kernel` at `threads` per CTA and `smem` bytes of
// dynamic shared memory, remembered per kernel, device and size.  Above 48 KB
// the kernel's dynamic shared memory limit is raised to all the device's
// opt-in maximum leaves beside the kernel's static shared memory, never to
// `smem` itself: a limit set for one size would otherwise shrink below a
// larger size whose entry is already remembered.
template <typename Kernel>
inline int resident_per_sm_smem(Kernel kernel, int threads, uint32_t smem) {
    // keyed by the kernel itself: instances of one template share a type
    struct Entry { const void* fn; int dev; int threads; uint32_t smem; int n; };
    static Entry cache[16] = {};
    static int next = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    cudaGetDevice(&dev);
    const void* fn = reinterpret_cast<const void*>(kernel);
    for (const Entry& e : cache)
        if (e.n && e.fn == fn && e.dev == dev && e.threads == threads && e.smem == smem) return e.n;
    if (smem > 48 * 1024) {
        // the limit covers dynamic memory only: static + dynamic must fit the opt-in maximum
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaFuncAttributes fa{};
        cudaFuncGetAttributes(&fa, kernel);
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             std::max(int(smem), optin - int(fa.sharedSizeBytes)));
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
    cache[next] = Entry{fn, dev, threads, smem, n};
    next = (next + 1) % 16;
    return n;
}

// Resident CTAs per SM of `kernel` at `threads` per CTA (no dynamic shared
// memory), looked up once per kernel, device and block size.
template <typename Kernel>
inline int resident_per_sm(Kernel kernel, int threads) {
    return resident_per_sm_smem(kernel, threads, 0);
}

}  // namespace fp4q
