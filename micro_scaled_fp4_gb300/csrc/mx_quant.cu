// MXFP4 quantize (BF16 / FP32 / FP8-E4M3 sources) and MXFP4 dequantize.
//
// MX format ("Pretraining large language models with MXFP4 on Native FP4
// Hardware", MX section): blocks of 32 elements share an E8M0 exponent
// E = floor(log2(block amax)) - 2 and each element is the E2M1 code nearest
// to x / 2^E.  Direct FP8 source ("Practical FP4 Training for Large-Scale MoE
// Models on Hopper GPUs", abstract and section 1): E4M3 codes times their
// 1x128 tile's FP32 scale, quantized with no BF16 step.
//
// Streaming design: one thread owns one 32-element block, so the block amax
// never leaves the thread's registers.  Loads are 256-bit (one 32-byte sector
// per lane per instruction), the 16 bytes of codes go out as one 128-bit store
// (a warp writes 512 contiguous bytes), the scale byte as one byte store
// (a warp writes 32 contiguous bytes in row-major layout).  The rounding is
// the hardware cvt.rn.satfinite.e2m1x2.f32, after an exact power-of-two
// multiply by 2^-E.
#include "common.cuh"

namespace fp4q {
namespace {

enum Src { kBF16 = 0, kFP32 = 1, kE4M3 = 2 };

__device__ __forceinline__ uint32_t pack4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
    return b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
}

template <int SRC>
__global__ void __launch_bounds__(256) mx_quantize_kernel(
    const uint8_t* __restrict__ x, const float* __restrict__ tile_scale, int64_t rows,
    uint32_t bpr, int64_t ld_x_bytes, uint8_t* __restrict__ q, uint8_t* __restrict__ s,
    int mma_layout) {
    const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= bpr) return;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        uint32_t codes[4];
        uint32_t sbyte;
        if constexpr (SRC == kBF16) {
            const uint8_t* p = x + r * ld_x_bytes + uint64_t(b) * 64;
            u32x8 a = ldg256(p), c = ldg256(p + 32);
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) { w[i] = a.v[i]; w[8 + i] = c.v[i]; }
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) m = __vmaxu2(m, w[i] & 0x7fff7fffu);
            uint32_t amax16 = max(m & 0xffffu, m >> 16);
            int e = mx_exponent_from_amax_bits(amax16 << 16);
            sbyte = uint32_t(e + 127);
            const float inv = exp2i(-e);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t bytes[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t ww = w[4 * k + j];
                    float lo = __fmul_rn(u2f(ww << 16), inv);
                    float hi = __fmul_rn(u2f(ww & 0xffff0000u), inv);
                    bytes[j] = cvt_e2m1x2(lo, hi);
                }
                codes[k] = pack4(bytes[0], bytes[1], bytes[2], bytes[3]);
            }
        } else if constexpr (SRC == kFP32) {
            const uint8_t* p = x + r * ld_x_bytes + uint64_t(b) * 128;
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                u32x8 a = ldg256(p + 32 * i);
#pragma unroll
                for (int j = 0; j < 8; ++j) w[8 * i + j] = a.v[j];
            }
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) m = max(m, w[i] & 0x7fffffffu);
            int e = mx_exponent_from_amax_bits(m);
            sbyte = uint32_t(e + 127);
            const float inv = exp2i(-e);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t bytes[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    bytes[j] = cvt_e2m1x2(__fmul_rn(u2f(w[8 * k + 2 * j]), inv),
                                          __fmul_rn(u2f(w[8 * k + 2 * j + 1]), inv));
                codes[k] = pack4(bytes[0], bytes[1], bytes[2], bytes[3]);
            }
        } else {
            const uint8_t* p = x + r * ld_x_bytes + uint64_t(b) * 32;
            u32x8 a = ldg256(p);
            const float ts = tile_scale[r * (bpr >> 2) + (b >> 2)];
            // The E4M3 encoding is monotone in magnitude, and so is the FP32
            // product with the tile scale: the block amax is the product of
            // the largest magnitude byte.
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = __vmaxu4(m, a.v[i] & 0x7f7f7f7fu);
            m = max(max(m & 0xffu, (m >> 8) & 0xffu), max((m >> 16) & 0xffu, m >> 24));
            float amax = fabsf(__fmul_rn(e4m3x2_to_f32x2(m).x, ts));
            int e = mx_exponent_from_amax_bits(f2u(amax));
            sbyte = uint32_t(e + 127);
            const float inv = exp2i(-e);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t bytes[4];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    uint32_t ww = a.v[2 * k + j];
                    float2 f01 = e4m3x2_to_f32x2(ww & 0xffffu);
                    float2 f23 = e4m3x2_to_f32x2(ww >> 16);
                    bytes[2 * j] = cvt_e2m1x2(__fmul_rn(__fmul_rn(f01.x, ts), inv),
                                              __fmul_rn(__fmul_rn(f01.y, ts), inv));
                    bytes[2 * j + 1] = cvt_e2m1x2(__fmul_rn(__fmul_rn(f23.x, ts), inv),
                                                  __fmul_rn(__fmul_rn(f23.y, ts), inv));
                }
                codes[k] = pack4(bytes[0], bytes[1], bytes[2], bytes[3]);
            }
        }
        *reinterpret_cast<uint4*>(q + r * (uint64_t(bpr) * 16) + uint64_t(b) * 16) =
            make_uint4(codes[0], codes[1], codes[2], codes[3]);
        const uint64_t so = mma_layout ? mma_scale_offset(uint64_t(r), b, bpr) : uint64_t(r) * bpr + b;
        s[so] = uint8_t(sbyte);
    }
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(256) mx_dequantize_kernel(
    const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t rows, uint32_t bpr,
    uint8_t* __restrict__ y) {
    const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= bpr) return;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const uint64_t blk = uint64_t(r) * bpr + b;
        const uint4 cw = *reinterpret_cast<const uint4*>(q + blk * 16);
        const float sc = exp2i(int(s[blk]) - 127);
        const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
        float v[32];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 f = e2m1x2_to_f32x2((words[k] >> (8 * j)) & 0xffu);
                v[8 * k + 2 * j] = __fmul_rn(f.x, sc);
                v[8 * k + 2 * j + 1] = __fmul_rn(f.y, sc);
            }
        if constexpr (OUT_BF16) {
            u32x8 o[2];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                uint32_t packed;
                asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed) : "f"(v[2 * i + 1]), "f"(v[2 * i]));
                o[i >> 3].v[i & 7] = packed;
            }
            stg256(y + blk * 64, o[0]);
            stg256(y + blk * 64 + 32, o[1]);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                u32x8 o;
#pragma unroll
                for (int j = 0; j < 8; ++j) o.v[j] = f2u(v[8 * i + j]);
                stg256(y + blk * 128 + 32 * i, o);
            }
        }
    }
}

inline dim3 grid_for_rows(int64_t rows, int nx) {
    int64_t gy = rows < 65535 ? rows : 65535;
    return dim3(unsigned(nx), unsigned(gy > 0 ? gy : 1), 1);
}

}  // namespace
}  // namespace fp4q

using namespace fp4q;

extern "C" fp4q_status fp4q_mx_quantize(const void* x, fp4q_dtype x_type, const float* tile_scale,
                                        int64_t rows, int64_t cols, int64_t ld_x, int block_axis,
                                        uint8_t* q, uint8_t* scales, fp4q_scale_layout layout,
                                        fp4q_stream_t stream) {
    if (x_type != FP4Q_BF16 && x_type != FP4Q_FP32 && x_type != FP4Q_E4M3)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "mx_quantize: x_type must be BF16, FP32 or E4M3");
    if (layout != FP4Q_SCALES_ROWMAJOR && layout != FP4Q_SCALES_MMA)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "mx_quantize: bad scale layout");
    if (rows < 0 || cols < 0 || ld_x < cols)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "mx_quantize: need rows >= 0, cols >= 0, ld_x >= cols");
    if (block_axis != 1) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "mx_quantize: only block_axis = 1 (last axis)");
    if (cols % 32) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "mx_quantize: cols %% 32 != 0");
    if (x_type == FP4Q_E4M3 && cols % 128)
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "mx_quantize: E4M3 source needs cols %% 128 == 0");
    if (rows == 0 || cols == 0) return FP4Q_OK;
    if (!x || !q || !scales || (x_type == FP4Q_E4M3 && !tile_scale))
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "mx_quantize: null pointer");
    const int64_t esz = x_type == FP4Q_BF16 ? 2 : (x_type == FP4Q_FP32 ? 4 : 1);
    if ((reinterpret_cast<uintptr_t>(x) & 31u) || (ld_x * esz) % 32 || !aligned16(q))
        return fail(FP4Q_ERR_MISALIGNED, "mx_quantize: x must be 32-byte aligned with ld_x*elem %% 32 == 0, q 16-byte aligned");
    if (x_type == FP4Q_E4M3 && (reinterpret_cast<uintptr_t>(tile_scale) & 3u))
        return fail(FP4Q_ERR_MISALIGNED, "mx_quantize: tile_scale must be 4-byte aligned");
    fp4q_status st = current_device(nullptr);
    if (st != FP4Q_OK) return st;
    const uint32_t bpr = uint32_t(cols / 32);
    int tpb, nx;
    row_launch_shape(bpr, &tpb, &nx);
    dim3 grid = grid_for_rows(rows, nx);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    const int mma = layout == FP4Q_SCALES_MMA;
    switch (x_type) {
        case FP4Q_BF16:
            mx_quantize_kernel<kBF16><<<grid, tpb, 0, s>>>(xb, nullptr, rows, bpr, ld_x * 2, q, scales, mma);
            break;
        case FP4Q_FP32:
            mx_quantize_kernel<kFP32><<<grid, tpb, 0, s>>>(xb, nullptr, rows, bpr, ld_x * 4, q, scales, mma);
            break;
        default:
            mx_quantize_kernel<kE4M3><<<grid, tpb, 0, s>>>(xb, tile_scale, rows, bpr, ld_x, q, scales, mma);
            break;
    }
    return check_launch("mx_quantize");
}

extern "C" fp4q_status fp4q_mx_dequantize(const uint8_t* q, const uint8_t* scales, int64_t rows,
                                          int64_t cols, int block_axis, void* y, fp4q_dtype y_type,
                                          fp4q_stream_t stream) {
    if (y_type != FP4Q_BF16 && y_type != FP4Q_FP32)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "mx_dequantize: y_type must be BF16 or FP32");
    if (rows < 0 || cols < 0) return fail(FP4Q_ERR_INVALID_ARGUMENT, "mx_dequantize: negative size");
    if (block_axis != 1) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "mx_dequantize: only block_axis = 1");
    if (cols % 32) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "mx_dequantize: cols %% 32 != 0");
    if (rows == 0 || cols == 0) return FP4Q_OK;
    if (!q || !scales || !y) return fail(FP4Q_ERR_INVALID_ARGUMENT, "mx_dequantize: null pointer");
    if (!aligned16(q) || (reinterpret_cast<uintptr_t>(y) & 31u))
        return fail(FP4Q_ERR_MISALIGNED, "mx_dequantize: q must be 16-byte and y 32-byte aligned");
    fp4q_status st = current_device(nullptr);
    if (st != FP4Q_OK) return st;
    const uint32_t bpr = uint32_t(cols / 32);
    int tpb, nx;
    row_launch_shape(bpr, &tpb, &nx);
    dim3 grid = grid_for_rows(rows, nx);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (y_type == FP4Q_BF16)
        mx_dequantize_kernel<true><<<grid, tpb, 0, s>>>(q, scales, rows, bpr, static_cast<uint8_t*>(y));
    else
        mx_dequantize_kernel<false><<<grid, tpb, 0, s>>>(q, scales, rows, bpr, static_cast<uint8_t*>(y));
    return check_launch("mx_dequantize");
}
