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
#include <algorithm>

#include "common.cuh"
#include "ring.cuh"

namespace fp4q {
namespace {

enum Src { kBF16 = 0, kFP32 = 1, kE4M3 = 2 };

// One 32-element block as loaded from memory.
template <int SRC> struct RawBlock;
template <> struct RawBlock<kBF16> { u32x8 a, b; };
template <> struct RawBlock<kFP32> { u32x8 a[4]; };
template <> struct RawBlock<kE4M3> { u32x8 a; float ts; };

template <int SRC>
__device__ __forceinline__ void load_block(const uint8_t* __restrict__ x, const float* __restrict__ tile_scale,
                                           int64_t r, uint32_t b, uint32_t bpr, int64_t ld_x_bytes,
                                           RawBlock<SRC>& raw) {
    if constexpr (SRC == kBF16) {
        const uint8_t* p = x + r * ld_x_bytes + uint64_t(b) * 64;
        raw.a = ldg256(p);
        raw.b = ldg256(p + 32);
    } else if constexpr (SRC == kFP32) {
        const uint8_t* p = x + r * ld_x_bytes + uint64_t(b) * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i) raw.a[i] = ldg256(p + 32 * i);
    } else {
        raw.a = ldg256(x + r * ld_x_bytes + uint64_t(b) * 32);
        raw.ts = __ldg(tile_scale + r * (bpr >> 2) + (b >> 2));
    }
}

// Block -> 16 bytes of codes and the E8M0 byte.
template <int SRC>
__device__ __forceinline__ void quantize_block(const RawBlock<SRC>& raw, uint4& codes, uint32_t& sbyte) {
    uint32_t w[4];
    if constexpr (SRC == kBF16) {
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) { v[i] = raw.a.v[i]; v[8 + i] = raw.b.v[i]; }
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = __vmaxu2(m, v[i] & 0x7fff7fffu);
        const int e = mx_exponent_from_amax_bits(max(m & 0xffffu, m >> 16) << 16);
        sbyte = uint32_t(e + 127);
        const uint64_t inv2 = f32x2_splat(exp2i(-e));   // exact power of two: x * inv is exact or below E2M1's range
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[2 * j] = u2f(v[4 * k + j] << 16);
                f[2 * j + 1] = u2f(v[4 * k + j] & 0xffff0000u);
                mul_f32x2(f[2 * j], f[2 * j + 1], inv2);
            }
            w[k] = cvt_e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
        }
    } else if constexpr (SRC == kFP32) {
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) m = max(m, raw.a[i].v[j] & 0x7fffffffu);
        const int e = mx_exponent_from_amax_bits(m);
        sbyte = uint32_t(e + 127);
        const uint64_t inv2 = f32x2_splat(exp2i(-e));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = u2f(raw.a[k].v[j]);
#pragma unroll
            for (int j = 0; j < 8; j += 2) mul_f32x2(f[j], f[j + 1], inv2);
            w[k] = cvt_e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
        }
    } else {
        const float ts = raw.ts;
        // Decode the 32 codes to FP16 pairs (exact: E4M3 is a subset of FP16).
        // The FP32 product with the tile scale is monotone in the magnitude, so
        // the block amax is the product of the largest |code| (found on the
        // FP16 pairs).
        uint32_t h[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n"
                " cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
                : "=r"(h[2 * i]), "=r"(h[2 * i + 1]) : "r"(raw.a.v[i]));
        }
        // max of magnitudes, two chains (max.xorsign.abs: |result| = max(|a|, |b|))
        uint32_t m0, m1, hm;
        asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(m0) : "r"(h[0]), "r"(h[1]));
        asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(m1) : "r"(h[2]), "r"(h[3]));
#pragma unroll
        for (int i = 4; i < 16; i += 2) {
            asm("max.xorsign.abs.f16x2 %0, %0, %1;" : "+r"(m0) : "r"(h[i]));
            asm("max.xorsign.abs.f16x2 %0, %0, %1;" : "+r"(m1) : "r"(h[i + 1]));
        }
        asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(hm) : "r"(m0), "r"(m1));
        asm("abs.f16x2 %0, %0;" : "+r"(hm));
        float mlo, mhi;
        asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.f32.f16 %0, lo;\n cvt.f32.f16 %1, hi;\n}"
            : "=f"(mlo), "=f"(mhi) : "r"(hm));
        const float amax = fabsf(__fmul_rn(fmaxf(mlo, mhi), ts));
        const int e = mx_exponent_from_amax_bits(f2u(amax));
        sbyte = uint32_t(e + 127);
        const float inv = exp2i(-e);
        if (fabsf(ts) >= 0x1p-117f) {
            // Every non-zero product decode(e4m3) * ts is a normal FP32, so
            // fl(fl(d * ts) * 2^-E) == fl(d * (ts * 2^-E)) whenever the result
            // is normal, and both lie below E2M1's smallest step otherwise:
            // one multiply by the exact ts * 2^-E gives the same codes.
            const float sc = amax == 0.0f ? copysignf(1.0f, ts) : __fmul_rn(ts, inv);
            const uint64_t sc2 = f32x2_splat(sc);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float f[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) f16x2_mul_f32x2(h[4 * k + j], sc2, f[2 * j], f[2 * j + 1]);
                w[k] = cvt_e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
            }
        } else {
            // tiny tile scale: products may be subnormal; round them first
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float f[4], g[4];
                e4m3x4_to_f32(raw.a.v[2 * k], f);
                e4m3x4_to_f32(raw.a.v[2 * k + 1], g);
                w[k] = cvt_e2m1x8(__fmul_rn(__fmul_rn(f[0], ts), inv), __fmul_rn(__fmul_rn(f[1], ts), inv),
                                  __fmul_rn(__fmul_rn(f[2], ts), inv), __fmul_rn(__fmul_rn(f[3], ts), inv),
                                  __fmul_rn(__fmul_rn(g[0], ts), inv), __fmul_rn(__fmul_rn(g[1], ts), inv),
                                  __fmul_rn(__fmul_rn(g[2], ts), inv), __fmul_rn(__fmul_rn(g[3], ts), inv));
            }
        }
    }
    codes = make_uint4(w[0], w[1], w[2], w[3]);
}

template <int SRC>
__device__ __forceinline__ void store_block(uint8_t* __restrict__ q, uint8_t* __restrict__ s, int64_t r, uint32_t b,
                                            uint32_t bpr, int mma_layout, const uint4& codes, uint32_t sbyte) {
    *reinterpret_cast<uint4*>(q + r * (uint64_t(bpr) * 16) + uint64_t(b) * 16) = codes;
    const uint64_t so = mma_layout ? mma_scale_offset(uint64_t(r), b, bpr) : uint64_t(r) * bpr + b;
    s[so] = uint8_t(sbyte);
}

// Each thread owns block b of rows blockIdx.y, blockIdx.y + gridDim.y, ...;
// two rows are loaded before either is processed.
template <int SRC>
__global__ void __launch_bounds__(256) mx_quantize_kernel(
    const uint8_t* __restrict__ x, const float* __restrict__ tile_scale, int64_t rows,
    uint32_t bpr, int64_t ld_x_bytes, uint8_t* __restrict__ q, uint8_t* __restrict__ s,
    int mma_layout) {
    const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= bpr) return;
    const int64_t step = gridDim.y;
    for (int64_t r = blockIdx.y; r < rows; r += 2 * step) {
        const int64_t r2 = r + step;
        RawBlock<SRC> A, B;
        load_block<SRC>(x, tile_scale, r, b, bpr, ld_x_bytes, A);
        if (r2 < rows) load_block<SRC>(x, tile_scale, r2, b, bpr, ld_x_bytes, B);
        uint4 c;
        uint32_t sb;
        quantize_block<SRC>(A, c, sb);
        store_block<SRC>(q, s, r, b, bpr, mma_layout, c, sb);
        if (r2 < rows) {
            quantize_block<SRC>(B, c, sb);
            store_block<SRC>(q, s, r2, b, bpr, mma_layout, c, sb);
        }
    }
}

// E4M3 source with two adjacent blocks per thread (one 1x128 tile holds both):
// one tile-scale load, one index computation and 64 bytes of loads per row.
struct RawPair { u32x8 a, b; float ts; };

// A CTA covers rpc rows side by side (blockDim.x / rpc threads per row).
__global__ void __launch_bounds__(224, 4) mx_quantize_e4m3x2_kernel(
    const uint8_t* __restrict__ x, const float* __restrict__ tile_scale, int64_t rows,
    uint32_t bpr, int64_t ld_x, uint8_t* __restrict__ q, uint8_t* __restrict__ s, int mma_layout, int rpc) {
    allow_dependent_launch();
    grid_dependency_wait();             // the inputs may come from the previous kernel on the stream
    const uint32_t upc = blockDim.x / uint32_t(rpc);
    const uint32_t u = blockIdx.x * upc + threadIdx.x % upc;      // pair index in the row
    if (u >= (bpr >> 1)) return;
    const int64_t step = int64_t(gridDim.y) * rpc;
    auto load = [&](int64_t r, RawPair& p) {
        const uint8_t* src = x + r * ld_x + uint64_t(u) * 64;
        p.a = ldg256(src);
        p.b = ldg256(src + 32);
        p.ts = __ldg(tile_scale + r * (bpr >> 2) + (u >> 1));
    };
    auto process = [&](int64_t r, const RawPair& p) {
        RawBlock<kE4M3> blk;
        uint4 c0, c1;
        uint32_t s0, s1;
        blk.ts = p.ts;
        blk.a = p.a;
        quantize_block<kE4M3>(blk, c0, s0);
        blk.a = p.b;
        quantize_block<kE4M3>(blk, c1, s1);
        uint4* dst = reinterpret_cast<uint4*>(q + r * (uint64_t(bpr) * 16) + uint64_t(u) * 32);
        dst[0] = c0;
        dst[1] = c1;
        const uint32_t b0 = 2 * u;
        const uint64_t so = mma_layout ? mma_scale_offset(uint64_t(r), b0, bpr) : uint64_t(r) * bpr + b0;
        *reinterpret_cast<uint16_t*>(s + so) = uint16_t(s0 | (s1 << 8));   // blocks 2u, 2u+1 are adjacent bytes
    };
    for (int64_t r = int64_t(blockIdx.y) * rpc + threadIdx.x / upc; r < rows; r += 2 * step) {
        const int64_t r2 = r + step;
        RawPair A, B;
        load(r, A);
        if (r2 < rows) load(r2, B);
        process(r, A);
        if (r2 < rows) process(r2, B);
    }
}

// Column-wise MXFP4 of BF16 (block axis 0): the row-wise quantization of X^T,
// written in the transposed layout (q [cols, rows/2], scales [cols, rows/32])
// without materialising X^T.  Persistent CTAs run a shared-memory ring
// (ring.cuh): the producer thread brings 128-row x 128-column BF16 tiles in
// with TMA tensor copies (dense 256-byte rows, 3 stages); consumer thread t
// reads column pair 2(t % 64), 2(t % 64) + 1 over rows 32(t / 64) .. + 31
// with one 32-bit shared load per row (a warp reads 32 consecutive words, no
// bank conflicts), repacks the halves into the two columns' 32-element blocks
// and quantizes them with the row-wise rule.
constexpr int kMxColRows = 128, kMxColCols = 128, kMxColStages = 3;
constexpr uint32_t kMxColTileBytes = kMxColRows * kMxColCols * 2;

__global__ void __launch_bounds__(ring::kMaxThreads) mx_quantize_col_kernel(
    const __grid_constant__ CUtensorMap tmap, int64_t rows, int64_t cols, uint8_t* __restrict__ q,
    uint8_t* __restrict__ s, int mma_layout, uint32_t* status) {
    extern __shared__ __align__(128) uint8_t smem[];
    const ring::Ring rg = ring::make_ring(smem, kMxColTileBytes, kMxColStages);
    const int64_t ctiles = cols / kMxColCols, ngroups = (rows / kMxColRows) * ctiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmap);
            ring::produce(rg, ngroups, status, kStatusStreamTimeout, [&](uint8_t* st, uint32_t fb, int64_t g) {
                const int64_t rt = g / ctiles, ct = g - rt * ctiles;
                tc::mbar_arrive_expect_tx(fb, kMxColTileBytes);
                tc::tma_load_2d(tc::smem_u32(st), &tmap, fb, int(ct * kMxColCols), int(rt * kMxColRows));
            });
        }
        return;
    }
    const uint32_t t = threadIdx.x - 32, cp = t & 63u, k = t >> 6;
    const uint32_t spr = uint32_t(rows / 32);
    // output tile staging, block-major: block k's 16 code bytes of output row
    // cl at oq[k * 2048 + 16 * (cl ^ 2k)] (the XOR keeps the row-wise reads
    // conflict-free).  A thread stores its two rows 2 cp + h in the order
    // h = (cp / 4) % 2 first, so any 8 lanes of one store instruction hit 8
    // different 16-byte bank groups.  Scale byte (cl, k) at 4 (cl + cl / 32) + k
    // (one padding word per 32 rows: lanes cp and cp + 16 in different banks).
    __shared__ __align__(16) uint8_t oq[kMxColCols * 64];
    __shared__ __align__(16) uint8_t os[kMxColCols * 4 + 16];
    ring::consume_together(rg, ngroups, status, kStatusStreamTimeout, [&](uint8_t* st, int64_t g) {
        const int64_t rt = g / ctiles, ct = g - rt * ctiles;
        const int64_t r0 = rt * kMxColRows, c0 = ct * kMxColCols;
        const uint32_t base = tc::smem_u32(st);
        RawBlock<kBF16> A, B;                      // columns 2cp and 2cp + 1, rows 32k .. 32k + 31
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            uint32_t w0, w1;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w0) : "r"(base + (32 * k + 2 * j) * (kMxColCols * 2) + 4 * cp));
            asm volatile("ld.shared.b32 %0, [%1];"
                         : "=r"(w1) : "r"(base + (32 * k + 2 * j + 1) * (kMxColCols * 2) + 4 * cp));
            const uint32_t lo = __byte_perm(w0, w1, 0x5410), hi = __byte_perm(w0, w1, 0x7632);
            if (j < 8) { A.a.v[j] = lo; B.a.v[j] = hi; } else { A.b.v[j - 8] = lo; B.b.v[j - 8] = hi; }
        }
        const uint32_t blk = uint32_t(r0 / 32) + k;
        uint4 codes[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t sb;
            quantize_block<kBF16>(h ? B : A, codes[h], sb);
            const uint32_t cl = 2 * cp + h;
            if (mma_layout) s[mma_scale_offset(uint64_t(c0 + cl), blk, spr)] = uint8_t(sb);
            else os[4 * (cl + (cl >> 5)) + k] = uint8_t(sb);
        }
        const uint32_t h0 = (cp >> 2) & 1u;
#pragma unroll
        for (uint32_t i = 0; i < 2; ++i) {
            const uint32_t h = h0 ^ i, cl = 2 * cp + h;
            *reinterpret_cast<uint4*>(oq + k * 2048 + 16 * (cl ^ (2 * k))) = h ? codes[1] : codes[0];
        }
        // all 256 consumers staged the tile: 64 contiguous code bytes (and 4
        // scale bytes) per output row
        tc::named_bar_sync(2, blockDim.x - 32);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t u = t + 256 * i, row = u >> 2, ch = u & 3u;
            *reinterpret_cast<uint4*>(q + (c0 + row) * (rows / 2) + r0 / 2 + 16 * ch) =
                *reinterpret_cast<const uint4*>(oq + ch * 2048 + 16 * (row ^ (2 * ch)));
        }
        if (!mma_layout && t < kMxColCols)
            *reinterpret_cast<uint32_t*>(s + (c0 + t) * int64_t(spr) + r0 / 32) =
                *reinterpret_cast<const uint32_t*>(os + 4 * (t + (t >> 5)));
        tc::named_bar_sync(2, blockDim.x - 32);                // the staging may be rewritten
    });
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

template <typename Kernel>
inline dim3 grid_for_rows(Kernel k, int tpb, int64_t rows, int nx, int sms) {
    return dim3(unsigned(nx), row_grid_y(rows, nx, sms, resident_per_sm(k, tpb)), 1);
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
    if (block_axis == 0) {
        if (x_type != FP4Q_BF16) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "mx_quantize: block_axis 0 needs a BF16 source");
        if (rows % kMxColRows || cols % kMxColCols)
            return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "mx_quantize: block_axis 0 needs rows %% 128 == 0, cols %% 128 == 0");
        if (rows == 0 || cols == 0) return FP4Q_OK;
        if (!x || !q || !scales) return fail(FP4Q_ERR_INVALID_ARGUMENT, "mx_quantize: null pointer");
        if ((reinterpret_cast<uintptr_t>(x) & 31u) || (ld_x * 2) % 32 || !aligned16(q))
            return fail(FP4Q_ERR_MISALIGNED, "mx_quantize: x 32-byte aligned with ld_x %% 16 == 0, q 16-byte aligned");
        int sms = 0;
        fp4q_status st = current_device(&sms);
        if (st != FP4Q_OK) return st;
        CUtensorMap tmap;
        if ((st = ring::encode_bf16_tile_map(&tmap, x, rows, cols, ld_x, kMxColCols, kMxColRows)) != FP4Q_OK)
            return st;
        const uint32_t smem = ring::smem_bytes(kMxColTileBytes, kMxColStages);
        const int per_sm = resident_per_sm_smem(mx_quantize_col_kernel, ring::kMaxThreads, smem);
        const int64_t ngroups = (rows / kMxColRows) * (cols / kMxColCols);
        const int64_t grid = std::min<int64_t>(ngroups, int64_t(per_sm) * sms);
        mx_quantize_col_kernel<<<unsigned(grid), ring::kMaxThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
            tmap, rows, cols, q, scales, layout == FP4Q_SCALES_MMA, status_word());
        return check_launch("mx_quantize (block_axis 0)");
    }
    if (block_axis != 1) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "mx_quantize: block_axis must be 0 or 1");
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
    int sms = 0;
    fp4q_status st = current_device(&sms);
    if (st != FP4Q_OK) return st;
    const uint32_t bpr = uint32_t(cols / 32);
    int tpb, nx;
    row_launch_shape(bpr, &tpb, &nx);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    const int mma = layout == FP4Q_SCALES_MMA;
    switch (x_type) {
        case FP4Q_BF16: {
            dim3 grid = grid_for_rows(mx_quantize_kernel<kBF16>, tpb, rows, nx, sms);
            mx_quantize_kernel<kBF16><<<grid, tpb, 0, s>>>(xb, nullptr, rows, bpr, ld_x * 2, q, scales, mma);
            break;
        }
        case FP4Q_FP32: {
            dim3 grid = grid_for_rows(mx_quantize_kernel<kFP32>, tpb, rows, nx, sms);
            mx_quantize_kernel<kFP32><<<grid, tpb, 0, s>>>(xb, nullptr, rows, bpr, ld_x * 4, q, scales, mma);
            break;
        }
        default: {
            int tpb2, nx2, rpc;
            packed_row_shape(bpr / 2, &tpb2, &nx2, &rpc, 224);       // at most 224 threads: 4 CTAs per SM
            dim3 grid = grid_for_rows(mx_quantize_e4m3x2_kernel, tpb2, (rows + rpc - 1) / rpc, nx2, sms);
            const cudaError_t e = launch_overlapped(mx_quantize_e4m3x2_kernel, grid, dim3(tpb2), 0, s, xb, tile_scale,
                                                    rows, bpr, ld_x, q, scales, mma, rpc);
            if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "mx_quantize: %s", cudaGetErrorString(e));
            break;
        }
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
    int sms = 0;
    fp4q_status st = current_device(&sms);
    if (st != FP4Q_OK) return st;
    const uint32_t bpr = uint32_t(cols / 32);
    int tpb, nx;
    row_launch_shape(bpr, &tpb, &nx);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (y_type == FP4Q_BF16)
        mx_dequantize_kernel<true><<<grid_for_rows(mx_dequantize_kernel<true>, tpb, rows, nx, sms), tpb, 0, s>>>(
            q, scales, rows, bpr, static_cast<uint8_t*>(y));
    else
        mx_dequantize_kernel<false><<<grid_for_rows(mx_dequantize_kernel<false>, tpb, rows, nx, sms), tpb, 0, s>>>(
            q, scales, rows, bpr, static_cast<uint8_t*>(y));
    return check_launch("mx_dequantize");
}
