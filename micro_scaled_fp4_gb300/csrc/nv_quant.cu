// NVFP4 quantize of BF16 with an optional 16-point random Hadamard
// transform and round-to-nearest-even or Philox stochastic rounding.
//
// "Pretraining Large Language Models with NVFP4", technical summary:
//  2.A  16-element E2M1 blocks, one E4M3 scale per block and one FP32
//       scale per tensor (two-level scaling);
//  2.B  random Hadamard transforms on the weight-gradient inputs to spread
//       outliers, stochastic rounding (unbiased) on gradients.
//
// Two passes over the input (the tensor amax must be known before any block
// scale): pass 1 rotates and reduces max|y| into a 32-bit word of the caller's
// workspace (atomicMax on the float bits of non-negative values); pass 2
// rotates again and quantizes.  With a caller-supplied amax only pass 2 runs.
// One thread owns one 16-element block = one Hadamard tile: a single 256-bit
// load, the butterflies in registers, the block amax in-thread, 8 bytes of
// codes and one scale byte out.  The FP32 steps use explicit round-to-nearest
// intrinsics so that no contraction or reassociation changes a result.
#include <algorithm>

#include "common.cuh"
#include "ring.cuh"

namespace fp4q {
namespace {

// (a0, a1), (b0, b1) -> (a0 + b0, a1 + b1), (a0 - b0, a1 - b1): two butterflies
// in packed FP32 pairs (add / sub .rn.f32x2: each lane an IEEE round-to-nearest
// operation, the same results as the scalar forms).
__device__ __forceinline__ void butterfly_f32x2(float& a0, float& a1, float& b0, float& b1) {
    asm("{\n .reg .b64 x, y, s, t;\n mov.b64 x, {%0, %1};\n mov.b64 y, {%2, %3};\n"
        " add.rn.f32x2 s, x, y;\n sub.rn.f32x2 t, x, y;\n mov.b64 {%0, %1}, s;\n mov.b64 {%2, %3}, t;\n}"
        : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

// (1/4) H16 diag(d) x, d_j = -1 iff bit j of `signs` is set.  Butterflies with
// strides 1, 2, 4, 8 map (a, b) -> (a + b, a - b) in FP32; strides 2, 4 and 8
// pair elements (i, i + 1) with (i + h, i + h + 1) and run as packed pairs, and
// so does the final x 1/4.  SKIP_ZERO: no sign flips when `signs` is 0 (the
// deterministic H16; a branch uniform over the grid).  The column kernels,
// which serve the Wgrad operands with the deterministic H16, take it; the row
// kernels keep the unconditional flips.
template <bool SKIP_ZERO = false>
__device__ __forceinline__ void rht16(float (&t)[16], uint32_t signs) {
    if (!SKIP_ZERO || signs) {
#pragma unroll
        for (int j = 0; j < 16; ++j) t[j] = u2f(f2u(t[j]) ^ (((signs >> j) & 1u) << 31));
    }
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float a = t[i], b = t[i + 1];
        t[i] = __fadd_rn(a, b);
        t[i + 1] = __fsub_rn(a, b);
    }
#pragma unroll
    for (int h = 2; h < 16; h <<= 1)
#pragma unroll
        for (int i = 0; i < 16; i += 2)
            if (!(i & h)) butterfly_f32x2(t[i], t[i + 1], t[i + h], t[i + h + 1]);
    const uint64_t quarter = f32x2_splat(0.25f);
#pragma unroll
    for (int i = 0; i < 16; i += 2) mul_f32x2(t[i], t[i + 1], quarter);
}

__device__ __forceinline__ uint32_t rht_signs(uint64_t seed) {
    return philox4x32_10(make_uint4(0, 0, 0, 0), uint32_t(seed), uint32_t(seed >> 32)).x & 0xffffu;
}

// 16 BF16 values (32 bytes) -> FP32.
__device__ __forceinline__ void unpack_tile(const u32x8& a, float (&t)[16]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        t[2 * i] = u2f(a.v[i] << 16);
        t[2 * i + 1] = u2f(a.v[i] & 0xffff0000u);
    }
}

// The sign flips of the RHT as eight pairs of +-1.0 (d_j = -1 iff bit j of
// `signs`), for packed multiplies: exact, and on the FMA pipe where the bit
// flips would take the integer pipe.
struct SignPairs {
    uint64_t p[8];
};
__device__ __forceinline__ SignPairs sign_pairs(uint32_t signs) {
    SignPairs sp;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float lo = ((signs >> (2 * i)) & 1u) ? -1.0f : 1.0f, hi = ((signs >> (2 * i + 1)) & 1u) ? -1.0f : 1.0f;
        asm("mov.b64 %0, {%1, %2};" : "=l"(sp.p[i]) : "f"(lo), "f"(hi));
    }
    return sp;
}
// rht16 with the sign flips given as packed pairs.
__device__ __forceinline__ void rht16_pairs(float (&t)[16], const SignPairs& sp) {
#pragma unroll
    for (int i = 0; i < 8; ++i) mul_f32x2(t[2 * i], t[2 * i + 1], sp.p[i]);
    rht16<true>(t, 0u);
}

__global__ void __launch_bounds__(256) nv_amax_kernel(const uint8_t* __restrict__ x, int64_t rows,
                                                      uint32_t tpr, int64_t ld_x_bytes, int rht,
                                                      uint64_t rht_seed, uint32_t* __restrict__ amax_bits) {
    const uint32_t signs = rht == 1 ? rht_signs(rht_seed) : 0u;
    const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    float fm = 0.0f;
    if (b < tpr) {
        const SignPairs sp = sign_pairs(signs);
        const uint8_t* col = x + uint64_t(b) * 32;
        auto take = [&](const u32x8& v) {
            float t[16];
            unpack_tile(v, t);
            if (rht) rht16_pairs(t, sp);
#pragma unroll
            for (int j = 0; j < 16; ++j) fm = fmaxf(fm, fabsf(t[j]));
        };
        // four of the thread's rows per iteration, their loads issued together
        // (one load in flight per thread left the pass waiting on memory)
        const int64_t g = gridDim.y;
        int64_t r = blockIdx.y;
        for (; r + 3 * g < rows; r += 4 * g) {
            const u32x8 v0 = ldg256(col + r * ld_x_bytes), v1 = ldg256(col + (r + g) * ld_x_bytes);
            const u32x8 v2 = ldg256(col + (r + 2 * g) * ld_x_bytes), v3 = ldg256(col + (r + 3 * g) * ld_x_bytes);
            take(v0);
            take(v1);
            take(v2);
            take(v3);
        }
        for (; r < rows; r += g) take(ldg256(col + r * ld_x_bytes));
    }
    uint32_t m = f2u(fm);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ uint32_t wmax[8];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t v = 0;
        for (int w = 0; w < int(blockDim.x >> 5); ++w) v = max(v, wmax[w]);
        if (v) atomicMax(amax_bits, v);
    }
}

// Stochastic rounding of v onto E2M1 with the 32-bit word r: up iff
// r < frac * 2^32, frac the exact position of |v| between its two grid
// neighbours; |v| >= 6 saturates; the sign is kept.  Returns the 4-bit code.
// Integer form on the FP32 bits u of a = min(|v|, 6), without branches (the
// clamp makes 6 and above land on code 7 with nothing to round up): for a in
// [2^k, 2^(k+1)), k >= 0, the grid points are 2^k and 1.5 * 2^k (step
// 2^(k-1)), the code below a is 2(k + 1) + (mantissa bit 22) = (u >> 22) - 252
// and frac * 2^32 = u << 10 (the mantissa bits below bit 22); in [0.5, 1) the
// step is 0.5 from 0.5 (code 1), frac * 2^32 = u << 9; below 0.5 the step is
// 0.5 from 0 and frac * 2^32 = a * 2^33 (exact), whose ceiling decides the
// strict comparison.
__device__ __forceinline__ uint32_t sr_e2m1_code(float v, uint32_t r) {
    const float a = fminf(fabsf(v), 6.0f);
    const uint32_t u = f2u(a);
    const uint32_t code_hi = uint32_t(max(int(u >> 22) - 252, 1));
    const uint32_t thr_hi = u << (u >= 0x3f800000u ? 10 : 9);
    const uint32_t thr_lo = __float2uint_ru(__fmul_rn(a, 8589934592.0f));   // a * 2^33, < 2^32 below 0.5
    const bool lt_half = u < 0x3f000000u;
    const uint32_t code = lt_half ? 0u : code_hi;
    const uint32_t thr = lt_half ? thr_lo : thr_hi;
    return ((f2u(v) >> 28) & 8u) | (code + (r < thr ? 1u : 0u));
}

// Magnitude (the low 3 bits) of sr_e2m1_code(v, r); the caller supplies the
// sign bit, e.g. from the RNE code of the same v (the RNE convert keeps the
// sign of v, also for results that round to zero).
__device__ __forceinline__ uint32_t sr_e2m1_mag(float v, uint32_t r) {
    const float a = fminf(fabsf(v), 6.0f);
    const uint32_t u = f2u(a);
    const uint32_t code_hi = uint32_t(max(int(u >> 22) - 252, 1));
    const uint32_t thr_hi = u << (u >= 0x3f800000u ? 10 : 9);
    const uint32_t thr_lo = __float2uint_ru(__fmul_rn(a, 8589934592.0f));   // a * 2^33, < 2^32 below 0.5
    const bool lt_half = u < 0x3f000000u;
    const uint32_t code = lt_half ? 0u : code_hi;
    const uint32_t thr = lt_half ? thr_lo : thr_hi;
    return code + (r < thr ? 1u : 0u);
}

// The ten round keys of Philox4x32-10 for one seed (key schedule (k0, k1) +=
// (0x9E3779B9, 0xBB67AE85) per round), computed on the host and passed as a
// kernel parameter, so that the rounds read them as constants.
struct PhiloxKeys {
    uint32_t k0[10], k1[10];
};

inline PhiloxKeys philox_keys(uint64_t seed) {
    PhiloxKeys k;
    uint32_t a = uint32_t(seed), b = uint32_t(seed >> 32);
    for (int i = 0; i < 10; ++i) {
        k.k0[i] = a;
        k.k1[i] = b;
        a += 0x9E3779B9u;
        b += 0xBB67AE85u;
    }
    return k;
}

// Philox4x32-10 of the counter (c0, c1, 0, 0) under the keys K: each round is
// two 32 x 32 -> 64-bit products (as separate high and low halves, 2 % faster
// in the SR pass than 64-bit products) and two three-way XORs.
__device__ __forceinline__ uint4 philox_ctr64(uint32_t c0, uint32_t c1, const PhiloxKeys& K) {
    uint32_t x = c0, y = c1, z = 0, w = 0;
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        const uint32_t h0 = __umulhi(0xD2511F53u, x), l0 = 0xD2511F53u * x;
        const uint32_t h1 = __umulhi(0xCD9E8D57u, z), l1 = 0xCD9E8D57u * z;
        const uint32_t nx = h1 ^ y ^ K.k0[i];
        const uint32_t nz = h0 ^ w ^ K.k1[i];
        y = l1;
        w = l0;
        x = nx;
        z = nz;
    }
    return make_uint4(x, y, z, w);
}

// Rounding of the quantize pass: kRne, kSr, or kSrRne (both, over the same
// scales from one read and one rotation: SR codes into q, RNE codes into q2).
enum NvMode { kRne = 0, kSr = 1, kSrRne = 2 };

template <int MODE>
__global__ void __launch_bounds__(256) nv_quant_kernel(
    const uint8_t* __restrict__ x, int64_t rows, uint32_t tpr, int64_t ld_x_bytes, int rht,
    uint64_t rht_seed, const PhiloxKeys sr_keys, const float* __restrict__ amax_ptr, float* __restrict__ amax_out,
    float* __restrict__ st_out, uint8_t* __restrict__ q, uint8_t* __restrict__ q2, uint8_t* __restrict__ s,
    int mma_layout) {
    const uint32_t signs = rht == 1 ? rht_signs(rht_seed) : 0u;
    const float amax = *amax_ptr;
    const float s_t = __fdiv_rn(amax, 2688.0f);        // 6 * 448
    const float denom = __fmul_rn(6.0f, s_t);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        if (amax_out) *amax_out = amax;
        *st_out = s_t;
    }
    const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= tpr) return;
    const uint64_t cols = uint64_t(tpr) * 16;
    const SignPairs sp = sign_pairs(signs);
    auto quantize_row = [&](int64_t r, float (&t)[16]) {
        if (rht) rht16_pairs(t, sp);
        float am = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) am = fmaxf(am, fabsf(t[j]));
        const uint32_t ab = f2u(am);
        uint32_t sb = 0;
        float rcp = 0.0f;
        if (s_t > 0.0f) {
            sb = cvt_e4m3(__fdiv_rn(u2f(ab), denom));
            if (sb & 0x7fu) rcp = __frcp_rn(__fmul_rn(e4m3x2_to_f32x2(sb).x, s_t));
        }
        uint32_t words[2], words2[2];
        if (rcp == 0.0f) {
            // zero tensor or block scale underflow: signed-zero codes
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                uint32_t w = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) w |= ((f2u(t[8 * k + j]) >> 31) << 3) << (4 * j);
                words[k] = w;
                words2[k] = w;
            }
        } else {
            // v = y * (1 / sf), the pairs as packed IEEE products
            float v[16];
            const uint64_t rcp2 = f32x2_splat(rcp);
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                v[j] = t[j];
                v[j + 1] = t[j + 1];
                mul_f32x2(v[j], v[j + 1], rcp2);
            }
            // RNE codes: every mode computes them, the SR codes take their signs
            uint32_t(&rw)[2] = MODE == kRne ? words : words2;
#pragma unroll
            for (int k = 0; k < 2; ++k)
                rw[k] = cvt_e2m1x8(v[8 * k], v[8 * k + 1], v[8 * k + 2], v[8 * k + 3], v[8 * k + 4], v[8 * k + 5],
                                   v[8 * k + 6], v[8 * k + 7]);
            if constexpr (MODE != kRne) {
                const uint64_t i0 = uint64_t(r) * cols + uint64_t(b) * 16;   // linear index, % 16 == 0
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    uint32_t w = words2[k] & 0x88888888u;                    // the signs
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t ctr = (i0 >> 2) + uint64_t(2 * k + h);
                        const uint4 rnd = philox_ctr64(uint32_t(ctr), uint32_t(ctr >> 32), sr_keys);
                        const int base = 8 * k + 4 * h;
                        const uint32_t rr[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) w += sr_e2m1_mag(v[base + e], rr[e]) << (4 * (4 * h + e));
                    }
                    words[k] = w;
                }
            }
        }
        *reinterpret_cast<uint2*>(q + uint64_t(r) * (cols / 2) + uint64_t(b) * 8) = make_uint2(words[0], words[1]);
        if constexpr (MODE == kSrRne)
            *reinterpret_cast<uint2*>(q2 + uint64_t(r) * (cols / 2) + uint64_t(b) * 8) =
                make_uint2(words2[0], words2[1]);
        const uint64_t so = mma_layout ? mma_scale_offset(uint64_t(r), b, tpr) : uint64_t(r) * tpr + b;
        s[so] = uint8_t(sb);
    };
    // the thread's next row is loaded before the current one is processed, so a
    // load stays in flight while the thread computes (quantize pass 67.7 -> 66.2 us
    // RNE, 212 -> 206 us SR on the 8192 x 14336 gradient)
    const uint8_t* col = x + uint64_t(b) * 32;
    u32x8 next;
    if (blockIdx.y < rows) next = ldg256(col + int64_t(blockIdx.y) * ld_x_bytes);
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const u32x8 cur = next;
        if (r + gridDim.y < rows) next = ldg256(col + (r + gridDim.y) * ld_x_bytes);
        float t[16];
        unpack_tile(cur, t);
        quantize_row(r, t);
    }
}

// Scale, reciprocal and codes of one 16-element block y (FP32) under the
// tensor scale s_t, with the rules of nv_quant_kernel; `ab` is the block's
// amax bits (the 2D form passes its tile's).  SR draws the words of linear
// elements i0 .. i0 + 15 (i0 % 16 == 0).
template <bool SR>
__device__ __forceinline__ uint32_t nv_block_codes(const float (&t)[16], uint32_t ab, float s_t, float denom,
                                                   uint64_t i0, const PhiloxKeys& sr_keys, uint2& words) {
    uint32_t sb = 0;
    float rcp = 0.0f;
    if (s_t > 0.0f) {
        sb = cvt_e4m3(__fdiv_rn(u2f(ab), denom));
        if (sb & 0x7fu) rcp = __frcp_rn(__fmul_rn(e4m3x2_to_f32x2(sb).x, s_t));
    }
    uint32_t w[2];
    if (rcp == 0.0f) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t v = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) v |= ((f2u(t[8 * k + j]) >> 31) << 3) << (4 * j);
            w[k] = v;
        }
    } else if constexpr (!SR) {
#pragma unroll
        for (int k = 0; k < 2; ++k)
            w[k] = cvt_e2m1x8(__fmul_rn(t[8 * k], rcp), __fmul_rn(t[8 * k + 1], rcp), __fmul_rn(t[8 * k + 2], rcp),
                              __fmul_rn(t[8 * k + 3], rcp), __fmul_rn(t[8 * k + 4], rcp),
                              __fmul_rn(t[8 * k + 5], rcp), __fmul_rn(t[8 * k + 6], rcp),
                              __fmul_rn(t[8 * k + 7], rcp));
    } else {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t v = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint64_t ctr = (i0 >> 2) + uint64_t(2 * k + h);
                const uint4 rnd = philox_ctr64(uint32_t(ctr), uint32_t(ctr >> 32), sr_keys);
                const uint32_t rr[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    v |= sr_e2m1_code(__fmul_rn(t[8 * k + 4 * h + e], rcp), rr[e]) << (4 * (4 * h + e));
            }
            w[k] = v;
        }
    }
    words = make_uint2(w[0], w[1]);
    return sb;
}

// `writer_tid`: the thread of CTA 0 that publishes amax and s_t.
__device__ __forceinline__ float nv_tensor_scale(const float* amax_ptr, float* amax_out, float* st_out,
                                                 uint32_t writer_tid = 0) {
    const float amax = *amax_ptr;
    const float s_t = __fdiv_rn(amax, 2688.0f);        // 6 * 448
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == writer_tid) {
        if (amax_out) *amax_out = amax;
        *st_out = s_t;
    }
    return s_t;
}

// 2D (16 x 16) block scaling for weights ("Pretraining Large Language Models
// with NVFP4", 2.B): one E4M3 scale per 16 x 16 tile from the tile amax, the
// 1D rules otherwise, no rotation; every row of the tile stores the same scale
// byte ([rows, cols/16] layout).  A CTA takes 16 rows x 16 blocks (256
// columns): warp w holds blocks 2w, 2w + 1, lane 16 h + j row j of block 2w + h
// (each row's 64 bytes read together), and the tile amax is a max over the
// half-warp.  Codes and scales are staged per CTA tile (block-major, rows
// XOR-swizzled by the block index: conflict-free both ways) so that each row's
// 128 code bytes go out contiguously.
template <bool SR>
__global__ void __launch_bounds__(256) nv_quant_2d_kernel(
    const uint8_t* __restrict__ x, int64_t rows, uint32_t tpr, int64_t ld_x_bytes, const PhiloxKeys sr_keys,
    const float* __restrict__ amax_ptr, float* __restrict__ amax_out, float* __restrict__ st_out,
    uint8_t* __restrict__ q, uint8_t* __restrict__ s, int mma_layout) {
    __shared__ __align__(16) uint8_t oq[16 * 128];
    __shared__ uint8_t os[16 * 16];
    const float s_t = nv_tensor_scale(amax_ptr, amax_out, st_out);
    const float denom = __fmul_rn(6.0f, s_t);
    const uint32_t ctiles = (tpr + 15) / 16;
    const int64_t ntiles = (rows / 16) * int64_t(ctiles);
    const uint32_t warp = threadIdx.x >> 5, j = threadIdx.x & 15u, h = (threadIdx.x >> 4) & 1u;
    const uint32_t bl = 2 * warp + h;                              // block within the CTA tile
    const uint64_t cols = uint64_t(tpr) * 16;
    // the next tile's 32 bytes are loaded before the current tile is processed,
    // so a load is in flight across the two block barriers of each tile
    auto fetch = [&](int64_t tile, u32x8& raw) {
        const int64_t tr = tile / ctiles;
        const uint32_t b = 16 * uint32_t(tile - tr * ctiles) + bl;
        if (tile < ntiles && b < tpr) raw = ldg256(x + (tr * 16 + j) * ld_x_bytes + uint64_t(b) * 32);
    };
    u32x8 next{};
    fetch(blockIdx.x, next);
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t tr = tile / ctiles;
        const uint32_t ct = uint32_t(tile - tr * ctiles);
        const uint32_t b = 16 * ct + bl, nblk = min(16u, tpr - 16 * ct);
        const bool valid = b < tpr;
        const int64_t r = tr * 16 + j;
        const u32x8 cur = next;
        fetch(tile + gridDim.x, next);
        float t[16];
        uint32_t ab = 0;
        if (valid) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                t[2 * i] = u2f(cur.v[i] << 16);
                t[2 * i + 1] = u2f(cur.v[i] & 0xffff0000u);
            }
            float fm = 0.0f;
#pragma unroll
            for (int e = 0; e < 16; ++e) fm = fmaxf(fm, fabsf(t[e]));
            ab = f2u(fm);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, o));
        if (valid) {
            uint2 words;
            const uint32_t sb = nv_block_codes<SR>(t, ab, s_t, denom, uint64_t(r) * cols + uint64_t(b) * 16, sr_keys,
                                                   words);
            *reinterpret_cast<uint2*>(oq + bl * 128 + 8 * (j ^ bl)) = words;     // block-major, XOR-swizzled rows
            if (mma_layout) s[mma_scale_offset(uint64_t(r), b, tpr)] = uint8_t(sb);
            else os[j * 16 + (bl ^ (4 * (j >> 3)))] = uint8_t(sb);    // rows j, j + 8 in different banks
        }
        __syncthreads();
        {   // row t / 16, block t % 16: 8 code bytes (16 threads = one row's 128 bytes)
            const uint32_t row = threadIdx.x >> 4, blk = threadIdx.x & 15u;
            if (blk < nblk) {
                const int64_t rr = tr * 16 + row;
                *reinterpret_cast<uint2*>(q + rr * int64_t(cols / 2) + (16 * ct + blk) * 8) =
                    *reinterpret_cast<const uint2*>(oq + blk * 128 + 8 * (row ^ blk));
                if (!mma_layout) s[rr * int64_t(tpr) + 16 * ct + blk] = os[row * 16 + (blk ^ (4 * (row >> 3)))];
            }
        }
        __syncthreads();
    }
}

// Column-wise NVFP4 (block axis 0): the row-wise quantization of X^T, written
// in the transposed layout, without materialising X^T.  Persistent CTAs run a
// shared-memory ring (ring.cuh): the producer thread brings 128-row x 64-column
// BF16 tiles in with TMA tensor copies (dense 128-byte rows, 4 stages);
// consumer thread t reads column pair 2(t % 32), 2(t % 32) + 1 over rows
// 16(t / 32) .. + 15 (one 32-bit shared load per row; a warp reads 32
// consecutive words, no bank conflicts) and quantizes the two 16-element
// blocks -- rotated along axis 0 when rht != 0 -- into rows c of
// q [cols, rows/2] and scales [cols, rows/16].  MODE 0: tensor amax only;
// 1: RNE; 2: SR (linear element index of X^T).
constexpr int kColRows = 128, kColCols = 64;
constexpr uint32_t kColTileBytes = kColRows * kColCols * 2;

template <int MODE>
__global__ void __launch_bounds__(ring::kMaxThreads, MODE == 2 ? 2 : 3) nv_col_kernel(
    const __grid_constant__ CUtensorMap tmap, int64_t rows, int64_t cols, int rht, uint64_t rht_seed,
    const PhiloxKeys sr_keys, const float* __restrict__ amax_ptr, float* __restrict__ amax_out,
    float* __restrict__ st_out, uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ q,
    uint8_t* __restrict__ s, int mma_layout, uint32_t* status) {
    extern __shared__ __align__(128) uint8_t smem[];
    const ring::Ring rg = ring::make_ring(smem, kColTileBytes);
    const int64_t ctiles = cols / kColCols, ngroups = (rows / kColRows) * ctiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmap);
            ring::produce(rg, ngroups, status, kStatusStreamTimeout, [&](uint8_t* st, uint32_t fb, int64_t g) {
                const int64_t rt = g / ctiles, ct = g - rt * ctiles;
                tc::mbar_arrive_expect_tx(fb, kColTileBytes);
                tc::tma_load_2d(tc::smem_u32(st), &tmap, fb, int(ct * kColCols), int(rt * kColRows));
            });
        }
        return;
    }
    const uint32_t signs = rht == 1 ? rht_signs(rht_seed) : 0u;
    float s_t = 0.0f, denom = 0.0f;
    if constexpr (MODE != 0) {
        s_t = nv_tensor_scale(amax_ptr, amax_out, st_out, 32);      // thread 0 is the producer
        denom = __fmul_rn(6.0f, s_t);
    }
    const uint32_t t = threadIdx.x - 32, cp = t & 31u, k = t >> 5;
    const uint32_t spr = uint32_t(rows / 16);                 // scale columns per output row
    // output tile staging, block-major: block k's 8 code bytes of output row cl
    // at oq[k * 512 + 8 * (cl ^ 4 (k / 2))].  A thread writes its two rows
    // (2 cp, 2 cp + 1) as one 16-byte store (any 8 lanes: 8 different 16-byte
    // bank groups) and the row-wise reads (4 rows x 4 block pairs per 16
    // lanes) land on 16 different bank pairs.  Scale bytes: (cl, k) at
    // 8 cl + 4 (cl / 16) + k, which puts a warp's 32 stores in 32 banks.
    __shared__ __align__(16) uint8_t oq[kColCols * 64];
    __shared__ __align__(16) uint8_t os[kColCols * 8 + 16];
    uint32_t m_all = 0;
    ring::consume_together(rg, ngroups, status, kStatusStreamTimeout, [&](uint8_t* st, int64_t g) {
        const int64_t rt = g / ctiles, ct = g - rt * ctiles;
        const int64_t r0 = rt * kColRows, c0 = ct * kColCols;
        const uint32_t base = tc::smem_u32(st);
        float a[16], b[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            uint32_t w;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w) : "r"(base + (16 * k + j) * (kColCols * 2) + 4 * cp));
            a[j] = u2f(w << 16);
            b[j] = u2f(w & 0xffff0000u);
        }
        if (rht) {
            rht16<true>(a, signs);
            rht16<true>(b, signs);
        }
        float fa = 0.0f, fb = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            fa = fmaxf(fa, fabsf(a[j]));
            fb = fmaxf(fb, fabsf(b[j]));
        }
        const uint32_t ma = f2u(fa), mb = f2u(fb);
        if constexpr (MODE == 0) {
            m_all = max(m_all, max(ma, mb));
        } else {
            uint2 words[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t cl = 2 * cp + h;                         // output row within the tile
                const int64_t c = c0 + cl;
                const int64_t rb = r0 + 16 * k;                      // first row of the block
                const uint32_t sb = nv_block_codes<MODE == 2>(h ? b : a, h ? mb : ma, s_t, denom,
                                                             uint64_t(c) * uint64_t(rows) + uint64_t(rb), sr_keys,
                                                             words[h]);
                if (mma_layout) s[mma_scale_offset(uint64_t(c), uint32_t(rb / 16), spr)] = uint8_t(sb);
                else os[8 * cl + 4 * (cl >> 4) + k] = uint8_t(sb);
            }
            *reinterpret_cast<uint4*>(oq + k * 512 + 16 * (cp ^ (2 * (k >> 1)))) =
                make_uint4(words[0].x, words[0].y, words[1].x, words[1].y);
            // all 256 consumers staged the tile: write 64 contiguous code bytes
            // (and 8 scale bytes) per output row
            tc::named_bar_sync(2, blockDim.x - 32);
            const uint32_t row = t >> 2, ch = t & 3u;           // blocks 2ch, 2ch + 1 of output row `row`
            const uint2 lo = *reinterpret_cast<const uint2*>(oq + (2 * ch) * 512 + 8 * (row ^ (4 * ch)));
            const uint2 hi = *reinterpret_cast<const uint2*>(oq + (2 * ch + 1) * 512 + 8 * (row ^ (4 * ch)));
            *reinterpret_cast<uint4*>(q + (c0 + row) * (rows / 2) + r0 / 2 + 16 * ch) = make_uint4(lo.x, lo.y, hi.x, hi.y);
            if (!mma_layout && t < kColCols) {
                const uint32_t* sw = reinterpret_cast<const uint32_t*>(os + 8 * t + 4 * (t >> 4));
                *reinterpret_cast<uint2*>(s + (c0 + t) * int64_t(spr) + r0 / 16) = make_uint2(sw[0], sw[1]);
            }
            tc::named_bar_sync(2, blockDim.x - 32);            // the staging may be rewritten
        }
    });
    if constexpr (MODE == 0) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m_all = max(m_all, __shfl_xor_sync(0xffffffffu, m_all, o));
        if (lane == 0 && m_all) atomicMax(amax_bits, m_all);
    }
}

}  // namespace
}  // namespace fp4q

using namespace fp4q;

extern "C" size_t fp4q_nv_quantize_workspace_bytes(int64_t rows, int64_t cols) {
    (void)rows;
    (void)cols;
    return 256;   // one 32-bit amax word (padded)
}

// Common argument checks; *amax_ptr is amax_in or, after the amax pass that
// `amax_pass` launches, the workspace word.
namespace {
fp4q_status nv_prologue(const char* who, const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                        fp4q_rounding rounding, const float* amax_in, float* tensor_scale_out, uint8_t* q,
                        uint8_t* scales, fp4q_scale_layout layout, void* workspace, size_t workspace_bytes) {
    if (rounding != FP4Q_RNE && rounding != FP4Q_SR)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "%s: bad rounding mode", who);
    if (layout != FP4Q_SCALES_ROWMAJOR && layout != FP4Q_SCALES_MMA)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "%s: bad scale layout", who);
    if (rows < 0 || cols < 0 || ld_x < cols)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "%s: need rows >= 0, cols >= 0, ld_x >= cols", who);
    if (cols % 16) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "%s: cols %% 16 != 0", who);
    if (!tensor_scale_out) return fail(FP4Q_ERR_INVALID_ARGUMENT, "%s: tensor_scale_out is NULL", who);
    if (rows > 0 && cols > 0 && (!x || !q || !scales)) return fail(FP4Q_ERR_INVALID_ARGUMENT, "%s: null pointer", who);
    if (!amax_in && (!workspace || workspace_bytes < fp4q_nv_quantize_workspace_bytes(rows, cols)))
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "%s: workspace missing or too small", who);
    if ((reinterpret_cast<uintptr_t>(x) & 31u) || (ld_x * 2) % 32 || (q && !aligned16(q)) ||
        (workspace && !aligned16(workspace)))
        return fail(FP4Q_ERR_MISALIGNED, "%s: x 32-byte aligned with ld_x %% 16 == 0; q, workspace 16-byte aligned",
                    who);
    return FP4Q_OK;
}

fp4q_status zero_amax_word(void* workspace, cudaStream_t s, const char* who) {
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "%s: memset: %s", who, cudaGetErrorString(e));
    return FP4Q_OK;
}
}  // namespace

extern "C" fp4q_status fp4q_nv_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                        int block_axis, int rht, uint64_t rht_seed,
                                        fp4q_rounding rounding, uint64_t sr_seed, const float* amax_in,
                                        float* amax_out, float* tensor_scale_out, uint8_t* q,
                                        uint8_t* scales, fp4q_scale_layout layout, void* workspace,
                                        size_t workspace_bytes, fp4q_stream_t stream) {
    fp4q_status st = nv_prologue("nv_quantize", x, rows, cols, ld_x, rounding, amax_in, tensor_scale_out, q, scales,
                                 layout, workspace, workspace_bytes);
    if (st != FP4Q_OK) return st;
    if (rht < 0 || rht > 2) return fail(FP4Q_ERR_INVALID_ARGUMENT, "nv_quantize: rht must be 0, 1 or 2");
    if (block_axis != 0 && block_axis != 1) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "nv_quantize: block_axis 0 or 1");
    if (block_axis == 0 && (rows % kColRows || cols % kColCols))
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "nv_quantize: block_axis 0 needs rows %% 128 == 0, cols %% 64 == 0");
    int sms = 0;
    if ((st = current_device(&sms)) != FP4Q_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    const float* amax_ptr = amax_in;
    const int mma = layout == FP4Q_SCALES_MMA;
    const PhiloxKeys keys = philox_keys(sr_seed);
    if (block_axis == 0) {
        if (!amax_in) {
            uint32_t* w = static_cast<uint32_t*>(workspace);
            if ((st = zero_amax_word(w, s, "nv_quantize")) != FP4Q_OK) return st;
            amax_ptr = reinterpret_cast<const float*>(w);
        }
        if (rows == 0 || cols == 0) {
            nv_quant_kernel<kRne><<<1, 32, 0, s>>>(xb, 0, 0, 0, 0, 0, keys, amax_ptr, amax_out, tensor_scale_out, q,
                                                   nullptr, scales, 0);
            return check_launch("nv_quantize");
        }
        CUtensorMap tmap;
        if ((st = ring::encode_bf16_tile_map(&tmap, x, rows, cols, ld_x, kColCols, kColRows)) != FP4Q_OK) return st;
        const uint32_t smem = ring::smem_bytes(kColTileBytes);
        const int64_t ngroups = (rows / kColRows) * (cols / kColCols);
        auto launch = [&](auto kernel, uint32_t* bits) {
            const int per_sm = resident_per_sm_smem(kernel, ring::kMaxThreads, smem);
            const int64_t grid = std::min<int64_t>(ngroups, int64_t(per_sm) * sms);
            kernel<<<unsigned(grid), ring::kMaxThreads, smem, s>>>(tmap, rows, cols, rht, rht_seed, keys, amax_ptr,
                                                                    amax_out, tensor_scale_out, bits, q, scales, mma,
                                                                    status_word());
            return check_launch("nv_quantize (block_axis 0)");
        };
        if (!amax_in && (st = launch(nv_col_kernel<0>, static_cast<uint32_t*>(workspace))) != FP4Q_OK) return st;
        return rounding == FP4Q_SR ? launch(nv_col_kernel<2>, nullptr) : launch(nv_col_kernel<1>, nullptr);
    }
    const uint32_t tpr = uint32_t(cols / 16);
    int tpb = 32, nx = 1;
    if (tpr) row_launch_shape(tpr, &tpb, &nx);
    // grids sized by each kernel's own residency (the passes differ in registers)
    auto grid_for = [&](auto kernel) {
        return dim3(unsigned(nx), row_grid_y(rows, nx, sms, resident_per_sm(kernel, tpb)), 1);
    };
    if (!amax_in) {
        uint32_t* w = static_cast<uint32_t*>(workspace);
        if ((st = zero_amax_word(w, s, "nv_quantize")) != FP4Q_OK) return st;
        if (rows > 0 && cols > 0) {
            nv_amax_kernel<<<grid_for(nv_amax_kernel), tpb, 0, s>>>(xb, rows, tpr, ld_x * 2, rht, rht_seed, w);
            if ((st = check_launch("nv_quantize amax")) != FP4Q_OK) return st;
        }
        amax_ptr = reinterpret_cast<const float*>(w);
    }
    if (rows == 0 || cols == 0) {
        // still publish s_t (and amax) for an empty tensor: both are 0
        nv_quant_kernel<kRne><<<1, 32, 0, s>>>(xb, 0, 0, 0, 0, 0, keys, amax_ptr, amax_out, tensor_scale_out, q,
                                               nullptr, scales, 0);
        return check_launch("nv_quantize");
    }
    if (rounding == FP4Q_SR)
        nv_quant_kernel<kSr><<<grid_for(nv_quant_kernel<kSr>), tpb, 0, s>>>(
            xb, rows, tpr, ld_x * 2, rht, rht_seed, keys, amax_ptr, amax_out, tensor_scale_out, q, nullptr, scales,
            mma);
    else
        nv_quant_kernel<kRne><<<grid_for(nv_quant_kernel<kRne>), tpb, 0, s>>>(
            xb, rows, tpr, ld_x * 2, rht, rht_seed, keys, amax_ptr, amax_out, tensor_scale_out, q, nullptr, scales,
            mma);
    return check_launch("nv_quantize");
}

extern "C" fp4q_status fp4q_nv_quantize_sr_rne(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int rht,
                                               uint64_t rht_seed, uint64_t sr_seed, const float* amax_in,
                                               float* amax_out, float* tensor_scale_out, uint8_t* q_sr,
                                               uint8_t* q_rne, uint8_t* scales, fp4q_scale_layout layout,
                                               void* workspace, size_t workspace_bytes, fp4q_stream_t stream) {
    fp4q_status st = nv_prologue("nv_quantize_sr_rne", x, rows, cols, ld_x, FP4Q_SR, amax_in, tensor_scale_out, q_sr,
                                 scales, layout, workspace, workspace_bytes);
    if (st != FP4Q_OK) return st;
    if (rht < 0 || rht > 2) return fail(FP4Q_ERR_INVALID_ARGUMENT, "nv_quantize_sr_rne: rht must be 0, 1 or 2");
    if (rows > 0 && cols > 0 && !q_rne) return fail(FP4Q_ERR_INVALID_ARGUMENT, "nv_quantize_sr_rne: q_rne is NULL");
    if (q_rne && !aligned16(q_rne)) return fail(FP4Q_ERR_MISALIGNED, "nv_quantize_sr_rne: q_rne 16-byte aligned");
    int sms = 0;
    if ((st = current_device(&sms)) != FP4Q_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    const float* amax_ptr = amax_in;
    const PhiloxKeys keys = philox_keys(sr_seed);
    const uint32_t tpr = uint32_t(cols / 16);
    int tpb = 32, nx = 1;
    if (tpr) row_launch_shape(tpr, &tpb, &nx);
    auto grid_for = [&](auto kernel) {
        return dim3(unsigned(nx), row_grid_y(rows, nx, sms, resident_per_sm(kernel, tpb)), 1);
    };
    if (!amax_in) {
        uint32_t* w = static_cast<uint32_t*>(workspace);
        if ((st = zero_amax_word(w, s, "nv_quantize_sr_rne")) != FP4Q_OK) return st;
        if (rows > 0 && cols > 0) {
            nv_amax_kernel<<<grid_for(nv_amax_kernel), tpb, 0, s>>>(xb, rows, tpr, ld_x * 2, rht, rht_seed, w);
            if ((st = check_launch("nv_quantize_sr_rne amax")) != FP4Q_OK) return st;
        }
        amax_ptr = reinterpret_cast<const float*>(w);
    }
    if (rows == 0 || cols == 0) {
        nv_quant_kernel<kRne><<<1, 32, 0, s>>>(xb, 0, 0, 0, 0, 0, keys, amax_ptr, amax_out, tensor_scale_out, q_sr,
                                               nullptr, scales, 0);
        return check_launch("nv_quantize_sr_rne");
    }
    nv_quant_kernel<kSrRne><<<grid_for(nv_quant_kernel<kSrRne>), tpb, 0, s>>>(
        xb, rows, tpr, ld_x * 2, rht, rht_seed, keys, amax_ptr, amax_out, tensor_scale_out, q_sr, q_rne, scales,
        layout == FP4Q_SCALES_MMA);
    return check_launch("nv_quantize_sr_rne");
}

extern "C" fp4q_status fp4q_nv_quantize_2d(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                           fp4q_rounding rounding, uint64_t sr_seed, const float* amax_in,
                                           float* amax_out, float* tensor_scale_out, uint8_t* q, uint8_t* scales,
                                           fp4q_scale_layout layout, void* workspace, size_t workspace_bytes,
                                           fp4q_stream_t stream) {
    fp4q_status st = nv_prologue("nv_quantize_2d", x, rows, cols, ld_x, rounding, amax_in, tensor_scale_out, q,
                                 scales, layout, workspace, workspace_bytes);
    if (st != FP4Q_OK) return st;
    if (rows % 16) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "nv_quantize_2d: rows %% 16 != 0");
    int sms = 0;
    if ((st = current_device(&sms)) != FP4Q_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    const float* amax_ptr = amax_in;
    const PhiloxKeys keys = philox_keys(sr_seed);
    const uint32_t tpr = uint32_t(cols / 16);
    if (!amax_in) {
        uint32_t* w = static_cast<uint32_t*>(workspace);
        if ((st = zero_amax_word(w, s, "nv_quantize_2d")) != FP4Q_OK) return st;
        if (rows > 0 && cols > 0) {
            int tpb = 32, nx = 1;
            row_launch_shape(tpr, &tpb, &nx);
            dim3 grid(unsigned(nx), row_grid_y(rows, nx, sms, resident_per_sm(nv_amax_kernel, tpb)), 1);
            nv_amax_kernel<<<grid, tpb, 0, s>>>(xb, rows, tpr, ld_x * 2, 0, 0, w);
            if ((st = check_launch("nv_quantize_2d amax")) != FP4Q_OK) return st;
        }
        amax_ptr = reinterpret_cast<const float*>(w);
    }
    if (rows == 0 || cols == 0) {
        nv_quant_kernel<kRne><<<1, 32, 0, s>>>(xb, 0, 0, 0, 0, 0, keys, amax_ptr, amax_out, tensor_scale_out, q,
                                               nullptr, scales, 0);
        return check_launch("nv_quantize_2d");
    }
    const int mma = layout == FP4Q_SCALES_MMA;
    const int64_t tiles = (rows / 16) * int64_t((tpr + 15) / 16);       // 16 rows x 16 blocks
    // persistent grid sized by the instance's own residency
    auto grid_2d = [&](auto kernel) {
        return unsigned(std::max<int64_t>(1, std::min<int64_t>(tiles, int64_t(resident_per_sm(kernel, 256)) * sms)));
    };
    if (rounding == FP4Q_SR)
        nv_quant_2d_kernel<true><<<grid_2d(nv_quant_2d_kernel<true>), 256, 0, s>>>(
            xb, rows, tpr, ld_x * 2, keys, amax_ptr, amax_out, tensor_scale_out, q, scales, mma);
    else
        nv_quant_2d_kernel<false><<<grid_2d(nv_quant_2d_kernel<false>), 256, 0, s>>>(
            xb, rows, tpr, ld_x * 2, keys, amax_ptr, amax_out, tensor_scale_out, q, scales, mma);
    return check_launch("nv_quantize_2d");
}
