// Scaled MXFP4 -> FP8-E4M3 with one FP32 scale per 1x128 tile.
//
// "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// section 2.B: the E2M1 sign / exponent / mantissa fields are rewritten as
// E4M3 fields with no floating-point arithmetic in between, and the four
// 32-element block scales of a 128-element tile are aligned to their maximum
// (the tile's FP8 scale), each element's exponent being shifted by its
// block's distance to that maximum.  The Spanish summary, section 2, adds
// that subnormal results keep their implicit bit.
//
// Kernel: one thread per 32-element block (16 bytes of codes in, 32 bytes of
// E4M3 out).  The shift d = E_i - Emax is the same for the whole block, so
// the block's 8 possible magnitudes are one 64-bit row of a small table
// indexed by -d (rows for -d >= 12 are all zero); eight output bytes then
// cost two byte-permute lookups plus the sign-bit spread.
#include <algorithm>

#include "common.cuh"
#include "ring.cuh"

namespace fp4q {
namespace {

constexpr int kShiftRows = 13;   // -d = 0..11 explicit, 12 = "12 or more"

// E4M3 magnitude byte of E2M1 magnitude code c (0..7) shifted by 2^-sh.
// E2M1 c = (1 + m/2) * 2^k with (k, m) = (-1, 0) for c = 1 and
// ((c >> 1) - 1, c & 1) for c >= 2.  t = k - sh:  t >= -6 is a normal E4M3
// (exponent field t + 7, mantissa m << 2); t = -7, -8, -9 are the subnormals
// 4 + 2m, 2 + m and 1 + m (the last one rounds 1.5 to 2, ties to even);
// smaller t lies below 2^-9 and flushes to zero.
__host__ __device__ constexpr uint32_t shifted_magnitude(uint32_t c, int sh) {
    if (c == 0) return 0;
    const int k = c == 1 ? -1 : int(c >> 1) - 1;
    const uint32_t m = c == 1 ? 0u : (c & 1u);
    const int t = k - sh;
    if (t >= -6) return (uint32_t(t + 7) << 3) | (m << 2);
    if (t == -7) return 4u + 2u * m;
    if (t == -8) return 2u + m;
    if (t == -9) return 1u + m;
    return 0u;
}

// The same table as a compile-time constant in global memory, for kernels
// whose CTAs are too short-lived to build a shared copy: row sh holds the
// magnitudes of codes 0..3 (lo) and 4..7 (hi).
struct ShiftTable { uint32_t lo[kShiftRows], hi[kShiftRows]; };
constexpr ShiftTable make_shift_table() {
    ShiftTable t{};
    for (int sh = 0; sh < kShiftRows; ++sh)
        for (uint32_t c = 0; c < 4; ++c) {
            t.lo[sh] |= shifted_magnitude(c, sh) << (8 * c);
            t.hi[sh] |= shifted_magnitude(c + 4, sh) << (8 * c);
        }
    return t;
}
__device__ constexpr ShiftTable kShiftTable = make_shift_table();

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Eight packed codes (one 32-bit word, element j in nibble j) -> eight E4M3
// bytes, given the magnitude row (lut.x = codes 0..3, lut.y = codes 4..7).
// The magnitudes are two byte-permute lookups (selector nibbles = the codes'
// low three bits).  The signs use prmt's sign-replicate selectors (selector
// bit 3): nibble 2k + 1's sign bit is the top bit of byte k of w, nibble 2k's
// the top bit of byte k of w << 4, so one permute spreads four signs to
// 0x00 / 0xff bytes.
__device__ __forceinline__ uint2 remap8(uint32_t w, uint2 lut) {
    const uint32_t wm = w & 0x77777777u;
    const uint32_t mag_lo = prmt(lut.x, lut.y, wm), mag_hi = prmt(lut.x, lut.y, wm >> 16);
    const uint32_t w4 = w << 4;
    const uint32_t sgn_lo = prmt(w, w4, 0x9D8Cu), sgn_hi = prmt(w, w4, 0xBFAEu);
    return make_uint2(mag_lo | (sgn_lo & 0x80808080u), mag_hi | (sgn_hi & 0x80808080u));
}

// One 32-element block: `cw` its 16 bytes of codes, `sw` the four E8M0 bytes of
// its 1x128 tile, b its block index (b % 4 = position in the tile).
__device__ __forceinline__ void convert_block(const uint4& cw, uint32_t sw, uint32_t b, const uint2* lut,
                                              uint8_t* __restrict__ yb, float* __restrict__ ts) {
    const uint32_t e_own = (sw >> (8 * (b & 3))) & 0xffu;
    const uint32_t m2 = __vmaxu4(sw, sw >> 16);
    const uint32_t emax = max(m2 & 0xffu, (m2 >> 8) & 0xffu);
    const uint32_t sh = min(emax - e_own, uint32_t(kShiftRows - 1));
    const uint2 L = lut[sh];
    const uint2 o0 = remap8(cw.x, L), o1 = remap8(cw.y, L), o2 = remap8(cw.z, L), o3 = remap8(cw.w, L);
    u32x8 o;
    o.v[0] = o0.x; o.v[1] = o0.y; o.v[2] = o1.x; o.v[3] = o1.y;
    o.v[4] = o2.x; o.v[5] = o2.y; o.v[6] = o3.x; o.v[7] = o3.y;
    stg256(yb, o);
    if ((b & 3) == 0) *ts = exp2i(int(emax) - 127);
}

// A CTA covers rpc rows side by side (blockDim.x / rpc threads per row).
__global__ void __launch_bounds__(512) fp4_to_fp8_kernel(
    const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t rows, uint32_t bpr,
    uint8_t* __restrict__ y, float* __restrict__ tile_scale, int rpc) {
    __shared__ uint2 lut[kShiftRows];
    if (threadIdx.x < kShiftRows) {
        uint32_t lo = 0, hi = 0;
        for (uint32_t c = 0; c < 4; ++c) {
            lo |= shifted_magnitude(c, threadIdx.x) << (8 * c);
            hi |= shifted_magnitude(c + 4, threadIdx.x) << (8 * c);
        }
        lut[threadIdx.x] = make_uint2(lo, hi);
    }
    __syncthreads();
    // two adjacent blocks (2u, 2u + 1) of one 1x128 tile per thread
    const uint32_t upc = blockDim.x / uint32_t(rpc);
    const uint32_t u = blockIdx.x * upc + threadIdx.x % upc;
    if (u >= (bpr >> 1)) return;
    const uint32_t b = 2 * u;
    const int64_t step = int64_t(gridDim.y) * rpc;
    for (int64_t r = int64_t(blockIdx.y) * rpc + threadIdx.x / upc; r < rows; r += 2 * step) {
        // two rows in flight: both rows' codes and tile exponents are loaded first
        const int64_t r2 = r + step;
        const bool two = r2 < rows;
        const uint64_t blk = uint64_t(r) * bpr + b, blk2 = uint64_t(r2) * bpr + b;
        const uint4* c1p = reinterpret_cast<const uint4*>(q + blk * 16);
        const uint4 cw0 = c1p[0], cw1 = c1p[1];
        const uint32_t sw = *reinterpret_cast<const uint32_t*>(s + uint64_t(r) * bpr + (b & ~3u));
        uint4 dw0 = make_uint4(0, 0, 0, 0), dw1 = dw0;
        uint32_t sw2 = 0;
        if (two) {
            const uint4* c2p = reinterpret_cast<const uint4*>(q + blk2 * 16);
            dw0 = c2p[0];
            dw1 = c2p[1];
            sw2 = *reinterpret_cast<const uint32_t*>(s + uint64_t(r2) * bpr + (b & ~3u));
        }
        float* ts = tile_scale + uint64_t(r) * (bpr >> 2) + (b >> 2);
        convert_block(cw0, sw, b, lut, y + blk * 32, ts);
        convert_block(cw1, sw, b + 1, lut, y + blk * 32 + 32, ts);
        if (two) {
            float* ts2 = tile_scale + uint64_t(r2) * (bpr >> 2) + (b >> 2);
            convert_block(dw0, sw2, b, lut, y + blk2 * 32, ts2);
            convert_block(dw1, sw2, b + 1, lut, y + blk2 * 32 + 32, ts2);
        }
    }
}

__device__ __forceinline__ void lut_setup(uint2* lut) {
    for (uint32_t t = threadIdx.x; t < kShiftRows; t += blockDim.x) {
        uint32_t lo = 0, hi = 0;
        for (uint32_t c = 0; c < 4; ++c) {
            lo |= shifted_magnitude(c, int(t)) << (8 * c);
            hi |= shifted_magnitude(c + 4, int(t)) << (8 * c);
        }
        lut[t] = make_uint2(lo, hi);
    }
}

// Shared-memory-staged form (ring.cuh): each group of `rps` rows arrives as one
// bulk copy of its codes and one of its E8M0 bytes.  A consumer thread converts
// a pair of blocks (32 bytes of codes) per step, reading its two 16-byte blocks
// in the order k ^ ((lane >> 2) & 1), which puts any 8 consecutive lanes on 8
// different 16-byte bank groups.
__global__ void __launch_bounds__(ring::kMaxThreads) fp4_to_fp8_staged_kernel(
    const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t rows, uint32_t cols,
    uint8_t* __restrict__ y, float* __restrict__ tile_scale, uint32_t rps, uint32_t* status) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint2 lut[kShiftRows];
    lut_setup(lut);                                      // make_ring's barrier publishes it
    const uint32_t code_bytes = cols / 2, scale_bytes = cols / 32;
    const ring::Ring rg = ring::make_ring(smem, rps * (code_bytes + scale_bytes));
    allow_dependent_launch();
    grid_dependency_wait();             // the codes may come from the previous kernel on the stream
    const int64_t ngroups = (rows + rps - 1) / rps;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bpr = cols / 32, ppr = cols / 64;
    if (warp == 0) {
        if (lane == 0)
            ring::produce(rg, ngroups, status, kStatusStreamTimeout, [&](uint8_t* st, uint32_t fb, int64_t g) {
                const int64_t r0 = g * rps;
                const uint32_t nr = uint32_t(min(int64_t(rps), rows - r0));
                tc::mbar_arrive_expect_tx(fb, nr * (code_bytes + scale_bytes));
                tc::bulk_load(tc::smem_u32(st), q + r0 * int64_t(code_bytes), nr * code_bytes, fb);
                tc::bulk_load(tc::smem_u32(st + rps * code_bytes), s + r0 * int64_t(scale_bytes), nr * scale_bytes,
                              fb);
            });
        return;
    }
    const uint32_t ct = threadIdx.x - 32;
    const uint32_t stride = blockDim.x - 32;
    const uint32_t rr0 = ct / ppr, u0 = ct % ppr, dr = stride / ppr, du = stride % ppr;
    const uint32_t sw = (uint32_t(lane) >> 2) & 1u;
    ring::consume(rg, ngroups, status, kStatusStreamTimeout, [&](uint8_t* st, int64_t g) {
        const int64_t r0 = g * rps;
        const uint32_t nr = uint32_t(min(int64_t(rps), rows - r0));
        const uint32_t units = nr * ppr;
        const uint32_t cbase = tc::smem_u32(st), sbase = cbase + rps * code_bytes;
        uint32_t rr = rr0, u = u0;
        for (uint32_t un = ct; un < units; un += stride) {
            uint4 c[2];
#pragma unroll
            for (uint32_t k = 0; k < 2; ++k)
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(c[k].x), "=r"(c[k].y), "=r"(c[k].z), "=r"(c[k].w)
                             : "r"(cbase + 32 * un + 16 * (k ^ sw)));
            uint32_t swd;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(swd) : "r"(sbase + rr * scale_bytes + 4 * (u >> 1)));
            const int64_t r = r0 + rr;
            float* ts = tile_scale + r * int64_t(bpr / 4) + (u >> 1);
#pragma unroll
            for (uint32_t k = 0; k < 2; ++k) {
                const uint32_t b = 2 * u + (k ^ sw);
                convert_block(c[k], swd, b, lut, y + (r * int64_t(bpr) + b) * 32, ts);
            }
            u += du;
            rr += dr;
            if (u >= ppr) { u -= ppr; ++rr; }
        }
    });
}

// FP4RowToFP8Col ("Practical FP4 Training for Large-Scale MoE Models on Hopper
// GPUs", Spanish summary section 2; French summary 2.C: dequantize, transpose
// and re-quantize in one kernel).  Input: row-wise MXFP4 [rows, cols]; output:
// E4M3 of the transpose [cols, rows] with one FP32 scale per 1x128 tile along
// the output rows ([cols, rows/128]).  A warp converts 128 input rows x 64
// input columns (two 32-blocks): lane l reads rows 4l .. 4l + 3 with one
// 32-byte load each, so the two output tiles' scales (2^Emax over the 128
// rows' block exponents) are warp maxima; each row is remapped with the shift
// table, and a 4 x 4 byte transpose in registers (eight byte permutes per 16
// bytes) turns the lane's 4 rows x 4 columns into four 32-bit words, one per
// output row: every store instruction writes 128 contiguous bytes of one
// output row.  No shared-memory staging of the tile is needed.
constexpr int kColTile = 128;

// One warp of FP4RowToFP8Col: input rows r0 .. r0 + 127 (MASKED: only the first
// nreal are read, the others count as zero codes with E8M0 byte 0, which never
// raise the tile maximum) x input columns c0 .. c0 + 63 -> bytes ycol ..
// ycol + 127 of output rows c0 .. c0 + 63 (row stride ld_y) and their tile
// scales at tile_scale[(c0 + k) * ld_ts + tcol].
template <bool MASKED>
__device__ __forceinline__ void row_to_col_warp(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                                int64_t cols, int64_t r0, int nreal, int64_t c0,
                                                uint8_t* __restrict__ y, int64_t ld_y, int64_t ycol,
                                                float* __restrict__ tile_scale, int64_t ld_ts, int64_t tcol,
                                                int lane) {
    const int64_t rb = r0 + 4 * lane;
    const int64_t spr = cols / 32;
    u32x8 cw[4];
    uint32_t e[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (!MASKED || 4 * lane + i < nreal) {
            cw[i] = ldg256(q + (rb + i) * (cols / 2) + c0 / 2);
            const uint32_t sw = *reinterpret_cast<const uint16_t*>(s + (rb + i) * spr + c0 / 32);
            e[i][0] = sw & 0xffu;
            e[i][1] = sw >> 8;
        } else {
            cw[i] = u32x8{};
            e[i][0] = e[i][1] = 0u;
        }
    }
    uint32_t emax[2];
#pragma unroll
    for (int b = 0; b < 2; ++b)
        emax[b] = __reduce_max_sync(0xffffffffu, max(max(e[0][b], e[1][b]), max(e[2][b], e[3][b])));
    tile_scale[(c0 + lane) * ld_ts + tcol] = exp2i(int(emax[0]) - 127);
    tile_scale[(c0 + 32 + lane) * ld_ts + tcol] = exp2i(int(emax[1]) - 127);
    uint2 L[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const uint32_t sh = min(emax[b] - e[i][b], uint32_t(kShiftRows - 1));
            L[i][b] = make_uint2(__ldg(&kShiftTable.lo[sh]), __ldg(&kShiftTable.hi[sh]));
        }
    uint8_t* yl = y + ycol + 4 * lane;
#pragma unroll
    for (int k = 0; k < 8; ++k) {                       // codes word k: columns 8k .. 8k + 7
        uint2 o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = remap8(cw[i].v[k], L[i][k >> 2]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {                   // columns 8k + 4h .. + 3
            const uint32_t w0 = h ? o[0].y : o[0].x, w1 = h ? o[1].y : o[1].x;
            const uint32_t w2 = h ? o[2].y : o[2].x, w3 = h ? o[3].y : o[3].x;
            const uint32_t t0 = __byte_perm(w0, w1, 0x5140), t1 = __byte_perm(w0, w1, 0x7362);
            const uint32_t t2 = __byte_perm(w2, w3, 0x5140), t3 = __byte_perm(w2, w3, 0x7362);
            const uint32_t col[4] = {__byte_perm(t0, t2, 0x5410), __byte_perm(t0, t2, 0x7632),
                                     __byte_perm(t1, t3, 0x5410), __byte_perm(t1, t3, 0x7632)};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                *reinterpret_cast<uint32_t*>(yl + (c0 + 8 * k + 4 * h + kk) * ld_y) = col[kk];
        }
    }
}

// FP4RowToFP8Col ("Practical FP4 Training for Large-Scale MoE Models on Hopper
// GPUs", Spanish summary section 2; French summary 2.C: dequantize, transpose
// and re-quantize in one kernel).  Input: row-wise MXFP4 [rows, cols]; output:
// E4M3 of the transpose [cols, rows] with one FP32 scale per 1x128 tile along
// the output rows ([cols, rows/128]).  A warp converts 128 input rows x 64
// input columns (two 32-blocks): lane l reads rows 4l .. 4l + 3 with one
// 32-byte load each, so the two output tiles' scales (2^Emax over the 128
// rows' block exponents) are warp maxima; each row is remapped with the shift
// table, and a 4 x 4 byte transpose in registers (eight byte permutes per 16
// bytes) turns the lane's 4 rows x 4 columns into four 32-bit words, one per
// output row: every store instruction writes 128 contiguous bytes of one
// output row.  No shared-memory staging of the tile is needed.
__global__ void __launch_bounds__(64) fp4_row_to_fp8_col_kernel(
    const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t rows, int64_t cols,
    uint8_t* __restrict__ y, float* __restrict__ tile_scale) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = int64_t(blockIdx.y) * kColTile;
    const int64_t c0 = int64_t(blockIdx.x) * kColTile + 64 * warp;     // 64 columns of this warp
    row_to_col_warp<false>(q, s, cols, r0, kColTile, c0, y, rows, r0, tile_scale, rows / kColTile, r0 / kColTile,
                           lane);
}

// The same on ragged expert groups (French summary 2.C: per-expert tensors
// located by precomputed offsets): the tiles restart at each group's first row
// and each group is padded to whole tiles in the output (group g's rows at
// columns 128 T_g .. 128 T_g + n_g - 1 of every output row, zeros up to its
// next tile; T_g = the tiles of the groups before g).  Persistent CTAs of
// eight warps; warp 0 first builds the group tables: the offsets clamped into
// a non-decreasing run inside [0, rows] (the clamp of offset g is its prefix
// maximum, clamped to [0, rows]) and the tile prefix sums, each lane taking
// nine consecutive entries.  Each warp then takes (tile, 64-column) items.
constexpr int kGroupedMax = 256;

__global__ void __launch_bounds__(256) fp4_row_to_fp8_col_grouped_kernel(
    const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t rows, int64_t cols,
    const int64_t* __restrict__ offsets, int groups, uint8_t* __restrict__ y, int64_t ld_y,
    float* __restrict__ tile_scale) {
    __shared__ int64_t off[kGroupedMax + 1];
    __shared__ int64_t tpre[kGroupedMax + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        constexpr int kPer = (kGroupedMax + 1 + 31) / 32;        // 9 entries per lane
        const int g0 = kPer * lane;
        int64_t v[kPer];
        int64_t run = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            v[j] = g0 + j <= groups ? offsets[g0 + j] : 0;
            run = max(run, v[j]);
            v[j] = run;                                          // running maximum within the lane
        }
        int64_t before = 0;                                      // maximum over the lanes below
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t up = __shfl_up_sync(0xffffffffu, run, o);
            if (lane >= o) run = max(run, up);
        }
        before = __shfl_up_sync(0xffffffffu, run, 1);
        if (lane == 0) before = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j)
            if (g0 + j <= groups) off[g0 + j] = min(max(v[j], before), rows);
        __syncwarp();
        int64_t t[kPer], sum = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            t[j] = g0 + j < groups ? (off[g0 + j + 1] - off[g0 + j] + 127) / 128 : 0;
            sum += t[j];
        }
        int64_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t up = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += up;
        }
        int64_t acc = incl - sum;                                // tiles of the lanes below
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (g0 + j <= groups) tpre[g0 + j] = acc;
            acc += t[j];
        }
    }
    __syncthreads();
    const int64_t ncc = cols / 64, ntiles = tpre[groups], items = ntiles * ncc;
    const int64_t wstep = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t it = int64_t(blockIdx.x) * (blockDim.x >> 5) + warp; it < items; it += wstep) {
        const int64_t tile = it / ncc, c0 = (it - tile * ncc) * 64;
        int lo = 0, hi = groups - 1;                             // the group of the tile
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tpre[mid] <= tile) lo = mid; else hi = mid - 1;
        }
        const int64_t r0 = off[lo] + (tile - tpre[lo]) * kColTile;
        const int nreal = int(min(int64_t(kColTile), off[lo + 1] - r0));
        row_to_col_warp<true>(q, s, cols, r0, nreal, c0, y, ld_y, tile * kColTile, tile_scale, ld_y / kColTile,
                              tile, lane);
    }
}

// FP32 power-of-two tile scales (one per 1x128 tile, as fp4_to_fp8 and
// fp4_row_to_fp8_col write them) -> E8M0 block scales, one per 32 elements
// (the tile's exponent repeated over its four blocks), for the MXFP8 GEMM.
// Exact: 2^e is E8M0 byte e + 127.  Anything that is not a power of two in
// [2^-127, 2^127] gives 0xFF (NaN) and sets a status bit.
__global__ void __launch_bounds__(256) fp8_tile_scales_to_e8m0_kernel(
    const float* __restrict__ tile_scale, int64_t rows, uint32_t tiles_per_row, uint8_t* __restrict__ s,
    int mma_layout, uint32_t* status) {
    const int64_t n = rows * int64_t(tiles_per_row);
    const uint32_t bpr = tiles_per_row * 4;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
        const uint32_t u = f2u(tile_scale[i]);
        const uint32_t ef = u >> 23;
        uint32_t b;
        if (u == 0x00400000u) b = 0u;                                  // 2^-127 (FP32 subnormal)
        else if ((u & 0x007fffffu) == 0 && ef >= 1u && ef <= 254u) b = ef;
        else { b = 0xffu; atomicOr(status, kStatusBadTileScale); }
        const int64_t r = i / tiles_per_row;
        const uint32_t t = uint32_t(i - r * tiles_per_row);
#pragma unroll
        for (uint32_t k = 0; k < 4; ++k) {
            const uint32_t c = 4 * t + k;
            s[mma_layout ? mma_scale_offset(uint64_t(r), c, bpr) : uint64_t(r) * bpr + c] = uint8_t(b);
        }
    }
}

}  // namespace
}  // namespace fp4q

using namespace fp4q;

extern "C" fp4q_status fp4q_fp8_tile_scales_to_e8m0(const float* tile_scale, int64_t rows, int64_t cols,
                                                   uint8_t* scales, fp4q_scale_layout layout, fp4q_stream_t stream) {
    if (rows < 0 || cols < 0) return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp8_tile_scales_to_e8m0: negative size");
    if (cols % 128) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "fp8_tile_scales_to_e8m0: cols %% 128 != 0");
    if (layout != FP4Q_SCALES_ROWMAJOR && layout != FP4Q_SCALES_MMA)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp8_tile_scales_to_e8m0: bad scale layout");
    if (rows == 0 || cols == 0) return FP4Q_OK;
    if (!tile_scale || !scales) return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp8_tile_scales_to_e8m0: null pointer");
    if (reinterpret_cast<uintptr_t>(tile_scale) & 3u)
        return fail(FP4Q_ERR_MISALIGNED, "fp8_tile_scales_to_e8m0: tile_scale 4-byte aligned");
    int sms = 0;
    fp4q_status st = current_device(&sms);
    if (st != FP4Q_OK) return st;
    const int64_t n = rows * (cols / 128);
    const int64_t grid = std::min<int64_t>((n + 255) / 256, int64_t(sms) * 8);
    fp8_tile_scales_to_e8m0_kernel<<<unsigned(grid), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        tile_scale, rows, uint32_t(cols / 128), scales, layout == FP4Q_SCALES_MMA, status_word());
    return check_launch("fp8_tile_scales_to_e8m0");
}

extern "C" fp4q_status fp4q_fp4_row_to_fp8_col(const uint8_t* q, const uint8_t* scales, int64_t rows,
                                               int64_t cols, uint8_t* y, float* tile_scale,
                                               fp4q_stream_t stream) {
    if (rows < 0 || cols < 0) return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp4_row_to_fp8_col: negative size");
    if (rows % kColTile || cols % kColTile)
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "fp4_row_to_fp8_col: rows %% 128 == 0 and cols %% 128 == 0");
    if (rows / kColTile > 65535) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "fp4_row_to_fp8_col: rows <= 8388480");
    if (rows == 0 || cols == 0) return FP4Q_OK;
    if (!q || !scales || !y || !tile_scale) return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp4_row_to_fp8_col: null pointer");
    if ((reinterpret_cast<uintptr_t>(q) & 31u) || (reinterpret_cast<uintptr_t>(y) & 31u) ||
        (reinterpret_cast<uintptr_t>(scales) & 3u) || (reinterpret_cast<uintptr_t>(tile_scale) & 3u))
        return fail(FP4Q_ERR_MISALIGNED, "fp4_row_to_fp8_col: q, y 32-byte aligned; scales, tile_scale 4-byte aligned");
    fp4q_status st = current_device(nullptr);
    if (st != FP4Q_OK) return st;
    const dim3 grid(unsigned(cols / kColTile), unsigned(rows / kColTile), 1);
    fp4_row_to_fp8_col_kernel<<<grid, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(q, scales, rows, cols, y,
                                                                                      tile_scale);
    return check_launch("fp4_row_to_fp8_col");
}

extern "C" int64_t fp4q_fp4_row_to_fp8_col_grouped_ld(int64_t rows, int64_t groups) {
    if (rows < 0 || groups < 1 || groups > kGroupedMax || rows > INT32_MAX) return 0;
    return kColTile * ((rows + kColTile - 1) / kColTile + groups);
}

extern "C" fp4q_status fp4q_fp4_row_to_fp8_col_grouped(const uint8_t* q, const uint8_t* scales, int64_t rows,
                                                       int64_t cols, const int64_t* offsets, int64_t groups,
                                                       uint8_t* y, float* tile_scale, fp4q_stream_t stream) {
    if (rows < 0 || cols < 0 || groups < 1 || groups > kGroupedMax)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp4_row_to_fp8_col_grouped: need rows, cols >= 0, 1 <= groups <= %d",
                    kGroupedMax);
    if (cols % kColTile) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "fp4_row_to_fp8_col_grouped: cols %% 128 != 0");
    if (rows > INT32_MAX || cols > INT32_MAX)
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "fp4_row_to_fp8_col_grouped: rows and cols at most 2^31 - 1");
    if (rows == 0 || cols == 0) return FP4Q_OK;
    if (!q || !scales || !offsets || !y || !tile_scale)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp4_row_to_fp8_col_grouped: null pointer");
    if ((reinterpret_cast<uintptr_t>(q) & 31u) || (reinterpret_cast<uintptr_t>(y) & 31u) ||
        (reinterpret_cast<uintptr_t>(scales) & 3u) || (reinterpret_cast<uintptr_t>(tile_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(offsets) & 7u))
        return fail(FP4Q_ERR_MISALIGNED,
                    "fp4_row_to_fp8_col_grouped: q, y 32-byte aligned; scales, tile_scale 4-byte; offsets 8-byte");
    int sms = 0;
    fp4q_status st = current_device(&sms);
    if (st != FP4Q_OK) return st;
    const int64_t ld = fp4q_fp4_row_to_fp8_col_grouped_ld(rows, groups);
    const int64_t items_upper = (ld / kColTile) * (cols / 64);
    const int64_t blocks = std::min<int64_t>((items_upper + 7) / 8,
                                             int64_t(sms) * resident_per_sm(fp4_row_to_fp8_col_grouped_kernel, 256));
    fp4_row_to_fp8_col_grouped_kernel<<<unsigned(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        q, scales, rows, cols, offsets, int(groups), y, ld, tile_scale);
    return check_launch("fp4_row_to_fp8_col_grouped");
}

extern "C" fp4q_status fp4q_fp4_to_fp8(const uint8_t* q, const uint8_t* scales, int64_t rows,
                                       int64_t cols, int block_axis, uint8_t* y, float* tile_scale,
                                       fp4q_stream_t stream) {
    if (rows < 0 || cols < 0) return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp4_to_fp8: negative size");
    if (block_axis != 1) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "fp4_to_fp8: only block_axis = 1");
    if (cols % 128) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "fp4_to_fp8: cols %% 128 != 0");
    if (rows == 0 || cols == 0) return FP4Q_OK;
    if (!q || !scales || !y || !tile_scale) return fail(FP4Q_ERR_INVALID_ARGUMENT, "fp4_to_fp8: null pointer");
    if (!aligned16(q) || (reinterpret_cast<uintptr_t>(y) & 31u) ||
        (reinterpret_cast<uintptr_t>(scales) & 3u) || (reinterpret_cast<uintptr_t>(tile_scale) & 3u))
        return fail(FP4Q_ERR_MISALIGNED, "fp4_to_fp8: q 16-byte, y 32-byte, scales/tile_scale 4-byte aligned");
    int sms = 0;
    fp4q_status st = current_device(&sms);
    if (st != FP4Q_OK) return st;
    const uint32_t bpr = uint32_t(cols / 32);
    const uint32_t row_bytes = uint32_t(cols / 2 + cols / 32);
    const ring::Shape sh = cols % 512 == 0 && aligned16(scales) && cols <= (1 << 20)
                               ? ring::ring_shape(uint32_t(cols / 64), row_bytes) : ring::Shape{0, 0};
    if (sh.rps) {
        const uint32_t smem = ring::smem_bytes(sh.rps * row_bytes);
        const int threads = 32 * int(1 + sh.warps);
        const int per_sm = resident_per_sm_smem(fp4_to_fp8_staged_kernel, threads, smem);
        const int64_t ngroups = (rows + sh.rps - 1) / sh.rps;
        const int64_t grid = std::min<int64_t>(ngroups, int64_t(per_sm) * sms);
        const cudaError_t e = launch_overlapped(fp4_to_fp8_staged_kernel, dim3(unsigned(grid)), dim3(threads), smem,
                                                reinterpret_cast<cudaStream_t>(stream), q, scales, rows,
                                                uint32_t(cols), y, tile_scale, sh.rps, status_word());
        if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "fp4_to_fp8: %s", cudaGetErrorString(e));
        return FP4Q_OK;
    }
    int tpb, nx, rpc;
    packed_row_shape(bpr / 2, &tpb, &nx, &rpc);
    dim3 grid(unsigned(nx), row_grid_y((rows + rpc - 1) / rpc, nx, sms, resident_per_sm(fp4_to_fp8_kernel, tpb)), 1);
    fp4_to_fp8_kernel<<<grid, tpb, 0, reinterpret_cast<cudaStream_t>(stream)>>>(q, scales, rows, bpr, y, tile_scale,
                                                                                rpc);
    return check_launch("fp4_to_fp8");
}
