// MoE dispatch of packed MXFP4 rows and the MXFP4 -> UE4M3 scale rebase
// that lets MXFP4 activations meet NVFP4 expert weights in one tcgen05
// block-scaled MMA kind.
//
// "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// section 2.A: activations are quantized to MXFP4 before the expert
// dispatch, so what moves is packed FP4 plus scales; section 2.C: ragged
// per-expert tensors with precomputed offsets and no padding.
//
// Dispatch (stable: inside an expert, ascending token id):
//   1. count:  one CTA per 256 tokens; per expert, a ballot over each warp
//              gives every (token, slot) its rank among the chunk's tokens
//              that chose the same expert, and the chunk's expert counts.
//   2. scan:   one CTA; chunk bases per expert, expert offsets [E + 1].
//   3. gather: one warp per dispatched row copies the packed codes
//              (16-byte vectors) and the E8M0 bytes of its token.
// Rebase: per row, B = max_j E_j - 8 and each 32-block's 2^E_j becomes the
// UE4M3 value 2^(E_j - B) for both of its 16-element halves (exact for
// E_j - B >= -9), written in the MMA scale layout with every group padded to
// whole 128-row tiles; the row factor 2^B goes to the GEMM epilogue.
#include <atomic>

#include "common.cuh"

namespace fp4q {
namespace {

constexpr int kChunk = 256;      // tokens per count CTA (8 warps)
constexpr int kMaxExperts = 256;

struct DispatchWs {
    int32_t* chunk_count;        // [chunks][E]
    int32_t* chunk_base;         // [chunks][E]
    int32_t* local_rank;         // [T * k]
};

__global__ void __launch_bounds__(kChunk) moe_count_kernel(const int32_t* __restrict__ topk, int64_t tokens, int k,
                                                           int E, int32_t* __restrict__ chunk_count,
                                                           int32_t* __restrict__ local_rank) {
    __shared__ int32_t warp_cnt[kChunk / 32][kMaxExperts];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = int64_t(blockIdx.x) * kChunk + threadIdx.x;
    const bool valid = t < tokens;
    int32_t mine[16];
    int32_t rank_in_warp[16];
    for (int j = 0; j < k; ++j) {
        mine[j] = valid ? topk[t * k + j] : -1;
        rank_in_warp[j] = 0;
    }
    const uint32_t lt = (1u << lane) - 1u;
    for (int e = 0; e < E; ++e) {
        bool has = false;
        for (int j = 0; j < k; ++j) has |= (mine[j] == e);
        const uint32_t m = __ballot_sync(0xffffffffu, has);
        if (lane == 0) warp_cnt[warp][e] = __popc(m);
        if (has)
            for (int j = 0; j < k; ++j)
                if (mine[j] == e) rank_in_warp[j] = __popc(m & lt);
    }
    __syncthreads();
    if (valid) {
        for (int j = 0; j < k; ++j) {
            const int e = mine[j];
            int r = -1;
            if (e >= 0 && e < E) {
                r = rank_in_warp[j];
                for (int w = 0; w < warp; ++w) r += warp_cnt[w][e];
            }
            local_rank[t * k + j] = r;
        }
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t c = 0;
        for (int w = 0; w < kChunk / 32; ++w) c += warp_cnt[w][e];
        chunk_count[int64_t(blockIdx.x) * E + e] = c;
    }
}

__global__ void moe_scan_kernel(const int32_t* __restrict__ chunk_count, int64_t chunks, int E,
                                int32_t* __restrict__ chunk_base, int64_t* __restrict__ offsets) {
    __shared__ int64_t total[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int64_t acc = 0;
        for (int64_t c = 0; c < chunks; ++c) {
            chunk_base[c * E + e] = int32_t(acc);
            acc += chunk_count[c * E + e];
        }
        total[e] = acc;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t acc = 0;
        for (int e = 0; e < E; ++e) {
            offsets[e] = acc;
            acc += total[e];
        }
        offsets[E] = acc;
    }
}

__global__ void __launch_bounds__(256) moe_gather_kernel(
    const int32_t* __restrict__ topk, int64_t tokens, int k, int E, const int32_t* __restrict__ chunk_base,
    const int32_t* __restrict__ local_rank, const int64_t* __restrict__ offsets, const uint8_t* __restrict__ q,
    const uint8_t* __restrict__ s, int64_t qbytes, int64_t sbytes, int32_t* __restrict__ row_token,
    uint8_t* __restrict__ q_out, uint8_t* __restrict__ s_out) {
    const int lane = threadIdx.x & 31;
    const int64_t pair = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;   // (token, slot)
    if (pair >= tokens * k) return;
    const int64_t t = pair / k;
    const int e = topk[pair];
    const int32_t r = local_rank[pair];
    if (e < 0 || e >= E || r < 0) return;
    const int64_t pos = offsets[e] + chunk_base[(t / kChunk) * E + e] + r;
    if (lane == 0) row_token[pos] = int32_t(t);
    const uint4* src = reinterpret_cast<const uint4*>(q + t * qbytes);
    uint4* dst = reinterpret_cast<uint4*>(q_out + pos * qbytes);
    for (int64_t i = lane; i < qbytes / 16; i += 32) dst[i] = src[i];
    for (int64_t i = lane; i < sbytes; i += 32) s_out[pos * sbytes + i] = s[t * sbytes + i];
}

// 2^k as FP32 for k in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float exp2_wide(int k) {
    if (k >= -126) return u2f(uint32_t(k + 127) << 23);
    return u2f(1u << (k + 149));
}

// UE4M3 byte of 2^k: normal for k >= -6 (exponent field k + 7), subnormal
// 1, 2, 4 for k = -9, -8, -7; 0 when k < -9 (not representable).
__device__ __forceinline__ uint32_t ue4m3_pow2(int k) {
    if (k >= -6) return uint32_t(k + 7) << 3;
    if (k >= -9) return 1u << (k + 9);
    return 0u;
}

// Group table of the rebase kernels (thread 0): the offsets clamped to a
// non-decreasing run inside [0, rows] -- well-formed offsets pass unchanged,
// and malformed ones can then neither read past the scales nor place more
// padded tiles than fp4q_rebased_scales_bytes covers -- and tpre[g], the
// padded 128-row tiles of the groups before g.
__device__ void rebase_group_table(const int64_t* __restrict__ offsets, int groups, int64_t rows, int64_t* off,
                                   int64_t* tpre) {
    int64_t acc = 0, prev = 0;
    for (int g = 0; g <= groups; ++g) {
        const int64_t o = min(max(offsets[g], prev), rows);
        if (g > 0) acc += (o - prev + 127) / 128;        // tiles of group g - 1
        off[g] = o;
        tpre[g] = acc;
        prev = o;
    }
}

__global__ void __launch_bounds__(256) mx_rebase_kernel(const uint8_t* __restrict__ s, int64_t rows, int S32,
                                                        const int64_t* __restrict__ offsets, int groups,
                                                        uint8_t* __restrict__ out, float* __restrict__ row_scale,
                                                        uint32_t* __restrict__ violations) {
    __shared__ int64_t off[kMaxExperts + 1];
    __shared__ int64_t tpre[kMaxExperts + 1];
    if (threadIdx.x == 0) rebase_group_table(offsets, groups, rows, off, tpre);
    __syncthreads();
    // persistent: the group table above is built once per CTA, then each warp
    // takes rows warp_id, warp_id + warps, ...
    const int lane = threadIdx.x & 31;
    const int64_t nrows = off[groups];
    const int64_t warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const uint32_t S16 = uint32_t(S32) * 2;
    uint32_t bad = 0;
    for (int64_t r = off[0] + ((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5); r < nrows; r += warps) {
        int lo = 0, hi = groups - 1;                 // group of row r: off[g] <= r < off[g + 1]
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (off[mid] <= r) lo = mid; else hi = mid - 1;
        }
        const int64_t prow = tpre[lo] * 128 + (r - off[lo]);   // row in the padded scale layout
        uint32_t m = 0;
        for (int j = lane; j < S32; j += 32) m = max(m, uint32_t(s[r * S32 + j]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int base = int(m) - 127 - 8;
        for (int j = lane; j < S32; j += 32) {
            const int kexp = int(s[r * S32 + j]) - 127 - base;
            const uint32_t b = ue4m3_pow2(kexp);
            bad += (kexp < -9);
            *reinterpret_cast<uint16_t*>(out + mma_scale_offset(uint64_t(prow), uint32_t(2 * j), S16)) =
                uint16_t(b | (b << 8));
        }
        if (lane == 0) row_scale[r] = exp2_wide(base);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad && violations) atomicAdd(violations, bad);
}

// UE4M3 byte of a block whose E8M0 byte lies d = (row maximum byte) - byte
// below its row's maximum: the exponent difference E - B is 8 - d, so the
// byte is (15 - d) << 3 for d <= 14 (normal), 4, 2, 1 for d = 15, 16, 17
// (the subnormals 2^-7 .. 2^-9) and 0 for d >= 18 (not representable,
// counted in `bad`).  Branch-free, so lanes with different d never diverge.
__device__ __forceinline__ uint32_t rebased_byte(uint32_t d, uint32_t& bad) {
    bad += uint32_t(d >= 18u);
    return d <= 14u ? (15u - d) << 3 : 4u >> min(d - 15u, 3u);
}

// The same rebase, one padded 128-row tile at a time.  In the MMA scale layout
// a 128-row tile's scales are one contiguous run of S16/4 chunks of 512 bytes,
// and its E8M0 source rows are one contiguous run of 128 * S32 bytes (fewer at
// a group's end).  Phase 1 stages that run in shared memory, each thread
// loading up to eight 32-bit words before it stores any, so a tile takes few
// load round trips (rows padded by 4 bytes: the column reads of phase 2 then
// fall in 32 different banks; rows past the group are zero); then two threads
// per row take the row's maximum E8M0 byte.
// Phase 2 writes every chunk as 16-byte stores -- thread (c4, i) the bytes of
// rows i, i + 32, i + 64, i + 96 for columns 4 c4 .. 4 c4 + 3 -- so a warp
// writes 512 contiguous bytes (rebased_byte per scale byte).  Padding rows
// are written as 0.
// wdiv = ceil(2^32 / (S32 / 4)): k / (S32 / 4) == (k * wdiv) >> 32 for every
// word index k < 128 * S32 / 4 of a tile.
__global__ void __launch_bounds__(256) mx_rebase_tiles_kernel(const uint8_t* __restrict__ s, int64_t rows, int S32,
                                                              uint64_t wdiv, const int64_t* __restrict__ offsets,
                                                              int groups, uint8_t* __restrict__ out,
                                                              float* __restrict__ row_scale,
                                                              uint32_t* __restrict__ violations) {
    extern __shared__ __align__(16) uint8_t stage[];     // [128][S32 + 4] E8M0 bytes, then uint16 mm[128]
    __shared__ int64_t off[kMaxExperts + 1];
    __shared__ int64_t tpre[kMaxExperts + 1];
    if (threadIdx.x == 0) rebase_group_table(offsets, groups, rows, off, tpre);
    __syncthreads();
    const int RS = S32 + 4;                               // staged row stride (bytes)
    const uint32_t wpr = uint32_t(S32) / 4;               // 32-bit words per row
    uint16_t* mm = reinterpret_cast<uint16_t*>(stage + 128 * RS);     // row max byte, twice
    const int lane = threadIdx.x & 31;
    const int64_t ntiles = tpre[groups];
    uint32_t bad = 0;
    for (int64_t T = blockIdx.x; T < ntiles; T += gridDim.x) {
        int lo = 0, hi = groups - 1;                      // group of padded tile T
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tpre[mid] <= T) lo = mid; else hi = mid - 1;
        }
        const int64_t r0 = off[lo] + (T - tpre[lo]) * 128;
        const int64_t left = off[lo + 1] - r0;
        const int nreal = left < 128 ? int(left) : 128;
        // phase 1: word k of the tile's run -> row k / wpr, word k % wpr
        const uint32_t* src = reinterpret_cast<const uint32_t*>(s + r0 * S32);
        const uint32_t nw = uint32_t(nreal) * wpr, total = 128u * wpr;
        for (uint32_t k0 = threadIdx.x; k0 < total; k0 += 8 * blockDim.x) {
            uint32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t k = k0 + u * blockDim.x;
                v[u] = k < nw ? __ldg(src + k) : 0u;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t k = k0 + u * blockDim.x;
                if (k < total) {
                    const uint32_t rr = uint32_t((uint64_t(k) * wdiv) >> 32);
                    *reinterpret_cast<uint32_t*>(stage + rr * RS + 4 * (k - rr * wpr)) = v[u];
                }
            }
        }
        __syncthreads();
        // row bases: threads 2 rr and 2 rr + 1 take the even and odd words of row rr
        for (uint32_t t = threadIdx.x; t < 256u; t += blockDim.x) {
            const uint32_t rr = t >> 1;
            uint32_t m = 0;
            for (uint32_t j = t & 1u; j < wpr; j += 2) {
                const uint32_t v = *reinterpret_cast<const uint32_t*>(stage + rr * RS + 4 * j);
                const uint32_t h = __vmaxu4(v, v >> 16);            // bytes 0 / 1: max of (0, 2) / (1, 3)
                m = max(m, max(h & 0xffu, (h >> 8) & 0xffu));
            }
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
            if ((t & 1u) == 0) {
                mm[rr] = uint16_t(m * 0x0101u);
                if (int(rr) < nreal) row_scale[r0 + rr] = exp2_wide(int(m) - 127 - 8);
            }
        }
        __syncthreads();
        // phase 2: 16-byte chunks of the tile's contiguous scale run
        uint8_t* tile_out = out + uint64_t(T) * uint64_t(S32 / 2) * 512u;
        for (int k = threadIdx.x; k < (S32 / 2) * 32; k += blockDim.x) {
            const int c4 = k >> 5, i = k & 31;
            uint32_t w[4];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const int rr = i + 32 * qq;
                const uint32_t e2 = *reinterpret_cast<const uint16_t*>(stage + rr * RS + 2 * c4);
                const uint32_t m = mm[rr] & 0xffu;
                const uint32_t b0 = rebased_byte(m - (e2 & 0xffu), bad), b1 = rebased_byte(m - (e2 >> 8), bad);
                w[qq] = rr < nreal ? b0 | (b0 << 8) | (b1 << 16) | (b1 << 24) : 0u;
            }
            *reinterpret_cast<uint4*>(tile_out + c4 * 512 + i * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();                                  // the staging is reused by the next tile
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad && violations) atomicAdd(violations, bad);
}

}  // namespace
}  // namespace fp4q

using namespace fp4q;

// The dispatched rows (tokens x top_k) and the token ids are indexed in int32.
static bool dispatch_too_large(int64_t tokens, int top_k) { return top_k > 0 && tokens > INT32_MAX / top_k; }

extern "C" size_t fp4q_moe_dispatch_workspace_bytes(int64_t tokens, int top_k, int n_experts) {
    if (tokens < 0 || top_k < 1 || top_k > 16 || n_experts < 1 || n_experts > kMaxExperts) return 0;
    if (dispatch_too_large(tokens, top_k)) return 0;
    const int64_t chunks = (tokens + kChunk - 1) / kChunk;
    return size_t(2 * chunks * n_experts + tokens * top_k) * 4u + 256u;
}

extern "C" fp4q_status fp4q_moe_dispatch(const int32_t* topk, int64_t tokens, int top_k, int n_experts,
                                         const uint8_t* q, const uint8_t* scales, int64_t cols, int64_t* offsets,
                                         int32_t* row_token, uint8_t* q_out, uint8_t* scales_out, void* workspace,
                                         size_t workspace_bytes, fp4q_stream_t stream) {
    if (tokens < 0 || top_k < 1 || top_k > 16 || n_experts < 1 || n_experts > kMaxExperts || cols < 0)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "moe_dispatch: need 1 <= top_k <= 16, 1 <= n_experts <= %d",
                    kMaxExperts);
    if (dispatch_too_large(tokens, top_k))
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "moe_dispatch: tokens x top_k above 2^31 - 1");
    if (cols % 32) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "moe_dispatch: cols %% 32 != 0");
    if (!offsets) return fail(FP4Q_ERR_INVALID_ARGUMENT, "moe_dispatch: offsets is NULL");
    if (tokens > 0 && (!topk || !q || !scales || !row_token || !q_out || !scales_out))
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "moe_dispatch: null pointer");
    if (!workspace || workspace_bytes < fp4q_moe_dispatch_workspace_bytes(tokens, top_k, n_experts))
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "moe_dispatch: workspace missing or too small");
    if (!aligned16(q) || !aligned16(q_out) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(offsets) & 7u) ||
        (reinterpret_cast<uintptr_t>(topk) & 3u) || (reinterpret_cast<uintptr_t>(row_token) & 3u))
        return fail(FP4Q_ERR_MISALIGNED, "moe_dispatch: q, q_out, workspace 16-byte aligned; offsets 8-byte");
    fp4q_status st = current_device(nullptr);
    if (st != FP4Q_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t chunks = (tokens + kChunk - 1) / kChunk;
    int32_t* ws = static_cast<int32_t*>(workspace);
    int32_t* chunk_count = ws;
    int32_t* chunk_base = ws + chunks * n_experts;
    int32_t* local_rank = ws + 2 * chunks * n_experts;
    if (chunks > 0) {
        moe_count_kernel<<<unsigned(chunks), kChunk, 0, s>>>(topk, tokens, top_k, n_experts, chunk_count, local_rank);
        if ((st = check_launch("moe_dispatch count")) != FP4Q_OK) return st;
    }
    moe_scan_kernel<<<1, 256, 0, s>>>(chunk_count, chunks, n_experts, chunk_base, offsets);
    if ((st = check_launch("moe_dispatch scan")) != FP4Q_OK) return st;
    const int64_t pairs = tokens * top_k;
    if (pairs > 0 && cols > 0) {
        const int64_t blocks = (pairs * 32 + 255) / 256;
        moe_gather_kernel<<<unsigned(blocks), 256, 0, s>>>(topk, tokens, top_k, n_experts, chunk_base, local_rank,
                                                           offsets, q, scales, cols / 2, cols / 32, row_token, q_out,
                                                           scales_out);
        if ((st = check_launch("moe_dispatch gather")) != FP4Q_OK) return st;
    }
    return FP4Q_OK;
}

// 0 when the size does not fit a size_t (sizes no allocation could hold)
extern "C" size_t fp4q_rebased_scales_bytes(int64_t rows, int64_t cols, int64_t groups) {
    const int64_t big = int64_t(1) << 60;
    if (rows < 0 || cols < 0 || groups < 0 || rows > big || cols > big || groups > big) return 0;
    size_t n = 0;
    if (__builtin_mul_overflow(size_t((rows + 127) / 128 + groups), size_t((cols / 16 + 3) / 4), &n) ||
        __builtin_mul_overflow(n, size_t(512), &n))
        return 0;
    return n;
}

extern "C" fp4q_status fp4q_mx_rebase_scales(const uint8_t* scales, int64_t rows, int64_t cols,
                                             const int64_t* offsets, int64_t groups, uint8_t* ue4m3_mma,
                                             float* row_scale, uint32_t* violations, fp4q_stream_t stream) {
    if (rows < 0 || cols < 0 || groups < 1 || groups > kMaxExperts)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "mx_rebase_scales: need rows >= 0, 1 <= groups <= %d", kMaxExperts);
    if (cols % 128) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "mx_rebase_scales: cols %% 128 != 0");
    if (rows == 0 || cols == 0) return FP4Q_OK;
    if (!scales || !offsets || !ue4m3_mma || !row_scale)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "mx_rebase_scales: null pointer");
    if ((reinterpret_cast<uintptr_t>(offsets) & 7u) || (reinterpret_cast<uintptr_t>(ue4m3_mma) & 15u) ||
        (reinterpret_cast<uintptr_t>(scales) & 3u) || (reinterpret_cast<uintptr_t>(row_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(violations) & 3u))
        return fail(FP4Q_ERR_MISALIGNED, "mx_rebase_scales: offsets 8-byte, output 16-byte, scales 4-byte aligned");
    int sms = 0;
    fp4q_status st = current_device(&sms);
    if (st != FP4Q_OK) return st;
    const int S32 = int(cols / 32);
    if (S32 <= 1024) {
        // tile-wise form: the padded tiles number at most rows / 128 + groups
        const uint32_t smem = uint32_t(128 * (S32 + 4) + 128 * 4);
        const int64_t tiles_upper = (rows + 127) / 128 + groups;
        const int64_t blocks = std::min<int64_t>(tiles_upper, int64_t(sms) *
                                                 resident_per_sm_smem(mx_rebase_tiles_kernel, 256, smem));
        const uint64_t wpr = uint64_t(S32 / 4);
        mx_rebase_tiles_kernel<<<unsigned(blocks), 256, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
            scales, rows, S32, ((uint64_t(1) << 32) + wpr - 1) / wpr, offsets, int(groups), ue4m3_mma, row_scale,
            violations);
        return check_launch("mx_rebase_scales");
    }
    const int64_t blocks = std::min<int64_t>((rows * 32 + 255) / 256,
                                             int64_t(sms) * resident_per_sm(mx_rebase_kernel, 256));
    mx_rebase_kernel<<<unsigned(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        scales, rows, int(cols / 32), offsets, int(groups), ue4m3_mma, row_scale, violations);
    return check_launch("mx_rebase_scales");
}

// ---------------------------------------------------------------------------
// Dispatch without a caller workspace.
//
// Some callers cannot hand the library a device workspace: processes that fix
// their whole device-memory budget at start-up and treat any later
// allocation as an error, plain C callers that only receive device pointers
// from the framework that owns the memory, and latency-sensitive loops where
// a cudaMalloc (which can synchronize the device) is not acceptable.  For
// them the dispatch scratch lives in this file-scope device array instead.
// Every GPU that loads the library holds it until the process exits; every
// call shares it, so calls that overlap on the GPU race on it.  Nothing in it
// needs to start at zero: the count, scan and gather kernels write every
// entry they later read.
// ---------------------------------------------------------------------------
namespace fp4q {
namespace {

static __device__ __align__(256) uint8_t g_dispatch_scratch[FP4Q_MOE_DISPATCH_STATIC_SCRATCH_BYTES];

std::atomic<void*> g_dispatch_scratch_addr[64] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the host-side name of the array is not a device address).
fp4q_status dispatch_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(FP4Q_ERR_UNSUPPORTED_DEVICE, "device index %d", dev);
    void* p = g_dispatch_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
        if (e != cudaSuccess || !p)
            return fail(FP4Q_ERR_CUDA, "cudaGetSymbolAddress(dispatch scratch): %s", cudaGetErrorString(e));
        g_dispatch_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return FP4Q_OK;
}

}  // namespace
}  // namespace fp4q

extern "C" fp4q_status fp4q_moe_dispatch_static(const int32_t* topk, int64_t tokens, int top_k, int n_experts,
                                                const uint8_t* q, const uint8_t* scales, int64_t cols,
                                                int64_t* offsets, int32_t* row_token, uint8_t* q_out,
                                                uint8_t* scales_out, fp4q_stream_t stream) {
    if (tokens < 0 || top_k < 1 || top_k > 16 || n_experts < 1 || n_experts > kMaxExperts || cols < 0)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "moe_dispatch_static: need 1 <= top_k <= 16, 1 <= n_experts <= %d",
                    kMaxExperts);
    if (dispatch_too_large(tokens, top_k))
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "moe_dispatch_static: tokens x top_k above 2^31 - 1");
    const size_t need = fp4q_moe_dispatch_workspace_bytes(tokens, top_k, n_experts);
    if (need > size_t(FP4Q_MOE_DISPATCH_STATIC_SCRATCH_BYTES))
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE,
                    "moe_dispatch_static: %lld tokens x top-%d over %d experts need %zu scratch bytes, more than the "
                    "%u-byte static array; use fp4q_moe_dispatch with a workspace",
                    (long long)tokens, top_k, n_experts, need, unsigned(FP4Q_MOE_DISPATCH_STATIC_SCRATCH_BYTES));
    if (cols % 32) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "moe_dispatch_static: cols %% 32 != 0");
    if (!offsets) return fail(FP4Q_ERR_INVALID_ARGUMENT, "moe_dispatch_static: offsets is NULL");
    if (tokens > 0 && (!topk || !q || !scales || !row_token || !q_out || !scales_out))
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "moe_dispatch_static: null pointer");
    if (!aligned16(q) || !aligned16(q_out) || (reinterpret_cast<uintptr_t>(offsets) & 7u) ||
        (reinterpret_cast<uintptr_t>(topk) & 3u) || (reinterpret_cast<uintptr_t>(row_token) & 3u))
        return fail(FP4Q_ERR_MISALIGNED, "moe_dispatch_static: q, q_out 16-byte aligned; offsets 8-byte");
    fp4q_status st = current_device(nullptr);
    if (st != FP4Q_OK) return st;
    void* scratch = nullptr;
    if ((st = dispatch_scratch(&scratch)) != FP4Q_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t chunks = (tokens + kChunk - 1) / kChunk;
    int32_t* ws = static_cast<int32_t*>(scratch);
    int32_t* chunk_count = ws;
    int32_t* chunk_base = ws + chunks * n_experts;
    int32_t* local_rank = ws + 2 * chunks * n_experts;
    if (chunks > 0) {
        moe_count_kernel<<<unsigned(chunks), kChunk, 0, s>>>(topk, tokens, top_k, n_experts, chunk_count, local_rank);
        if ((st = check_launch("moe_dispatch_static count")) != FP4Q_OK) return st;
    }
    moe_scan_kernel<<<1, 256, 0, s>>>(chunk_count, chunks, n_experts, chunk_base, offsets);
    if ((st = check_launch("moe_dispatch_static scan")) != FP4Q_OK) return st;
    const int64_t pairs = tokens * top_k;
    if (pairs > 0 && cols > 0) {
        const int64_t blocks = (pairs * 32 + 255) / 256;
        moe_gather_kernel<<<unsigned(blocks), 256, 0, s>>>(topk, tokens, top_k, n_experts, chunk_base, local_rank,
                                                           offsets, q, scales, cols / 2, cols / 32, row_token, q_out,
                                                           scales_out);
        if ((st = check_launch("moe_dispatch_static gather")) != FP4Q_OK) return st;
    }
    return FP4Q_OK;
}
