// Block-scaled FP4 GEMM D = A . B^T on the sm_103a tensor cores.
//
// "Pretraining large language models with MXFP4 on Native FP4 Hardware",
// investigation section: the forward GEMM of a linear layer Y = X W^T with
// both operands in FP4 along the reduction axis, run on native FP4 tensor
// cores.  "Pretraining Large Language Models with NVFP4", section 2: NVFP4
// operands (E4M3 scale per 16, FP32 tensor scale); a Hadamard rotation of
// both operands along K cancels in the product.
//
// Persistent, warp-specialised kernel, one CTA per SM, 128 x 256 output tile
// per step, K consumed 256 elements (128 bytes) per pipeline stage:
//   warp 0      TMA producer: A and B tiles (128-byte swizzle) and the
//               stage's block scales (contiguous chunks of the MMA scale
//               layout) into a 4-stage shared-memory ring.
//   warp 1      allocates TMEM; one thread issues tcgen05.cp (scales ->
//               TMEM) and tcgen05.mma kind::mxf4 (UE8M0 per 32) or
//               kind::mxf4nvf4 (UE4M3 per 16), FP32 accumulator in TMEM.
//   warps 2..5  epilogue: tcgen05.ld of the 128 x 256 FP32 accumulator,
//               tensor-scale multiply (NVFP4), BF16 round-to-nearest-even
//               or FP32, stores; the accumulator is handed back to the MMA
//               thread as soon as it has been read.
// Every mbarrier wait is bounded in time; a wait that gives up sets a bit in
// the library's status word, tells the other roles to stop, and the kernel
// drains its own asynchronous work and frees TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"

namespace fp4q {
namespace {

constexpr int BM = 128, BN = 256, BK = 256;           // elements
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK / 2;             // 16384
constexpr uint32_t B_BYTES = BN * BK / 2;             // 32768
constexpr uint32_t SFA_BYTES = 4 * 512;               // up to 4 chunks (NVFP4)
constexpr uint32_t SFB_BYTES = 2 * 4 * 512;           // 2 row tiles x 4 chunks
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;   // 55296
constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + 256 + 1024;
constexpr int kThreads = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_SFA = 256;                    // 16 columns
constexpr uint32_t TMEM_SFB = 272;                    // 32 columns
constexpr uint64_t kWaitLimitNs = 4000000000ull;      // 4 s

struct GemmArgs {
    int M, N, K;
    int m_tiles, n_tiles, k_stages;
    int nv;                          // 0 = MXFP4, 1 = NVFP4
    const uint8_t* sfa;
    const uint8_t* sfb;
    uint64_t sfa_tile_stride;        // bytes per 128-row tile of A's scales
    uint64_t sfb_tile_stride;
    const float* ts_a;
    const float* ts_b;
    uint8_t* D;
    int64_t ldd;                     // elements
    int d_bf16;
    uint32_t* status;
};

__device__ __forceinline__ void flag_abort(volatile int* abort, uint32_t* status) {
    if (!*abort) {
        *abort = 1;
        atomicOr(status, kStatusGemmTimeout);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
            const GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    // bars[0..3] full, [4..7] empty, [8] tmem_full, [9] tmem_empty, [10] mma drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
    volatile int* abort = reinterpret_cast<volatile int*>(bars + 13);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = tc::smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t tmem_full = bar0 + 8u * 8, tmem_empty = bar0 + 8u * 9, drain_bar = bar0 + 8u * 10;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full_bar(s), 1);
            tc::mbar_init(empty_bar(s), 1);
        }
        tc::mbar_init(tmem_full, 1);
        tc::mbar_init(tmem_empty, 4);       // one arrival per epilogue warp
        tc::mbar_init(drain_bar, 1);
        *abort = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tmap_a);
        tc::tma_prefetch_desc(&tmap_b);
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int num_tiles = args.m_tiles * args.n_tiles;
    const uint32_t chunk_elems = args.nv ? 64 : 128;  // K elements per 512-byte scale chunk

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const int mt = tile % args.m_tiles, nt = tile / args.m_tiles;
            for (int kb = 0; kb < args.k_stages; ++kb) {
                if (!tc::mbar_wait(empty_bar(stage), phase ^ 1, abort, kWaitLimitNs)) {
                    flag_abort(abort, args.status);
                    ok = false;
                    break;
                }
                const int k_elems = min(BK, args.K - kb * BK);
                const uint32_t chunks = uint32_t(k_elems) / chunk_elems;
                const uint32_t ct0 = uint32_t(kb * BK) / chunk_elems;
                const bool rt1 = (2 * nt + 1) * 128 < args.N;
                const uint32_t sf_bytes = chunks * 512u * (rt1 ? 3u : 2u);
                uint8_t* st = smem + stage * STAGE_BYTES;
                const uint32_t fb = full_bar(stage);
                tc::mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES + sf_bytes);
                tc::tma_load_2d(tc::smem_u32(st), &tmap_a, fb, kb * (BK / 2), mt * BM);
                tc::tma_load_2d(tc::smem_u32(st + A_BYTES), &tmap_b, fb, kb * (BK / 2), nt * BN);
                tc::bulk_load(tc::smem_u32(st + A_BYTES + B_BYTES),
                              args.sfa + uint64_t(mt) * args.sfa_tile_stride + uint64_t(ct0) * 512u,
                              chunks * 512u, fb);
                uint8_t* sfb_smem = st + A_BYTES + B_BYTES + SFA_BYTES;
                tc::bulk_load(tc::smem_u32(sfb_smem),
                              args.sfb + uint64_t(2 * nt) * args.sfb_tile_stride + uint64_t(ct0) * 512u,
                              chunks * 512u, fb);
                if (rt1)
                    tc::bulk_load(tc::smem_u32(sfb_smem + 4 * 512),
                                  args.sfb + uint64_t(2 * nt + 1) * args.sfb_tile_stride + uint64_t(ct0) * 512u,
                                  chunks * 512u, fb);
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
        // drain: every stage issued last must have landed before the CTA exits
        for (int i = 0; i < STAGES && i < issued; ++i) {
            if (--stage < 0) { stage = STAGES - 1; phase ^= 1; }
            if (!tc::mbar_wait(full_bar(stage), phase, abort, kWaitLimitNs)) { flag_abort(abort, args.status); break; }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int tcount = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++tcount) {
            if (!tc::mbar_wait(tmem_empty, (tcount & 1) ^ 1, abort, kWaitLimitNs)) {
                flag_abort(abort, args.status);
                break;
            }
            tc::fence_after_sync();
            for (int kb = 0; kb < args.k_stages; ++kb) {
                if (!tc::mbar_wait(full_bar(stage), phase, abort, kWaitLimitNs)) {
                    flag_abort(abort, args.status);
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const int k_elems = min(BK, args.K - kb * BK);
                const uint32_t chunks = uint32_t(k_elems) / chunk_elems;
                const uint32_t nmma = uint32_t(k_elems) / 64;
                uint8_t* st = smem + stage * STAGE_BYTES;
                const uint32_t sa = tc::smem_u32(st), sb = tc::smem_u32(st + A_BYTES);
                const uint32_t ssfa = tc::smem_u32(st + A_BYTES + B_BYTES);
                const uint32_t ssfb = tc::smem_u32(st + A_BYTES + B_BYTES + SFA_BYTES);
                // block scales -> TMEM: chunk c of A at column TMEM_SFA + 4c, chunk c
                // of B's row tile r at TMEM_SFB + 8c + 4r
                for (uint32_t c = 0; c < chunks; ++c) {
                    tc::tc_cp_32x128b_warpx4(tmem + TMEM_SFA + 4 * c, tc::smem_desc(ssfa + 512 * c, 0, 128, 0));
                    tc::tc_cp_32x128b_warpx4(tmem + TMEM_SFB + 8 * c, tc::smem_desc(ssfb + 512 * c, 0, 128, 0));
                    tc::tc_cp_32x128b_warpx4(tmem + TMEM_SFB + 8 * c + 4,
                                             tc::smem_desc(ssfb + 4 * 512 + 512 * c, 0, 128, 0));
                }
                for (uint32_t j = 0; j < nmma; ++j) {
                    const uint64_t da = tc::smem_desc(sa + 32 * j, 16, 1024, 2);
                    const uint64_t db = tc::smem_desc(sb + 32 * j, 16, 1024, 2);
                    const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
                    if (args.nv) {
                        const uint32_t id = tc::idesc_block_scaled(BM, BN, false, 0, 0);
                        tc::mma_nvf4(tmem, da, db, id, tmem + TMEM_SFA + 4 * j, tmem + TMEM_SFB + 8 * j, acc);
                    } else {
                        const uint32_t sfid = (j & 1) * 2;
                        const uint32_t id = tc::idesc_block_scaled(BM, BN, true, sfid, sfid);
                        tc::mma_mxf4(tmem, da, db, id, tmem + TMEM_SFA + 4 * (j >> 1), tmem + TMEM_SFB + 8 * (j >> 1),
                                     acc);
                    }
                }
                tc::tc_commit(empty_bar(stage));
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            tc::tc_commit(tmem_full);
        }
        // drain: all MMAs and scale copies of this thread complete
        tc::tc_commit(drain_bar);
        if (!tc::mbar_wait(drain_bar, 0, abort, kWaitLimitNs)) flag_abort(abort, args.status);
    } else if (warp >= 2) {
        // ---------------- epilogue ----------------
        const int q = warp & 3;                         // TMEM lane quadrant of this warp
        const float alpha = args.nv ? __fmul_rn(*args.ts_a, *args.ts_b) : 1.0f;
        int tcount = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tcount) {
            if (!tc::mbar_wait(tmem_full, tcount & 1, abort, kWaitLimitNs)) {
                flag_abort(abort, args.status);
                break;
            }
            tc::fence_after_sync();
            const int mt = tile % args.m_tiles, nt = tile / args.m_tiles;
            const int row = mt * BM + q * 32 + lane;
            const int col0 = nt * BN;
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tc::tmem_ld_32x32b_x32(tmem + (uint32_t(q * 32) << 16) + uint32_t(c * 32), r);
                tc::tmem_ld_wait();
                if (c == BN / 32 - 1) {
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(tmem_empty);
                }
                const int col = col0 + c * 32;
                if (row >= args.M || col >= args.N) continue;
                const int ncol = min(32, args.N - col);
                if (args.d_bf16) {
                    uint32_t p[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float lo = __fmul_rn(u2f(r[2 * i]), alpha), hi = __fmul_rn(u2f(r[2 * i + 1]), alpha);
                        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(p[i]) : "f"(hi), "f"(lo));
                    }
                    uint8_t* dst = args.D + (int64_t(row) * args.ldd + col) * 2;
                    if (ncol == 32) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            reinterpret_cast<uint4*>(dst)[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < ncol) reinterpret_cast<uint16_t*>(dst)[i] = uint16_t(p[i >> 1] >> (16 * (i & 1)));
                    }
                } else {
                    float* dst = reinterpret_cast<float*>(args.D) + int64_t(row) * args.ldd + col;
                    if (ncol == 32) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            reinterpret_cast<float4*>(dst)[i] =
                                make_float4(__fmul_rn(u2f(r[4 * i]), alpha), __fmul_rn(u2f(r[4 * i + 1]), alpha),
                                            __fmul_rn(u2f(r[4 * i + 2]), alpha), __fmul_rn(u2f(r[4 * i + 3]), alpha));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < ncol) dst[i] = __fmul_rn(u2f(r[i]), alpha);
                    }
                }
            }
        }
    }
    __syncwarp();          // the elected lanes rejoin their warps before the block barrier
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

fp4q_status get_encoder() {
    if (g_encode) return FP4Q_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(FP4Q_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return FP4Q_OK;
}

// 2D map over packed FP4 bytes [rows, K/2], box (128 bytes) x box_rows, 128B swizzle.
fp4q_status encode_operand_map(CUtensorMap* map, const uint8_t* q, int64_t rows, int64_t K, uint32_t box_rows) {
    cuuint64_t dims[2] = {cuuint64_t(K / 2), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(K / 2)};
    cuuint32_t box[2] = {128u, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FP4Q_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return FP4Q_OK;
}

}  // namespace
}  // namespace fp4q

using namespace fp4q;

extern "C" fp4q_status fp4q_block_scaled_gemm(const fp4q_operand* A, const fp4q_operand* B, int64_t M,
                                              int64_t N, int64_t K, void* D, fp4q_dtype d_type, int64_t ldd,
                                              fp4q_stream_t stream) {
    if (!A || !B) return fail(FP4Q_ERR_INVALID_ARGUMENT, "gemm: operand is NULL");
    if (A->format != B->format || (A->format != FP4Q_MXFP4 && A->format != FP4Q_NVFP4))
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "gemm: A and B must both be MXFP4 or both NVFP4");
    if (d_type != FP4Q_BF16 && d_type != FP4Q_FP32)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "gemm: d_type must be BF16 or FP32");
    if (M < 0 || N < 0 || K < 0 || ldd < N) return fail(FP4Q_ERR_INVALID_ARGUMENT, "gemm: bad sizes");
    if (K % 128) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "gemm: K %% 128 != 0");
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "gemm: sizes beyond 2^30");
    if (M == 0 || N == 0) return FP4Q_OK;
    if (!A->q || !B->q || !A->scales || !B->scales || !D)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "gemm: null pointer");
    const bool nv = A->format == FP4Q_NVFP4;
    if (nv && (!A->tensor_scale || !B->tensor_scale))
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "gemm: NVFP4 operands need tensor scales");
    const int64_t esz = d_type == FP4Q_BF16 ? 2 : 4;
    if (!aligned16(A->q) || !aligned16(B->q) || !aligned16(A->scales) || !aligned16(B->scales) || !aligned16(D) ||
        (ldd * esz) % 16)
        return fail(FP4Q_ERR_MISALIGNED, "gemm: q, scales, D must be 16-byte aligned and ldd*elem %% 16 == 0");
    if (K == 0) {
        cudaError_t e = cudaMemset2DAsync(D, size_t(ldd * esz), 0, size_t(N * esz), size_t(M),
                                          reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? FP4Q_OK : fail(FP4Q_ERR_CUDA, "gemm: memset: %s", cudaGetErrorString(e));
    }
    int sms = 0;
    fp4q_status st = current_device(&sms);
    if (st != FP4Q_OK) return st;
    if ((st = get_encoder()) != FP4Q_OK) return st;
    CUtensorMap ma, mb;
    if ((st = encode_operand_map(&ma, A->q, M, K, BM)) != FP4Q_OK) return st;
    if ((st = encode_operand_map(&mb, B->q, N, K, BN)) != FP4Q_OK) return st;

    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM_BYTES));
        if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "gemm: smem attribute: %s", cudaGetErrorString(e));
        attr_set[dev & 63] = true;
    }
    GemmArgs a;
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.m_tiles = int((M + BM - 1) / BM);
    a.n_tiles = int((N + BN - 1) / BN);
    a.k_stages = int((K + BK - 1) / BK);
    a.nv = nv ? 1 : 0;
    a.sfa = A->scales;
    a.sfb = B->scales;
    const int64_t s4 = nv ? K / 64 : K / 128;          // 4-scale chunks per row tile
    a.sfa_tile_stride = uint64_t(s4) * 512u;
    a.sfb_tile_stride = uint64_t(s4) * 512u;
    a.ts_a = A->tensor_scale;
    a.ts_b = B->tensor_scale;
    a.D = static_cast<uint8_t*>(D);
    a.ldd = ldd;
    a.d_bf16 = d_type == FP4Q_BF16;
    a.status = status_word();
    const int tiles = a.m_tiles * a.n_tiles;
    const int grid = tiles < sms ? tiles : sms;
    gemm_kernel<<<grid, kThreads, SMEM_BYTES, reinterpret_cast<cudaStream_t>(stream)>>>(ma, mb, a);
    return check_launch("block_scaled_gemm");
}
